"""NVFP4 encoding of expert weights (input preparation, not part of the decode step).

Format: e2m1 element codes (1 sign, 2 exponent, 1 mantissa bit; magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6),
one e4m3 scale per block of 16 consecutive inputs (the contiguous, last axis), and one fp32 scale
per expert tensor. A weight decodes as  e2m1(code) * e4m3(scale) * tensor_scale.

Encoding used here (the plainest reading of "quantised from N(0, 0.02) draws"):
  G   = amax(|w|) / (6 * 448)                          (fp32, per tensor)
  s_b = e4m3_rne(amax_b / (6 G)), clamped to 448        (per 16-block; an all-zero block gets 0)
  q   = e2m1_rne(w / (s_b G)), clamped to +-6, ties to the even code
Codes are packed two per byte, element 2i in the low nibble and 2i+1 in the high nibble.
"""
from __future__ import annotations

import torch

# magnitude of code c (c = 0..7); code | 8 is the negative value
E2M1_GRID = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)
_MIDS = (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0)


def _e2m1_code(v: torch.Tensor) -> torch.Tensor:
    """Round fp32 values to the nearest e2m1 code, ties to the even code (uint8, 0..15)."""
    mag = v.abs().clamp(max=6.0)
    mids = torch.tensor(_MIDS, dtype=v.dtype, device=v.device)
    # number of midpoints strictly below mag: the lower neighbour's code on a tie
    code = torch.searchsorted(mids, mag.contiguous(), right=False)
    on_tie = (code < len(_MIDS)) & (mids[code.clamp(max=len(_MIDS) - 1)] == mag)
    code = torch.where(on_tie & (code % 2 == 1), code + 1, code)
    sign = (v < 0) & (code > 0)
    return (code + 8 * sign.to(code.dtype)).to(torch.uint8)


def _encode(w: torch.Tensor, g: torch.Tensor):
    """Block scales and codes of ``w`` [..., K] given its tensor scale ``g`` (broadcastable to w's
    leading dims + one trailing block axis)."""
    blocks = w.reshape(*w.shape[:-1], w.shape[-1] // 16, 16)
    amax_b = blocks.abs().amax(dim=-1)
    s = (amax_b / (6.0 * g)).clamp(max=448.0).to(torch.float8_e4m3fn)
    s_val = s.float()
    denom = (s_val * g).unsqueeze(-1)
    safe = torch.where(denom > 0, denom, torch.ones_like(denom))
    scaled = torch.where(denom > 0, blocks / safe, torch.zeros_like(blocks))
    codes = _e2m1_code(scaled).reshape(*w.shape)
    packed = codes[..., 0::2] | (codes[..., 1::2] << 4)
    return packed.contiguous(), s.view(torch.uint8).contiguous()


def quantize_nvfp4(w: torch.Tensor):
    """Encode fp32 ``w`` [..., K] (K % 16 == 0). Returns (packed uint8 [..., K/2],
    e4m3 scale bits uint8 [..., K/16], fp32 tensor scale [1])."""
    assert w.shape[-1] % 16 == 0
    w = w.float()
    amax = w.abs().max()
    g = (amax / (6.0 * 448.0)).reshape(1).float()
    if float(amax) == 0.0:
        g = torch.ones(1, dtype=torch.float32, device=w.device)
    packed, s = _encode(w, g)
    return packed, s, g


def quantize_nvfp4_experts(w: torch.Tensor):
    """``quantize_nvfp4`` applied to each w[e] of a stack [E, rows, K] at once (one tensor scale per
    expert); the same bytes as the per-expert calls. Returns (packed [E, rows, K/2], scales
    [E, rows, K/16], tensor scales [E])."""
    assert w.dim() == 3 and w.shape[-1] % 16 == 0
    w = w.float()
    amax = w.abs().amax(dim=(1, 2))
    g = (amax / (6.0 * 448.0)).float()
    g = torch.where(amax == 0.0, torch.ones_like(g), g)
    packed, s = _encode(w, g.reshape(-1, 1, 1))
    return packed, s, g
