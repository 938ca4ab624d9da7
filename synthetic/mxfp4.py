"""MXFP4 expert weights and their FP8-E4M3 re-encoding (input preparation, not part of the decode step).

The pages' own expert format: the experts ship in MXFP4; the loader re-encodes each expert's gate and up
projections into FP8 E4M3 with one BF16 scale per 256 rows, checks bit for bit that the new encoding decodes
to the same values and raises if it does not; the down projection stays MXFP4 (Kimi K3's TPU megakernel,
"How it maps onto a TPU v7", the precision paragraph).

MXFP4 (the OCP microscaling format): e2m1 element codes (magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6) in blocks of
32 consecutive inputs (the contiguous, last axis), one E8M0 scale byte per block (value 2^(byte - 127)).
Encoding used here, the format's plainest rule: the block's shared exponent X = floor(log2 amax) - 2 (2 being
the largest e2m1 exponent), clamped to [-127, 127]; q = e2m1_rne(w / 2^X), saturating at +-6, ties to the
even code; an all-zero block gets X = -127. Codes are packed two per byte, element 2i in the low nibble.

FP8 re-encoding (the loader's step, read plainly): "rows" are the output rows of a gate / up matrix
[rows, K]; rows 256 j .. 256 j + 255 share one scale S_j, a power of two (exact in bf16) chosen as
2^(E_max - 8), E_max being the largest block exponent X + 2 in those rows, so that the largest
representable MXFP4 value, 6 * 2^X = 1.5 * 2^(X + 2), maps to at most 384 <= 448. Each value v becomes the
e4m3 code of v / S_j; the re-encoding is accepted only if every code decodes to exactly v / S_j.
"""
from __future__ import annotations

import torch

from .nvfp4 import _e2m1_code

ROWS_PER_SCALE = 256
MX_BLOCK = 32


def quantize_mxfp4(w: torch.Tensor):
    """Encode fp32 ``w`` [..., K] (K % 32 == 0). Returns (packed uint8 [..., K/2], E8M0 scale bytes uint8
    [..., K/32])."""
    assert w.shape[-1] % MX_BLOCK == 0
    w = w.float()
    blocks = w.reshape(*w.shape[:-1], w.shape[-1] // MX_BLOCK, MX_BLOCK)
    amax = blocks.abs().amax(dim=-1)
    # floor(log2 amax) from the float's own exponent (frexp: amax = m 2^e with m in [0.5, 1))
    _, e = torch.frexp(amax)
    x = torch.where(amax > 0, (e - 1 - 2).to(torch.int32), torch.full_like(e, -127, dtype=torch.int32))
    x = x.clamp(-127, 127)
    scale = torch.ldexp(torch.ones_like(amax), x)
    codes = _e2m1_code(blocks / scale.unsqueeze(-1)).reshape(*w.shape)
    packed = codes[..., 0::2] | (codes[..., 1::2] << 4)
    return packed.contiguous(), (x + 127).to(torch.uint8).contiguous()


def mxfp4_values(packed: torch.Tensor, e8m0: torch.Tensor) -> torch.Tensor:
    """The exact values (float64) of MXFP4 weights: e2m1(code) * 2^(e8m0 - 127). Used by the re-encoder to
    check itself; the oracle decodes with its own routine."""
    grid = torch.tensor((0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0), dtype=torch.float64, device=packed.device)
    lo = (packed & 0x0F).long()
    hi = (packed >> 4).long()
    codes = torch.stack([lo, hi], dim=-1).reshape(*packed.shape[:-1], packed.shape[-1] * 2)
    mag = grid[codes & 7]
    vals = torch.where(codes >= 8, -mag, mag)
    x = e8m0.to(torch.float64) - 127.0
    return vals * torch.repeat_interleave(torch.exp2(x), MX_BLOCK, dim=-1)


def reencode_fp8_rows(packed: torch.Tensor, e8m0: torch.Tensor):
    """Re-encode MXFP4 gate / up weights [rows, K] (as ``quantize_mxfp4`` returns them) into e4m3 codes
    uint8 [rows, K] and bf16 scale bits uint16 [ceil(rows / 256)], one scale per 256 rows. Raises
    ValueError if any value does not survive the re-encoding exactly."""
    rows = packed.shape[0]
    v = mxfp4_values(packed, e8m0)
    nblk = -(-rows // ROWS_PER_SCALE)
    codes = torch.empty(v.shape, dtype=torch.uint8, device=v.device)
    sbits = torch.empty(nblk, dtype=torch.int32, device=v.device)
    for j in range(nblk):
        r0, r1 = j * ROWS_PER_SCALE, min(rows, (j + 1) * ROWS_PER_SCALE)
        emax = int(e8m0[r0:r1].to(torch.int32).max()) - 127 + 2
        s = 2.0 ** (emax - 8)
        scaled = v[r0:r1] / s
        f8 = scaled.to(torch.float8_e4m3fn)
        if not torch.equal(f8.to(torch.float64) * s, v[r0:r1]):
            raise ValueError(f"rows {r0}..{r1 - 1}: the values are not exact in e4m3 with one scale")
        codes[r0:r1] = f8.view(torch.uint8)
        sb = torch.tensor([s], dtype=torch.float32).to(torch.bfloat16)
        if float(sb) != s:
            raise ValueError(f"rows {r0}..{r1 - 1}: scale 2^{emax - 8} is not a bf16 value")
        sbits[j] = int(sb.view(torch.int16).item()) & 0xFFFF
    return codes, sbits.to(torch.int32)
