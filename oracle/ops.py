"""Primitive operations of the decode step, in plain numpy float64.

Citations name the page and section of the source material. The pages name the operations
(RMSNorm, residual, grouped-query attention, MLA with a 576-wide latent, the KDA / gated-delta-net
recurrence, sigmoid top-k routing, SwiGLU experts, NVFP4 and MXFP4 / FP8-E4M3 experts) but print almost no formulas, so
most definitions below are the plainest standard reading of those names; each says which.
"""
from __future__ import annotations

import numpy as np

F64 = np.float64


# ----------------------------------------------------------------------------------------------
# storage rounding
# ----------------------------------------------------------------------------------------------
def bf16_round(x) -> np.ndarray:
    """Round to bfloat16 (round to nearest, ties to even) and return float64.

    The value is first rounded to float32 (as every fp32 producer would hold it), then its low 16 bits
    are rounded away. The step itself rounds nothing; this serves the tests that reason about bf16
    storage.
    Pinned: equals torch's float32 -> bfloat16 conversion (tests/test_oracle_ops.py)."""
    f = np.asarray(x, dtype=np.float32)
    bits = f.view(np.uint32).astype(np.uint64)
    lsb = (bits >> 16) & 1
    rounded = ((bits + 0x7FFF + lsb) >> 16) << 16
    return rounded.astype(np.uint32).view(np.float32).astype(F64)


# ----------------------------------------------------------------------------------------------
# matrix products with float64 accumulation
# ----------------------------------------------------------------------------------------------
def linear(x: np.ndarray, w: np.ndarray, block: int = 4096) -> np.ndarray:
    """y = x @ w.T with x [..., K] float64 and w [O, K] (float32 holding bf16 values).

    The weight is widened to float64 one block of rows at a time, so the product and its
    accumulation are float64 without holding a float64 copy of a large matrix."""
    x = np.asarray(x, dtype=F64)
    lead = x.shape[:-1]
    x2 = x.reshape(-1, x.shape[-1])
    out = np.empty((x2.shape[0], w.shape[0]), dtype=F64)
    for o0 in range(0, w.shape[0], block):
        wb = np.asarray(w[o0:o0 + block], dtype=F64)
        out[:, o0:o0 + block] = x2 @ wb.T
    return out.reshape(*lead, w.shape[0])


# ----------------------------------------------------------------------------------------------
# normalisation, activation, rotary embedding
# ----------------------------------------------------------------------------------------------
def rmsnorm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm over the last axis: x / sqrt(mean(x^2) + eps) * g.

    The pages list RMSNorm among the vector-unit work of the kernel (Kimi K3's TPU megakernel,
    "How it maps onto a TPU v7"); the gain multiplies (not 1 + g). Pinned: torch rms_norm,
    constant-vector closed form."""
    x = np.asarray(x, dtype=F64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(g, dtype=F64)


def silu(z: np.ndarray) -> np.ndarray:
    """silu(z) = z / (1 + exp(-z)); the SwiGLU gate. Pinned: torch silu."""
    z = np.asarray(z, dtype=F64)
    return z / (1.0 + np.exp(-z))


def sigmoid(z: np.ndarray) -> np.ndarray:
    z = np.asarray(z, dtype=F64)
    return 1.0 / (1.0 + np.exp(-z))


def rope(x: np.ndarray, pos, theta: float) -> np.ndarray:
    """Rotary embedding, rotate-half pairing: dims (i, i + D/2) rotate by angle pos * theta^(-2i/D).

    x [..., D]; ``pos`` broadcasts against x's leading axes (one position per row).
    The pages only name RoPE; rotate-half over the full rotated width is the reading taken.
    Pinned: identity at position 0, norm preservation, complex-multiplication form, relative-position
    property of the rotated dot product."""
    x = np.asarray(x, dtype=F64)
    d = x.shape[-1]
    half = d // 2
    inv_freq = theta ** (-(2.0 * np.arange(half, dtype=F64)) / d)
    ang = np.asarray(pos, dtype=F64)[..., None] * inv_freq
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


# ----------------------------------------------------------------------------------------------
# attention
# ----------------------------------------------------------------------------------------------
def softmax_attend(scores: np.ndarray, values: np.ndarray) -> np.ndarray:
    """Max-subtracted softmax over the last axis of scores [.., T], applied to values [.., T, Dv].
    Masked positions carry -inf and get weight 0."""
    m = np.max(scores, axis=-1, keepdims=True)
    p = np.exp(scores - m)
    p = p / np.sum(p, axis=-1, keepdims=True)
    return p @ values


def gqa_block_attention(q: np.ndarray, K: np.ndarray, V: np.ndarray, p0: int) -> np.ndarray:
    """Causal grouped-query attention for a block of R rows at positions p0 .. p0+R-1.

    q [R, Hq, hd] (already rotated); K, V [p0 + R, Hkv, hd] hold the cache including the block.
    Row r attends over cache positions 0 .. p0 + r. Query head h reads kv head floor(h * Hkv / Hq).
    Scale 1/sqrt(hd). The causal rule within a block follows the verify description: an anchor plus
    seven drafts are verified as eight rows of one sequence (Kimi K3's TPU megakernel, "What DSpark
    changes per step"), each row seeing the rows before it.
    Pinned: torch scaled_dot_product_attention, single-key case, block == row-by-row decode."""
    R, hq, hd = q.shape
    hkv = K.shape[1]
    T = p0 + R
    kv_of = (np.arange(hq) * hkv) // hq
    mask = np.arange(T)[None, :] <= (p0 + np.arange(R))[:, None]   # [R, T]
    o = np.empty((R, hq, hd))
    for g in range(hkv):
        heads = np.nonzero(kv_of == g)[0]                  # the query heads that read kv head g
        Kg, Vg = K[:T, g], V[:T, g]                        # [T, hd]
        scores = np.transpose(q[:, heads], (1, 0, 2)) @ Kg.T / np.sqrt(hd)   # [heads, R, T]
        scores = np.where(mask[None], scores, -np.inf)
        o[:, heads] = np.transpose(softmax_attend(scores, Vg), (1, 0, 2))
    return o


# ----------------------------------------------------------------------------------------------
# delta-rule recurrences (gated delta net, Kimi delta attention)
# ----------------------------------------------------------------------------------------------
def l2_normalize(x: np.ndarray, eps: float = 1e-6) -> np.ndarray:
    x = np.asarray(x, dtype=F64)
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)


def delta_rule_step(S, q_hat, k_hat, v, alpha, beta):
    """One token of the gated delta rule for one head.

    S [dk, dv] state; q_hat, k_hat [dk]; v [dv]; alpha a scalar (gated delta net, one decay per
    head) or a [dk] vector (KDA, one decay per key channel); beta a scalar.
        S <- Diag(alpha) S              (alpha * S when alpha is a scalar)
        u  = v - S^T k_hat
        S <- S + beta * k_hat u^T
        o  = S^T q_hat
    The pages place the KDA recurrence on the vector unit and note its state does not grow with
    context (Kimi K3's TPU megakernel, "Why one user at a time is a bandwidth problem"); the update
    itself is the standard gated delta rule. Pinned: the explicit product/sum form on T <= 6,
    identity at alpha = 1, beta = 0, exact overwrite at beta = 1 with a unit key."""
    alpha = np.asarray(alpha, dtype=F64)
    if alpha.ndim == 0:
        S = alpha * S
    else:
        S = alpha[:, None] * S
    u = v - S.T @ k_hat
    S = S + beta * np.outer(k_hat, u)
    return S, S.T @ q_hat


# ----------------------------------------------------------------------------------------------
# mixture-of-experts routing
# ----------------------------------------------------------------------------------------------
def route(z: np.ndarray, bias: np.ndarray, top_k: int, scale: float):
    """Sigmoid top-k routing for one row.

    s = sigmoid(z); experts are picked by top_k sequential argmax passes over s + bias, the lowest
    index winning a tie (the pages' router takes its top-16 as sixteen sequential argmax passes,
    Kimi K3's TPU megakernel, "How it maps onto a TPU v7"). The weights are the picked sigmoid
    scores renormalised to sum to 1 and multiplied by ``scale``; the bias only steers selection.
    Returns (indices in pick order, weights, biased scores of all experts).
    Pinned: a full stable sort gives the same set and order."""
    s = sigmoid(z)
    biased = s + np.asarray(bias, dtype=F64)
    avail = biased.copy()
    picked = []
    for _ in range(top_k):
        i = int(np.argmax(avail))  # first occurrence on ties
        picked.append(i)
        avail[i] = -np.inf
    idx = np.array(picked, dtype=np.int64)
    w = scale * s[idx] / np.sum(s[idx])
    return idx, w, biased


def greedy_accept(logits: np.ndarray, block_tokens) -> tuple:
    """Greedy acceptance of one verify block: logits [R, V] of rows 0..R-1 (row 0 the anchor, rows 1.. the
    drafts), block_tokens [R] their tokens. Draft r + 1 is accepted while it equals the greedy token of row r
    (lowest index on ties); returns (accepted rows a, 1 <= a <= R, and the bonus token: the greedy token of
    row a - 1). The block emits its accepted prefix plus that one bonus token (Kimi K3's TPU megakernel,
    "What DSpark changes per step"). Pinned: equals the prefix that sequential greedy decoding from the
    anchor would have produced."""
    R = logits.shape[0]
    a = 1
    while a < R and int(np.argmax(logits[a - 1])) == int(block_tokens[a]):
        a += 1
    return a, int(np.argmax(logits[a - 1]))


def swiglu(y: np.ndarray, w_gate, w_up, w_down) -> np.ndarray:
    """SwiGLU feed-forward: (silu(y Wg^T) * (y Wu^T)) Wd^T."""
    return linear(silu(linear(y, w_gate)) * linear(y, w_up), w_down)


# ----------------------------------------------------------------------------------------------
# NVFP4 decoding
# ----------------------------------------------------------------------------------------------
def e2m1_value(code: np.ndarray) -> np.ndarray:
    """Value of a 4-bit e2m1 code: sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0.
    Exponent 0 is subnormal: m * 0.5. Pinned against the enumerated e2m1 grid."""
    code = np.asarray(code).astype(np.int64)
    sign = np.where(code & 8, -1.0, 1.0)
    e = (code >> 1) & 3
    m = code & 1
    mag = np.where(e == 0, 0.5 * m, np.exp2(e - 1.0) * (1.0 + 0.5 * m))
    return sign * mag


def e4m3_value(bits: np.ndarray) -> np.ndarray:
    """Value of an e4m3 (fn variant) byte: sign bit 7, exponent bits 6..3 (bias 7), mantissa 2..0;
    exponent 0 is subnormal (m/8 * 2^-6); S.1111.111 is NaN. Pinned against torch float8_e4m3fn."""
    b = np.asarray(bits).astype(np.int64)
    sign = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 3) & 15
    m = b & 7
    mag = np.where(e == 0, (m / 8.0) * 2.0 ** -6, np.exp2(e - 7.0) * (1.0 + m / 8.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sign * mag


def e8m0_value(bits: np.ndarray) -> np.ndarray:
    """Value of an E8M0 scale byte (the microscaling formats' shared scale): 2^(bits - 127); 0xFF is NaN.
    Pinned by its closed forms (1, 2, 2^-127, 2^127, NaN)."""
    b = np.asarray(bits).astype(np.int64)
    return np.where(b == 255, np.nan, np.exp2(b - 127.0))


def bf16_value(bits: np.ndarray) -> np.ndarray:
    """Value of a bfloat16 bit pattern (the high half of a float32). Pinned against torch's bfloat16."""
    b = (np.asarray(bits).astype(np.int64) & 0xFFFF).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(F64)


def mxfp4_decode(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """Decode MXFP4 weights [..., K] from packed e2m1 codes q [..., K/2] (element 2i in the low nibble) and
    E8M0 block scales s [..., K/32]: w = e2m1(code) * 2^(s - 127). The down projection of the pages' own
    expert format is MXFP4 (Kimi K3's TPU megakernel, "How it maps onto a TPU v7"); blocks of 32 along the
    input axis with an E8M0 scale are the microscaling format's definition.
    Pinned: a hand-built block, the encoder's grid round trip, and the FP8 re-encoding's exactness."""
    q = np.asarray(q, dtype=np.uint8)
    codes = np.stack([q & 0x0F, q >> 4], axis=-1).reshape(*q.shape[:-1], q.shape[-1] * 2)
    return e2m1_value(codes) * np.repeat(e8m0_value(s), 32, axis=-1)


def fp8_rows_decode(codes: np.ndarray, scale_bits: np.ndarray, rows_per_scale: int = 256) -> np.ndarray:
    """Decode FP8-E4M3 gate / up weights [rows, K] from their e4m3 codes and one bf16 scale per
    ``rows_per_scale`` consecutive rows: w[r, k] = e4m3(codes[r, k]) * bf16(scale_bits[r // 256]) (the
    loader's re-encoding of the MXFP4 gate / up projections: Kimi K3's TPU megakernel, "How it maps onto a
    TPU v7"; "rows" read as the matrix's output rows).
    Pinned: rows 255 and 256 take different scales in a hand-built case; decodes the re-encoder's output
    to the MXFP4 values bit for bit."""
    codes = np.asarray(codes, dtype=np.uint8)
    rows = codes.shape[0]
    scale = bf16_value(scale_bits)[np.arange(rows) // rows_per_scale]
    return e4m3_value(codes) * scale[:, None]


def nvfp4_decode(q: np.ndarray, s: np.ndarray, g: float) -> np.ndarray:
    """Decode NVFP4 weights [..., K] from packed codes q [..., K/2] (element 2i in the low nibble),
    e4m3 block scales s [..., K/16] and the fp32 tensor scale g: w = e2m1 * e4m3(block) * g.
    The pages name NVFP4 as the Muse-Spark-Open weight format (tpu-megakernels README, intro).
    Pinned: round trip of on-grid values through the encoder is exact."""
    q = np.asarray(q, dtype=np.uint8)
    lo = q & 0x0F
    hi = q >> 4
    codes = np.stack([lo, hi], axis=-1).reshape(*q.shape[:-1], q.shape[-1] * 2)
    vals = e2m1_value(codes)
    scales = np.repeat(e4m3_value(s), 16, axis=-1)
    return vals * scales * np.float64(np.float32(g))
