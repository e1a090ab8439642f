"""CPU oracle for the routed top-k Mixture-of-Experts experts forward.

TEST INFRASTRUCTURE ONLY.  Only the tests, the package's smoke check and the
benchmark's CPU-baseline leg may import this module; the product path never
calls it and shares no code with it.

Source of the method: Hugging Face Transformers documentation page
"Experts backends" (experts_interface), introduction: a router ranks the
experts of every token and keeps k of them; the token's hidden state passes
through each kept expert, and the k expert outputs are summed with the
routing weights as coefficients.
The "eager" row of the backends table describes the plain form this oracle
follows: loop over the selected experts and apply the projections to their
tokens.  The gated MLP is "up projection, SwiGLU, down projection" (the
deepgemm_megamoe row of the backends table and the "Fused Mega MoE on
Blackwell" section); the SonicMoE section maps the gate activations silu,
gelu and relu to SwiGLU, GeGLU and ReGLU.  FP8 experts carry float32 or UE8M0 block scales (paragraph after the
backends table) and activations take dynamic per-row scales ("FP8 and FP4
quantized experts" section).

Everything the page leaves open is fixed by the readings listed in the
project's design notes:
  * router: softmax over all E logits, keep the top k, renormalise over the
    k kept (the full-softmax denominator cancels, so the weights are a softmax
    over the kept logits); ties go to the lower expert index; slots are
    ordered by descending logit, ties by ascending index; a row whose largest
    logit is -inf gets uniform weights 1/k;
  * fused gate/up weight W_gate_up[e] is [2I, H], rows 0..I-1 gate and rows
    I..2I-1 up; W_down[e] is [H, I] (the [out, in] convention);
  * SwiGLU: h = silu(g) * u, silu(x) = x / (1 + exp(-x)), no bias, no clamp;
    GeGLU: h = gelu(g) * u with the exact GELU x * Phi(x) = x/2 (1 + erf(x/sqrt 2))
    (the page says only "gelu"; the tanh approximation is a different name);
    ReGLU: h = max(g, 0) * u;
  * combine: out[t] = sum_j w[t,j] * y[t,j], summed in the oracle's float
    type and rounded once to bf16 (round to nearest even);
  * dispatch: expert-contiguous rows, stable in the flat index f = t*k + j;
  * FP8: e4m3fn codes, round to nearest even with saturation to +-448;
    128x128 weight blocks, 1x128 activation blocks along the contraction
    axis; scale s = amax/448 in fp32 (float format) or the smallest power of
    two >= that fp32 quotient (UE8M0 format); amax = 0 gives s = 1; codes are
    e4m3(x * (1/s)) with the reciprocal and product in fp32; the down
    projection's input h is quantised the same way along I.

All floating point is float64 unless stated; the quantiser works in fp32 on
purpose, because it decides integer codes and both sides must take that
decision in the same precision.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "route", "route_weights_full_softmax", "dispatch", "silu", "gelu", "relu",
    "ACTIVATIONS",
    "expert_mlp", "forward", "forward_brute", "round_to_bf16",
    "bf16_bits_to_f32", "e4m3_encode", "e4m3_decode", "ue8m0_from_quotient",
    "quantize_blocks", "dequantize_blocks", "requantize_rows", "forward_fp8",
    "e2m1_encode", "e2m1_decode", "pack_e2m1", "unpack_e2m1", "quantize_fp4_blocks",
    "dequantize_fp4_blocks", "forward_fp4",
    "touched_weight_bytes", "rel_max_err",
]


# --------------------------------------------------------------------------
# bf16 helpers (storage format of the hidden states, weights and output)
# --------------------------------------------------------------------------

def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float32 values (exact widening)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32)


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round to the nearest bf16 value, ties to even; returns float32 values
    that are exactly representable in bf16.  Float64 input is first rounded
    to float32 (the output is compared under a tolerance, so the double
    rounding does not matter)."""
    f = np.asarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)) << np.uint64(16)
    r = r.astype(np.uint32)
    nan = np.isnan(f)
    r[nan] = np.uint32(0x7FC00000)
    return r.view(np.float32)


# --------------------------------------------------------------------------
# Router (introduction of the page: a router picks the top-k experts of each token)
# --------------------------------------------------------------------------

def route(logits: np.ndarray, k: int):
    """Top-k routing of fp32 logits [T, E].

    Returns (topk_idx int32 [T,k], topk_w float64 [T,k]).  Selection orders
    experts by (logit descending, index ascending) and keeps the first k; the
    weights are the softmax over all E renormalised over the kept k, written
    here in the cancelled form exp(l_j - l_0) / sum_i exp(l_i - l_0)."""
    logits = np.asarray(logits, dtype=np.float32)
    T, E = logits.shape
    if not (1 <= k <= E):
        raise ValueError("k must be in [1, E]")
    index = np.broadcast_to(np.arange(E), (T, E))
    # np.lexsort sorts by the last key first: primary -logit, secondary index
    order = np.lexsort((index, -logits.astype(np.float64)), axis=-1)
    idx = order[:, :k].astype(np.int32)
    sel = np.take_along_axis(logits, idx, axis=1).astype(np.float64)
    top = sel[:, :1]
    w = np.empty_like(sel)
    dead = np.isneginf(top[:, 0])
    live = ~dead
    ex = np.exp(sel[live] - top[live])
    w[live] = ex / ex.sum(axis=1, keepdims=True)
    w[dead] = 1.0 / k
    return idx, w


def route_weights_full_softmax(logits: np.ndarray, idx: np.ndarray) -> np.ndarray:
    """Second formula for the routing weights: p = softmax over all E
    (float64), then w_j = p[S_j] / sum_{i in S} p[i]."""
    l = np.asarray(logits, dtype=np.float64)
    m = l.max(axis=1, keepdims=True)
    p = np.exp(l - m)
    p = p / p.sum(axis=1, keepdims=True)
    ps = np.take_along_axis(p, idx.astype(np.int64), axis=1)
    return ps / ps.sum(axis=1, keepdims=True)


# --------------------------------------------------------------------------
# Dispatch (grouped_mm / deepgemm rows of the backends table: tokens are sorted
# by their selected expert before one grouped GEMM)
# --------------------------------------------------------------------------

def dispatch(topk_idx: np.ndarray, E: int):
    """Counting sort of the flat routing entries f = t*k + j by expert.

    Returns counts int32 [E], offsets int32 [E+1] (exclusive scan, offsets[E]
    = T*k), sorted_f int32 [T*k] (row r of the expert-contiguous order holds
    flat entry sorted_f[r], ascending f within an expert) and row_of int32
    [T*k] (its inverse)."""
    flat = np.asarray(topk_idx, dtype=np.int64).reshape(-1)
    n = flat.size
    if n and (flat.min() < 0 or flat.max() >= E):
        raise ValueError("expert index out of range")
    counts = np.zeros(E, dtype=np.int64)
    for e in flat:
        counts[e] += 1
    offsets = np.zeros(E + 1, dtype=np.int64)
    for e in range(E):
        offsets[e + 1] = offsets[e] + counts[e]
    cursor = offsets[:-1].copy()
    sorted_f = np.empty(n, dtype=np.int64)
    for f in range(n):
        e = flat[f]
        sorted_f[cursor[e]] = f
        cursor[e] += 1
    row_of = np.empty(n, dtype=np.int64)
    row_of[sorted_f] = np.arange(n)
    return (counts.astype(np.int32), offsets.astype(np.int32),
            sorted_f.astype(np.int32), row_of.astype(np.int32))


# --------------------------------------------------------------------------
# Gated expert MLP ("up projection, SwiGLU, down projection")
# --------------------------------------------------------------------------

def silu(x: np.ndarray) -> np.ndarray:
    """silu(x) = x * sigmoid(x) = x / (1 + exp(-x)), written to avoid
    overflow warnings for large negative x."""
    x = np.asarray(x)
    out = np.empty_like(x)
    pos = x >= 0
    out[pos] = x[pos] / (1.0 + np.exp(-x[pos]))
    ex = np.exp(x[~pos])
    out[~pos] = x[~pos] * ex / (1.0 + ex)
    return out


def _erf(x: np.ndarray) -> np.ndarray:
    try:
        from scipy.special import erf
        return erf(x)
    except ImportError:                      # plain per-element fallback
        import math
        return np.vectorize(math.erf, otypes=[np.float64])(x)


def gelu(x: np.ndarray) -> np.ndarray:
    """Exact GELU: x * Phi(x) = x/2 * (1 + erf(x / sqrt(2)))."""
    x = np.asarray(x, dtype=np.float64)
    return 0.5 * x * (1.0 + _erf(x / np.sqrt(2.0)))


def relu(x: np.ndarray) -> np.ndarray:
    """max(x, 0)."""
    return np.maximum(np.asarray(x), 0.0)


# gate activation of the gated MLP, by name: SwiGLU, GeGLU, ReGLU
ACTIVATIONS = {"silu": silu, "gelu": gelu, "relu": relu}


def expert_mlp(x: np.ndarray, w_gate_up_e: np.ndarray, w_down_e: np.ndarray,
               dtype=np.float64, act: str = "silu") -> np.ndarray:
    """One expert's gated MLP on rows x [M, H]: g = x Wg^T, u = x Wu^T,
    h = act(g) * u, y = h Wd^T.  Returns y [M, H] in ``dtype``."""
    I = w_gate_up_e.shape[0] // 2
    x = np.asarray(x, dtype=dtype)
    wg = np.asarray(w_gate_up_e[:I], dtype=dtype)
    wu = np.asarray(w_gate_up_e[I:], dtype=dtype)
    wd = np.asarray(w_down_e, dtype=dtype)
    g = x @ wg.T
    u = x @ wu.T
    h = ACTIVATIONS[act](g) * u
    return h @ wd.T


def forward(hidden: np.ndarray, topk_idx: np.ndarray, topk_w: np.ndarray,
            w_gate_up: np.ndarray, w_down: np.ndarray, dtype=np.float64,
            round_h_bf16: bool = False, act: str = "silu") -> np.ndarray:
    """Eager loop over experts (the "eager" backend's plain form).

    hidden [T,H], w_gate_up [E,2I,H], w_down [E,H,I] as float arrays holding
    the bf16 values; topk_idx [T,k]; topk_w [T,k].  Returns the un-rounded
    output [T,H] in ``dtype``; apply round_to_bf16 for the stored output.
    ``round_h_bf16`` rounds the intermediate h to bf16 (diagnostic only);
    ``act`` names the gate activation (silu, gelu or relu)."""
    T, H = hidden.shape
    E = w_gate_up.shape[0]
    k = topk_idx.shape[1]
    I = w_gate_up.shape[1] // 2
    counts, offsets, sorted_f, _ = dispatch(topk_idx, E)
    w = np.asarray(topk_w, dtype=dtype)
    out = np.zeros((T, H), dtype=dtype)
    for e in range(E):
        if counts[e] == 0:
            continue
        rows = sorted_f[offsets[e]:offsets[e + 1]].astype(np.int64)
        toks = rows // k
        slots = rows % k
        x = np.asarray(hidden[toks], dtype=dtype)
        wg = np.asarray(w_gate_up[e, :I], dtype=dtype)
        wu = np.asarray(w_gate_up[e, I:], dtype=dtype)
        g = x @ wg.T
        u = x @ wu.T
        h = ACTIVATIONS[act](g) * u
        if round_h_bf16:
            h = round_to_bf16(h).astype(dtype)
        y = h @ np.asarray(w_down[e], dtype=dtype).T
        np.add.at(out, toks, w[toks, slots][:, None] * y)
    return out


def forward_brute(hidden, topk_idx, topk_w, w_gate_up, w_down, act: str = "silu") -> np.ndarray:
    """Float64 loop over (token, slot) with explicit dot products, no
    dispatch and no batching; for tiny inputs only."""
    T, H = hidden.shape
    k = topk_idx.shape[1]
    I = w_gate_up.shape[1] // 2
    out = np.zeros((T, H), dtype=np.float64)
    for t in range(T):
        x = np.asarray(hidden[t], dtype=np.float64)
        for j in range(k):
            e = int(topk_idx[t, j])
            h = np.empty(I, dtype=np.float64)
            for i in range(I):
                g = float(np.dot(x, np.asarray(w_gate_up[e, i], np.float64)))
                u = float(np.dot(x, np.asarray(w_gate_up[e, I + i], np.float64)))
                if act == "silu":
                    s = g / (1.0 + np.exp(-g)) if g >= 0 else g * np.exp(g) / (1.0 + np.exp(g))
                elif act == "gelu":
                    import math
                    s = 0.5 * g * (1.0 + math.erf(g / math.sqrt(2.0)))
                else:
                    s = g if g > 0 else 0.0
                h[i] = s * u
            for c in range(H):
                out[t, c] += float(topk_w[t, j]) * float(
                    np.dot(h, np.asarray(w_down[e, c], np.float64)))
    return out


# --------------------------------------------------------------------------
# FP8 e4m3 block quantisation (float32 or UE8M0 scales; dynamic per-row
# activation scales)
# --------------------------------------------------------------------------

E4M3_MAX = 448.0


def e4m3_encode(x: np.ndarray) -> np.ndarray:
    """fp32 -> e4m3fn codes (uint8), round to nearest even, saturating to
    +-448 (no infinities in e4m3fn).  NaN maps to 0x7F/0xFF."""
    x = np.asarray(x, dtype=np.float32)
    sign = (x.view(np.uint32) >> np.uint32(31)).astype(np.uint8) << np.uint8(7)
    a = np.abs(x).astype(np.float64)
    code = np.zeros(x.shape, dtype=np.uint8)
    nz = a > 0
    av = a[nz]
    _, ex = np.frexp(av)                 # av = m * 2**ex, 0.5 <= m < 1
    e_unb = np.maximum(ex - 1, -6)       # floor(log2 av), clamped to min normal
    quantum = np.ldexp(1.0, e_unb - 3)   # spacing of 3 mantissa bits
    n = np.rint(av / quantum)            # exact division; rint is ties-to-even
    val = n * quantum
    val = np.minimum(val, E4M3_MAX)      # satfinite
    c = np.zeros(av.shape, dtype=np.int64)
    sub = val < 2.0 ** -6
    c[sub] = np.rint(val[sub] * 2.0 ** 9).astype(np.int64)
    nrm = ~sub
    _, ve = np.frexp(val[nrm])
    e_field = (ve - 1) + 7
    mant = np.rint((val[nrm] / np.ldexp(1.0, ve - 1) - 1.0) * 8.0).astype(np.int64)
    c[nrm] = (e_field.astype(np.int64) << 3) | mant
    code[nz] = c.astype(np.uint8)
    code = code | sign
    nan = np.isnan(x)
    code[nan] = sign[nan] | np.uint8(0x7F)
    return code


def e4m3_decode(code: np.ndarray) -> np.ndarray:
    """e4m3fn codes -> float32 values."""
    c = np.asarray(code, dtype=np.uint8).astype(np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    val = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.ldexp(1.0, e - 7))
    val = s * val
    val = np.where((e == 15) & (m == 7), np.nan, val)
    return val.astype(np.float32)


def ue8m0_from_quotient(v: np.ndarray):
    """Smallest power of two >= v (v > 0, fp32), read from v's bits.
    Returns (scale float32, biased exponent byte uint8 with s = 2**(b-127))."""
    v = np.asarray(v, dtype=np.float32)
    bits = v.view(np.uint32)
    ex = ((bits >> np.uint32(23)) & np.uint32(0xFF)).astype(np.int64)
    mant = (bits & np.uint32(0x7FFFFF)).astype(np.int64)
    b = ex + (mant != 0)
    b = np.clip(b, 0, 254)
    s = np.ldexp(np.float32(1.0), (b - 127).astype(np.int32)).astype(np.float32)
    return s, b.astype(np.uint8)


def _block_scales(amax: np.ndarray, fmt: str):
    amax = np.asarray(amax, dtype=np.float32)
    zero = amax == 0
    q = (amax / np.float32(E4M3_MAX)).astype(np.float32)     # fp32 IEEE division
    if fmt == "f32":
        s = q
        s = np.where(zero, np.float32(1.0), s).astype(np.float32)
        return s, s.copy()
    if fmt == "ue8m0":
        s, b = ue8m0_from_quotient(np.where(zero, np.float32(1.0), q))
        s = np.where(zero, np.float32(1.0), s).astype(np.float32)
        b = np.where(zero, np.uint8(127), b).astype(np.uint8)
        return s, b
    raise ValueError("fmt must be 'f32' or 'ue8m0'")


def quantize_blocks(x: np.ndarray, block_rows: int, block_cols: int, fmt: str):
    """Block quantisation of x [..., R, C] (float32 values) into e4m3 codes.

    Blocks are block_rows x block_cols over the last two axes (128x128 for
    weights, 1x128 for activations).  Returns (codes uint8 [..., R, C],
    stored scales [..., R/br, C/bc]: float32 for 'f32', uint8 exponent bytes
    for 'ue8m0', scale values float32 [..., R/br, C/bc])."""
    x = np.asarray(x, dtype=np.float32)
    *lead, R, C = x.shape
    if R % block_rows or C % block_cols:
        raise ValueError("shape not divisible by the block size")
    nb_r, nb_c = R // block_rows, C // block_cols
    xb = x.reshape(*lead, nb_r, block_rows, nb_c, block_cols)
    amax = np.abs(xb).max(axis=(-3, -1))
    s, stored = _block_scales(amax, fmt)
    inv = (np.float32(1.0) / s).astype(np.float32)           # fp32 IEEE division
    y = (xb * inv[..., :, None, :, None]).astype(np.float32)  # fp32 product
    codes = e4m3_encode(y).reshape(*lead, R, C)
    return codes, stored, s


def dequantize_blocks(codes: np.ndarray, scales: np.ndarray, block_rows: int,
                      block_cols: int, dtype=np.float64) -> np.ndarray:
    """codes [..., R, C] with scale values [..., R/br, C/bc] -> values."""
    v = e4m3_decode(codes).astype(dtype)
    s = np.asarray(scales, dtype=dtype)
    s = np.repeat(np.repeat(s, block_rows, axis=-2), block_cols, axis=-1)
    return v * s


def scale_values(stored: np.ndarray, fmt: str) -> np.ndarray:
    """Stored scales -> float32 scale values."""
    if fmt == "f32":
        return np.asarray(stored, dtype=np.float32)
    b = np.asarray(stored, dtype=np.uint8).astype(np.int32)
    return np.ldexp(np.float32(1.0), b - 127).astype(np.float32)


def requantize_rows(x: np.ndarray, block: int, fmt: str) -> np.ndarray:
    """Dynamic activation quantisation ("FP8 and FP4 quantized experts"
    section: activation scales are computed on the fly, per row): each row of
    x [M, C] (taken as fp32) is cut into 1 x block blocks along C, quantised
    to e4m3 codes with the block's scale in ``fmt`` and returned as the
    dequantised values (float64)."""
    q, _, s = quantize_blocks(np.asarray(x, dtype=np.float32), 1, block, fmt)
    return dequantize_blocks(q, s, 1, block)


def forward_fp8(hidden, topk_idx, topk_w, wq_gate_up, ws_gate_up, wq_down,
                ws_down, fmt: str, quantize_act: bool = True,
                quantize_h: bool = True, act: str = "silu") -> np.ndarray:
    """FP8 block-scaled forward, mirrored: the same dequantised weights and
    the same dynamic 1x128 activation quantisation as the device path, math
    in float64 otherwise.  wq_* are e4m3 codes, ws_* stored scales (fp32 or
    UE8M0 bytes) of 128x128 blocks.  Returns the un-rounded output [T,H]."""
    T, H = hidden.shape
    E = wq_gate_up.shape[0]
    k = topk_idx.shape[1]
    I = wq_gate_up.shape[1] // 2
    wgu = dequantize_blocks(wq_gate_up, scale_values(ws_gate_up, fmt), 128, 128)
    wd = dequantize_blocks(wq_down, scale_values(ws_down, fmt), 128, 128)
    counts, offsets, sorted_f, _ = dispatch(topk_idx, E)
    w = np.asarray(topk_w, dtype=np.float64)
    out = np.zeros((T, H), dtype=np.float64)
    for e in range(E):
        if counts[e] == 0:
            continue
        rows = sorted_f[offsets[e]:offsets[e + 1]].astype(np.int64)
        toks = rows // k
        slots = rows % k
        x = np.asarray(hidden[toks], dtype=np.float32)
        x = requantize_rows(x, 128, fmt) if quantize_act else x.astype(np.float64)
        g = x @ wgu[e, :I].T
        u = x @ wgu[e, I:].T
        h = ACTIVATIONS[act](g) * u
        if quantize_h:
            h = requantize_rows(h, 128, fmt)
        y = h @ wd[e].T
        np.add.at(out, toks, w[toks, slots][:, None] * y)
    return out


# --------------------------------------------------------------------------
# FP4 (e2m1) experts.  The page ("FP8 and FP4 quantized experts"; the
# paragraph after the backends table) fixes only e2m1 codes packed in int8
# with UE8M0 weight scales.  Readings: blocks of 1x32 along the contraction
# axis (the MX convention; the page gives no size); scale = the smallest
# power of two >= amax/6 (amax = 0 gives 1), as for FP8 with 6 in place of
# 448; codes e2m1(x * (1/s)), round to nearest even, saturating to +-6; two
# codes per byte, the even element in the low nibble.  The activations and
# h of an FP4 forward are e4m3 with the same 1x32 UE8M0 blocks.
# --------------------------------------------------------------------------

E2M1_MAX = 6.0
# magnitudes of the codes 0..7 (bit 3 is the sign): 0, then 2^(e-1)(1 + m/2)
_E2M1_MAG = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def e2m1_decode(code: np.ndarray) -> np.ndarray:
    """e2m1 codes (0..15, bit 3 = sign) -> float32 values."""
    c = np.asarray(code, dtype=np.uint8).astype(np.int64)
    mag = _E2M1_MAG[c & 7]
    return np.where(c & 8, -mag, mag).astype(np.float32)


def e2m1_encode(x: np.ndarray) -> np.ndarray:
    """fp32 -> e2m1 codes (uint8 0..15): the nearest of the eight magnitudes,
    ties to the even code (mantissa bit 0), magnitudes above 6 saturate to
    6; the sign bit is x's sign bit (so -0.0 -> 8)."""
    x = np.asarray(x, dtype=np.float32)
    a = np.abs(x).astype(np.float64)
    hi = np.clip(np.searchsorted(_E2M1_MAG, a, side="left"), 1, 7)   # first magnitude >= a
    lo = hi - 1
    d_lo = a - _E2M1_MAG[lo]
    d_hi = _E2M1_MAG[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    mag = np.where(pick_hi, hi, lo)
    mag = np.where(a >= E2M1_MAX, 7, mag)
    sign = (x.view(np.uint32) >> np.uint32(31)).astype(np.int64)
    return (mag | (sign << 3)).astype(np.uint8)


def pack_e2m1(codes: np.ndarray) -> np.ndarray:
    """codes [..., C] (C even) -> bytes [..., C/2], element 2i in the low nibble."""
    c = np.asarray(codes, dtype=np.uint8)
    return (c[..., 0::2] | (c[..., 1::2] << np.uint8(4))).astype(np.uint8)


def unpack_e2m1(packed: np.ndarray) -> np.ndarray:
    """bytes [..., C/2] -> codes [..., C]."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = p & np.uint8(0xF)
    out[..., 1::2] = p >> np.uint8(4)
    return out


def _ue8m0_block_scales(amax: np.ndarray, elem_max: float):
    amax = np.asarray(amax, dtype=np.float32)
    zero = amax == 0
    q = (amax / np.float32(elem_max)).astype(np.float32)      # fp32 IEEE division
    s, b = ue8m0_from_quotient(np.where(zero, np.float32(1.0), q))
    s = np.where(zero, np.float32(1.0), s).astype(np.float32)
    b = np.where(zero, np.uint8(127), b).astype(np.uint8)
    return s, b


def quantize_fp4_blocks(x: np.ndarray, block: int = 32):
    """x [..., C] (float32 values) -> (packed e2m1 bytes [..., C/2], UE8M0
    exponent bytes [..., C/block], scale values float32 [..., C/block])."""
    x = np.asarray(x, dtype=np.float32)
    *lead, C = x.shape
    if C % block or block % 2:
        raise ValueError("last axis not divisible by the block size")
    xb = x.reshape(*lead, C // block, block)
    s, b = _ue8m0_block_scales(np.abs(xb).max(axis=-1), E2M1_MAX)
    y = (xb * (np.float32(1.0) / s)[..., None]).astype(np.float32)   # exact: s is 2^j
    codes = e2m1_encode(y).reshape(*lead, C)
    return pack_e2m1(codes), b, s


def dequantize_fp4_blocks(packed: np.ndarray, scales: np.ndarray, block: int = 32,
                          dtype=np.float64) -> np.ndarray:
    """packed e2m1 bytes [..., C/2] with scale values [..., C/block] -> values."""
    v = e2m1_decode(unpack_e2m1(packed)).astype(dtype)
    return v * np.repeat(np.asarray(scales, dtype=dtype), block, axis=-1)


def forward_fp4(hidden, topk_idx, topk_w, wq_gate_up, ws_gate_up, wq_down, ws_down,
                block: int = 32, quantize_act: bool = True, quantize_h: bool = True,
                act: str = "silu") -> np.ndarray:
    """FP4-weight forward, mirrored: weights are packed e2m1 [E, 2I, H/2] and
    [E, H, I/2] with UE8M0 exponent bytes [E, 2I, H/block] and [E, H, I/block];
    the hidden rows and h are quantised to e4m3 in 1 x block UE8M0 blocks;
    math in float64 otherwise.  Returns the un-rounded output [T,H]."""
    T, H = hidden.shape
    E = wq_gate_up.shape[0]
    k = topk_idx.shape[1]
    I = wq_gate_up.shape[1] // 2
    wgu = dequantize_fp4_blocks(wq_gate_up, scale_values(ws_gate_up, "ue8m0"), block)
    wd = dequantize_fp4_blocks(wq_down, scale_values(ws_down, "ue8m0"), block)
    counts, offsets, sorted_f, _ = dispatch(topk_idx, E)
    w = np.asarray(topk_w, dtype=np.float64)
    out = np.zeros((T, H), dtype=np.float64)
    for e in range(E):
        if counts[e] == 0:
            continue
        rows = sorted_f[offsets[e]:offsets[e + 1]].astype(np.int64)
        toks = rows // k
        slots = rows % k
        x = np.asarray(hidden[toks], dtype=np.float32)
        x = requantize_rows(x, block, "ue8m0") if quantize_act else x.astype(np.float64)
        g = x @ wgu[e, :I].T
        u = x @ wgu[e, I:].T
        h = ACTIVATIONS[act](g) * u
        if quantize_h:
            h = requantize_rows(h, block, "ue8m0")
        y = h @ wd[e].T
        np.add.at(out, toks, w[toks, slots][:, None] * y)
    return out


# --------------------------------------------------------------------------
# Metrics used by the parity tests and the benchmark
# --------------------------------------------------------------------------

def rel_max_err(out: np.ndarray, ref: np.ndarray) -> float:
    """max |out - ref| / rms(ref), computed in float64."""
    o = np.asarray(out, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    rms = float(np.sqrt(np.mean(r * r)))
    if rms == 0.0:
        return float(np.max(np.abs(o - r))) if o.size else 0.0
    return float(np.max(np.abs(o - r))) / rms


def touched_weight_bytes(counts: np.ndarray, H: int, I: int,
                         bytes_per_weight: float, scale_bytes_per_expert: int = 0) -> int:
    """Weight bytes of the experts that received at least one row."""
    touched = int(np.count_nonzero(np.asarray(counts) > 0))
    return int(touched * (3 * H * I * bytes_per_weight + scale_bytes_per_expert))
