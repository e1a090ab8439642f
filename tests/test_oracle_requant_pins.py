"""Pins for the oracle's dynamic activation re-quantisation steps: the 1x128
e4m3 quantisation of the hidden rows and of h in the FP8 forward, and the
1x32 e4m3 quantisation of both in the FP4 forward.

Three kinds of checks tie these steps to something other than the oracle:

* a scalar brute force written from the format definitions alone (the e4m3
  and e2m1 value tables built from sign/exponent/mantissa fields, the
  nearest code found by search, the UE8M0 scale from math.frexp, one block
  and one element at a time, a plain loop per (token, slot));
* hand-derived cases under tests/golden/ whose expected outputs follow from
  the block arithmetic written out in the fixture;
* the same comparisons with a deliberate mistake planted in the oracle (on
  the CPU, through monkeypatch): a transposed block, a wrong block size or
  the other scale format must each make a pin fail.

Source: Hugging Face Transformers "Experts backends" page, "FP8 and FP4
quantized experts" section (dynamic per-row activation scales; FP4 weights
with UE8M0 scales) and the paragraph after the backends table (float32 or
UE8M0 block scales, FP4 packed in int8).
"""
import bisect
import json
import math
import os

import numpy as np
import pytest

import oracle as O
from oracle import moe_oracle as OM

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------
# number formats from their field definitions
# --------------------------------------------------------------------------

def _e4m3_value(c):
    """e4m3fn code -> value: sign bit 7, exponent bits 6..3 (bias 7), mantissa
    bits 2..0; exponent 0 is subnormal (m * 2^-9); 0x7F / 0xFF are NaN."""
    s = -1.0 if c & 0x80 else 1.0
    e, m = (c >> 3) & 0xF, c & 0x7
    if e == 15 and m == 7:
        return math.nan
    return s * (m * 2.0 ** -9 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7))


_E4M3_POS = [_e4m3_value(c) for c in range(0x7F)]      # codes 0..126, ascending values


def _e4m3_nearest(y):
    """Nearest e4m3fn code to the float y by search over the finite
    magnitudes, ties to the even code, magnitudes above 448 saturating."""
    a = min(abs(y), 448.0)
    i = bisect.bisect_left(_E4M3_POS, a)
    if i == 0:
        c = 0
    elif i == len(_E4M3_POS):
        c = len(_E4M3_POS) - 1
    else:
        lo, hi = i - 1, i
        dl, dh = a - _E4M3_POS[lo], _E4M3_POS[hi] - a
        c = hi if (dh < dl or (dh == dl and hi % 2 == 0)) else lo
    neg = math.copysign(1.0, y) < 0
    return c | (0x80 if neg else 0)


_E2M1_MAG = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _e2m1_value(c):
    """e2m1 code -> value: sign bit 3, exponent bits 2..1 (bias 1), mantissa
    bit 0; exponent 0 is subnormal (m * 0.5)."""
    e, m = (c >> 1) & 3, c & 1
    mag = m * 0.5 if e == 0 else (1.0 + m / 2.0) * 2.0 ** (e - 1)
    return -mag if c & 8 else mag


def _pow2_ceil(q):
    """Smallest power of two >= q > 0 (q an fp32 value, exact through frexp)."""
    m, e = math.frexp(float(q))
    return 2.0 ** (e - 1) if m == 0.5 else 2.0 ** e


def _block_scale(amax, fmt):
    """Scale of one block: amax/448 by fp32 division, or its power-of-two
    ceiling; an all-zero block has scale 1."""
    if amax == 0.0:
        return 1.0
    q = np.float32(amax) / np.float32(448.0)
    return float(q) if fmt == "f32" else _pow2_ceil(q)


def _quant_row(row, block, fmt):
    """Quantise one row in 1 x block blocks: per block the scale from its
    absolute maximum, then e4m3(x * (1/s)) with the reciprocal and product in
    fp32, then dequantised (code value * s)."""
    out = []
    for b0 in range(0, len(row), block):
        blk = [float(np.float32(v)) for v in row[b0:b0 + block]]
        s = _block_scale(max(abs(v) for v in blk), fmt)
        inv = np.float32(1.0) / np.float32(s)
        for v in blk:
            out.append(_e4m3_value(_e4m3_nearest(float(np.float32(v) * inv))) * s)
    return out


def _act(g, act):
    if act == "silu":
        return g / (1.0 + math.exp(-g)) if g >= 0 else g * math.exp(g) / (1.0 + math.exp(g))
    if act == "gelu":
        return 0.5 * g * (1.0 + math.erf(g / math.sqrt(2.0)))
    return max(g, 0.0)


def _forward_scalar(hidden, idx, w, deq_gu, deq_d, block, fmt, act):
    """Routed forward, one (token, slot) at a time: quantise the token's row,
    gate/up dot products, activation, quantise h, down dot products, add
    w * y into the token's output.  deq_gu[e][r][c] / deq_d[e][r][c] are the
    dequantised weights as nested lists."""
    T, H = len(hidden), len(hidden[0])
    k = len(idx[0])
    out = [[0.0] * H for _ in range(T)]
    for t in range(T):
        xq = _quant_row(hidden[t], block, fmt)
        for j in range(k):
            e = idx[t][j]
            wgu, wd = deq_gu[e], deq_d[e]
            I = len(wgu) // 2
            h = []
            for i in range(I):
                g = sum(a * b for a, b in zip(xq, wgu[i]))
                u = sum(a * b for a, b in zip(xq, wgu[I + i]))
                h.append(_act(g, act) * u)
            hq = _quant_row(h, block, fmt)
            for c in range(H):
                out[t][c] += w[t][j] * sum(a * b for a, b in zip(hq, wd[c]))
    return np.array(out)


def _deq_fp8(codes, stored, fmt):
    """e4m3 weight codes [E, R, C] with 128x128 block scales -> nested lists."""
    E, R, C = codes.shape
    res = []
    for e in range(E):
        m = []
        for r in range(R):
            row = []
            for c in range(C):
                sb = stored[e, r // 128, c // 128]
                s = float(sb) if fmt == "f32" else math.ldexp(1.0, int(sb) - 127)
                row.append(_e4m3_value(int(codes[e, r, c])) * s)
            m.append(row)
        res.append(m)
    return res


def _deq_fp4(packed, scale_bytes):
    """Packed e2m1 weights [E, R, C/2] (even element in the low nibble) with
    one UE8M0 byte per 1x32 block [E, R, C/32] -> nested lists."""
    E, R, C2 = packed.shape
    res = []
    for e in range(E):
        m = []
        for r in range(R):
            row = []
            for c in range(2 * C2):
                byte = int(packed[e, r, c // 2])
                code = byte & 0xF if c % 2 == 0 else byte >> 4
                row.append(_e2m1_value(code) * math.ldexp(1.0, int(scale_bytes[e, r, c // 32]) - 127))
            m.append(row)
        res.append(m)
    return res


# --------------------------------------------------------------------------
# the brute force itself, against closed forms
# --------------------------------------------------------------------------

def test_scalar_formats_against_closed_forms():
    assert _e4m3_value(0x38) == 1.0 and _e4m3_value(0x7E) == 448.0
    assert _e4m3_value(0x01) == 2.0 ** -9 and _e4m3_value(0x08) == 2.0 ** -6
    assert _e4m3_nearest(1.5 * 2 ** -9) == 0x02          # tie -> even code
    assert _e4m3_nearest(2.5 * 2 ** -9) == 0x02
    assert _e4m3_nearest(1e6) == 0x7E and _e4m3_nearest(-1e6) == 0xFE
    assert [_e2m1_value(c) for c in range(8)] == _E2M1_MAG
    assert _pow2_ceil(np.float32(1.0)) == 1.0 and _pow2_ceil(np.float32(0.3)) == 0.5
    assert _block_scale(24.0, "ue8m0") == 2.0 ** -4


# --------------------------------------------------------------------------
# FP8: brute force on random inputs, both scale formats, three activations
# --------------------------------------------------------------------------

def _fp8_case(fmt, seed):
    rng = np.random.default_rng(seed)
    T, H, I, E, k = 3, 256, 256, 3, 2
    hid = (rng.standard_normal((T, H)) * np.exp(rng.uniform(-3, 3, (T, 1)))).astype(np.float32)
    # the two 1x128 blocks of a row differ in range by about 2^12, and so do
    # the two blocks of h (through the up rows of features 128..255): a block
    # of the wrong size or axis then pushes the smaller values into other
    # (often subnormal) e4m3 codes
    # (and a quarter of block 0 differs from the rest of it the same way,
    # so that too small a block shows as well)
    hid[:, 128:] *= np.float32(2.0 ** -12)
    hid[:, 32:64] *= np.float32(2.0 ** -12)
    hid[1, 7] = 0.0
    wgu = (rng.standard_normal((E, 2 * I, H)) * 0.05).astype(np.float32)
    wgu[:, I + 128:, :] *= np.float32(2.0 ** -10)
    wgu[:, I + 32:I + 64, :] *= np.float32(2.0 ** -10)
    wd = (rng.standard_normal((E, H, I)) * 0.05).astype(np.float32)
    wd[:, :, :128] *= np.float32(3.0)
    qgu, sgu, _ = O.quantize_blocks(wgu, 128, 128, fmt)
    qd, sd, _ = O.quantize_blocks(wd, 128, 128, fmt)
    idx = np.array([[0, 2], [1, 0], [2, 1]], np.int32)
    w = np.array([[0.625, 0.375], [0.5, 0.5], [0.875, 0.125]])
    return hid, idx, w, qgu, sgu, qd, sd


@pytest.mark.parametrize("fmt,act,seed", [("ue8m0", "silu", 0), ("f32", "silu", 1),
                                          ("ue8m0", "gelu", 2), ("f32", "relu", 3)])
def test_fp8_forward_matches_scalar_brute_force(fmt, act, seed):
    hid, idx, w, qgu, sgu, qd, sd = _fp8_case(fmt, seed)
    got = O.forward_fp8(hid, idx, w, qgu, sgu, qd, sd, fmt, act=act)
    want = _forward_scalar(hid.tolist(), idx.tolist(), w.tolist(), _deq_fp8(qgu, sgu, fmt),
                           _deq_fp8(qd, sd, fmt), 128, fmt, act)
    np.testing.assert_allclose(got, want, rtol=1e-9, atol=1e-12 * np.abs(want).max())


# --------------------------------------------------------------------------
# FP4: brute force on random inputs, three activations
# --------------------------------------------------------------------------

def _fp4_case(seed):
    rng = np.random.default_rng(seed)
    T, H, I, E, k = 4, 64, 96, 3, 2
    hid = (rng.standard_normal((T, H)) * np.exp(rng.uniform(-3, 3, (T, 1)))).astype(np.float32)
    # the 1x32 blocks of a row, and blocks 0 and 1 of h, differ in range by
    # about 2^12 and 2^10 (see the FP8 case)
    hid[:, 32:] *= np.float32(2.0 ** -12)
    hid[:, 8:16] *= np.float32(2.0 ** -12)
    wgu = (rng.standard_normal((E, 2 * I, H)) * 0.05).astype(np.float32)
    wgu[:, I + 32:I + 64, :] *= np.float32(2.0 ** -10)
    wgu[:, I + 8:I + 16, :] *= np.float32(2.0 ** -10)
    wd = (rng.standard_normal((E, H, I)) * 0.05).astype(np.float32)
    wd[:, :, 64:] *= np.float32(1e-2)
    qgu, bgu, _ = O.quantize_fp4_blocks(wgu, 32)
    qd, bd, _ = O.quantize_fp4_blocks(wd, 32)
    idx = np.array([[0, 2], [1, 0], [2, 1], [1, 2]], np.int32)
    w = np.array([[0.625, 0.375], [0.5, 0.5], [0.875, 0.125], [0.25, 0.75]])
    return hid, idx, w, qgu, bgu, qd, bd


@pytest.mark.parametrize("act,seed", [("silu", 0), ("gelu", 1), ("relu", 2)])
def test_fp4_forward_matches_scalar_brute_force(act, seed):
    hid, idx, w, qgu, bgu, qd, bd = _fp4_case(seed)
    got = O.forward_fp4(hid, idx, w, qgu, bgu, qd, bd, 32, act=act)
    want = _forward_scalar(hid.tolist(), idx.tolist(), w.tolist(), _deq_fp4(qgu, bgu),
                           _deq_fp4(qd, bd), 32, "ue8m0", act)
    np.testing.assert_allclose(got, want, rtol=1e-9, atol=1e-12 * np.abs(want).max())


# --------------------------------------------------------------------------
# hand-derived cases (tests/golden/)
# --------------------------------------------------------------------------

def _golden(name):
    return json.load(open(os.path.join(GOLDEN, name)))


def _fp8_golden_inputs(fx):
    T, H, I, E = fx["T"], fx["H"], fx["I"], fx["E"]
    hid = np.zeros((T, H), np.float32)
    for c, v in fx["hidden"]:
        hid[0, c] = v
    qgu = np.zeros((E, 2 * I, H), np.uint8)
    for r, c, code in fx["w_gate_codes"]:
        qgu[0, r, c] = code
    for r, c, code in fx["w_up_codes"]:
        qgu[0, I + r, c] = code
    sgu = np.full((E, 2 * I // 128, H // 128), 127, np.uint8)
    for rb, cb, b in fx["w_up_scale_bytes"]:
        sgu[0, I // 128 + rb, cb] = b
    qd = np.zeros((E, H, I), np.uint8)
    for c in range(min(H, I)):
        qd[0, c, c] = fx["w_down_identity_code"]
    sd = np.full((E, H // 128, I // 128), 127, np.uint8)
    idx = np.zeros((T, 1), np.int32)
    w = np.ones((T, 1))
    return hid, idx, w, qgu, sgu, qd, sd


def _fp4_golden_inputs(fx):
    T, H, I, E, blk = fx["T"], fx["H"], fx["I"], fx["E"], fx["block"]
    hid = np.zeros((T, H), np.float32)
    for c, v in fx["hidden"]:
        hid[0, c] = v
    codes = np.zeros((E, 2 * I, H), np.uint8)
    sgu = np.full((E, 2 * I, H // blk), 127, np.uint8)
    for r, c, code, b in fx["w_gate_entries"]:
        codes[0, r, c] = code
        sgu[0, r, c // blk] = b
    for r, c, code, b in fx["w_up_entries"]:
        codes[0, I + r, c] = code
        sgu[0, I + r, c // blk] = b
    cd = np.zeros((E, H, I), np.uint8)
    for c in range(min(H, I)):
        cd[0, c, c] = fx["w_down_identity_code"]
    pack = lambda a: (a[..., 0::2] | (a[..., 1::2] << 4)).astype(np.uint8)
    sd = np.full((E, H, I // blk), 127, np.uint8)
    return hid, np.zeros((T, 1), np.int32), np.ones((T, 1)), pack(codes), sgu, pack(cd), sd


def _dense_expect(fx, H):
    want = np.zeros((fx["T"], H))
    for c, v in fx["expect_out"]:
        want[0, c] = v
    return want


def test_fp8_requant_golden():
    fx = _golden("fp8_requant_1x128_ue8m0.json")
    out = O.forward_fp8(*_fp8_golden_inputs(fx), fx["fmt"], act=fx["act"])
    np.testing.assert_array_equal(out, _dense_expect(fx, fx["H"]))


def test_fp4_requant_golden():
    fx = _golden("fp4_requant_1x32_ue8m0.json")
    out = O.forward_fp4(*_fp4_golden_inputs(fx), fx["block"], act=fx["act"])
    np.testing.assert_array_equal(out, _dense_expect(fx, fx["H"]))


def test_golden_inputs_agree_with_the_scalar_brute_force():
    """The fixtures' inputs through the scalar path give the same outputs as
    written in the fixtures (so the derivations are checked twice)."""
    fx = _golden("fp8_requant_1x128_ue8m0.json")
    hid, idx, w, qgu, sgu, qd, sd = _fp8_golden_inputs(fx)
    got = _forward_scalar(hid.tolist(), idx.tolist(), w.tolist(), _deq_fp8(qgu, sgu, "ue8m0"),
                          _deq_fp8(qd, sd, "ue8m0"), 128, "ue8m0", fx["act"])
    np.testing.assert_array_equal(got, _dense_expect(fx, fx["H"]))
    fx = _golden("fp4_requant_1x32_ue8m0.json")
    hid, idx, w, qgu, sgu, qd, sd = _fp4_golden_inputs(fx)
    got = _forward_scalar(hid.tolist(), idx.tolist(), w.tolist(), _deq_fp4(qgu, sgu),
                          _deq_fp4(qd, sd), 32, "ue8m0", fx["act"])
    np.testing.assert_array_equal(got, _dense_expect(fx, fx["H"]))


# --------------------------------------------------------------------------
# planted mistakes: every pin above must catch each of them
# --------------------------------------------------------------------------

def _mistake(kind, real):
    """A wrong version of the oracle's row re-quantisation step."""
    def wrong(x, block, fmt):
        x = np.asarray(x, dtype=np.float32)
        if kind == "token_axis":            # blocks along the token axis
            n = x.shape[0]
            xp = np.concatenate([x, np.zeros(((-n) % block, x.shape[1]), np.float32)])
            return real(xp.T, block, fmt).T[:n]
        if kind == "quarter_block":
            return real(x, block // 4, fmt)
        if kind == "double_block":
            b = 2 * block if x.shape[1] % (2 * block) == 0 else x.shape[1]
            return real(x, b, fmt)
        if kind == "other_format":
            return real(x, block, "f32" if fmt == "ue8m0" else "ue8m0")
        raise ValueError(kind)
    return wrong


MISTAKES = ["token_axis", "quarter_block", "double_block", "other_format"]


@pytest.mark.parametrize("kind", MISTAKES)
def test_planted_mistakes_are_caught_fp8(monkeypatch, kind):
    real = OM.requantize_rows
    # the brute force is computed before the mistake is planted
    hid, idx, w, qgu, sgu, qd, sd = _fp8_case("ue8m0", 0)
    want = _forward_scalar(hid.tolist(), idx.tolist(), w.tolist(), _deq_fp8(qgu, sgu, "ue8m0"),
                           _deq_fp8(qd, sd, "ue8m0"), 128, "ue8m0", "silu")
    fx = _golden("fp8_requant_1x128_ue8m0.json")
    monkeypatch.setattr(OM, "requantize_rows", _mistake(kind, real))
    got = O.forward_fp8(hid, idx, w, qgu, sgu, qd, sd, "ue8m0")
    assert not np.allclose(got, want, rtol=1e-9, atol=1e-12 * np.abs(want).max())
    gold = O.forward_fp8(*_fp8_golden_inputs(fx), fx["fmt"], act=fx["act"])
    assert not np.array_equal(gold, _dense_expect(fx, fx["H"]))


@pytest.mark.parametrize("kind", MISTAKES)
def test_planted_mistakes_are_caught_fp4(monkeypatch, kind):
    real = OM.requantize_rows
    hid, idx, w, qgu, bgu, qd, bd = _fp4_case(0)
    want = _forward_scalar(hid.tolist(), idx.tolist(), w.tolist(), _deq_fp4(qgu, bgu),
                           _deq_fp4(qd, bd), 32, "ue8m0", "silu")
    fx = _golden("fp4_requant_1x32_ue8m0.json")
    monkeypatch.setattr(OM, "requantize_rows", _mistake(kind, real))
    got = O.forward_fp4(hid, idx, w, qgu, bgu, qd, bd, 32)
    assert not np.allclose(got, want, rtol=1e-9, atol=1e-12 * np.abs(want).max())
    gold = O.forward_fp4(*_fp4_golden_inputs(fx), fx["block"], act=fx["act"])
    assert not np.array_equal(gold, _dense_expect(fx, fx["H"]))
