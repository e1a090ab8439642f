"""Pins for the CPU oracle: each check ties the oracle to something other than
itself (a hand-derived worked example, brute force, a library routine, a
closed form or an invariant the method fixes), so that a dropped term, a wrong
sign or index or a transposed operand in the oracle fails at least one test.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle as O
from workloads import MoEShape, make_inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _np_inputs(shape, seed=0):
    d = make_inputs(shape, seed=seed, device="cpu")
    return (d["logits"].numpy(), d["hidden"].float().numpy(),
            d["w_gate_up"].float().numpy(), d["w_down"].float().numpy())


# --------------------------------------------------------------------------
# worked example with closed-form results
# --------------------------------------------------------------------------

def test_worked_example_closed_form():
    fx = json.load(open(os.path.join(GOLDEN, "worked_example_closed_form.json")))
    logits = np.array(fx["logits"], np.float32)
    idx, w = O.route(logits, fx["k"])
    assert idx.tolist() == fx["expect_topk_idx"]
    np.testing.assert_allclose(w, fx["expect_topk_w"], rtol=1e-6)
    counts, offsets, sorted_f, row_of = O.dispatch(idx, fx["E"])
    assert counts.tolist() == fx["expect_counts"]
    assert offsets.tolist() == fx["expect_offsets"]
    assert sorted_f.tolist() == fx["expect_sorted_f"]
    out = O.forward(np.array(fx["hidden"], np.float32), idx, w,
                    np.array(fx["w_gate_up"], np.float32),
                    np.array(fx["w_down"], np.float32))
    np.testing.assert_allclose(out, fx["expect_out"], rtol=1e-6)


# --------------------------------------------------------------------------
# router
# --------------------------------------------------------------------------

def _route_brute(logits, k):
    T, E = logits.shape
    idx = np.zeros((T, k), np.int32)
    for t in range(T):
        pairs = sorted(range(E), key=lambda e: (-float(logits[t, e]), e))
        idx[t] = pairs[:k]
    return idx


@pytest.mark.parametrize("T,E,k", [(17, 8, 2), (9, 60, 4), (5, 256, 8), (3, 7, 7)])
def test_route_indices_brute_force(T, E, k):
    rng = np.random.default_rng(1)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    # plant exact ties so the tie-break is exercised
    logits[:, E // 2] = logits[:, 0]
    logits[0, :] = 0.5
    idx, w = O.route(logits, k)
    assert np.array_equal(idx, _route_brute(logits, k))


def test_route_weights_two_formulas_and_sum():
    rng = np.random.default_rng(2)
    logits = (rng.standard_normal((64, 60)) * 3).astype(np.float32)
    idx, w = O.route(logits, 4)
    w2 = O.route_weights_full_softmax(logits, idx)
    np.testing.assert_allclose(w, w2, rtol=1e-12, atol=0)
    np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=1e-12)
    # slots hold descending weights
    assert np.all(np.diff(w, axis=1) <= 0)


def test_route_all_equal_and_k_equals_E():
    logits = np.full((4, 6), 1.25, np.float32)
    idx, w = O.route(logits, 3)
    assert idx.tolist() == [[0, 1, 2]] * 4
    np.testing.assert_allclose(w, 1 / 3, rtol=1e-15)
    rng = np.random.default_rng(3)
    logits = rng.standard_normal((5, 6)).astype(np.float32)
    idx, w = O.route(logits, 6)
    # k = E keeps every expert: indices are the argsort by descending logit,
    # weights the plain softmax
    assert np.array_equal(idx, np.argsort(-logits, axis=1, kind="stable"))
    p = torch.softmax(torch.from_numpy(logits).double(), dim=1).numpy()
    np.testing.assert_allclose(w, np.take_along_axis(p, idx.astype(np.int64), 1), rtol=1e-12)


def test_route_neg_inf():
    l = np.array([[-np.inf, 0.0, -np.inf, 1.0],
                  [-np.inf, -np.inf, -np.inf, -np.inf]], np.float32)
    idx, w = O.route(l, 3)
    assert idx.tolist() == [[3, 1, 0], [0, 1, 2]]
    np.testing.assert_allclose(w[0], [np.e / (1 + np.e), 1 / (1 + np.e), 0.0], rtol=1e-12)
    np.testing.assert_allclose(w[1], 1 / 3)


# --------------------------------------------------------------------------
# dispatch
# --------------------------------------------------------------------------

@pytest.mark.parametrize("T,E,k", [(64, 8, 2), (333, 60, 4), (100, 256, 8), (1, 4, 4)])
def test_dispatch_invariants_and_stable_argsort(T, E, k):
    rng = np.random.default_rng(T)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    idx, _ = O.route(logits, k)
    counts, offsets, sorted_f, row_of = O.dispatch(idx, E)
    flat = idx.reshape(-1)
    assert counts.sum() == T * k and offsets[-1] == T * k and offsets[0] == 0
    assert np.array_equal(np.diff(offsets), counts)
    assert np.array_equal(np.sort(sorted_f), np.arange(T * k))
    assert np.all(np.diff(flat[sorted_f]) >= 0)
    for e in range(E):
        seg = sorted_f[offsets[e]:offsets[e + 1]]
        assert np.all(flat[seg] == e) and np.all(np.diff(seg) > 0)
    assert np.array_equal(row_of[sorted_f], np.arange(T * k))
    # library routines: bincount and a stable argsort
    assert np.array_equal(counts, np.bincount(flat, minlength=E))
    assert np.array_equal(sorted_f, np.argsort(flat, kind="stable"))


def test_dispatch_empty_and_out_of_range():
    counts, offsets, sorted_f, row_of = O.dispatch(np.zeros((0, 2), np.int32), 4)
    assert counts.tolist() == [0] * 4 and offsets.tolist() == [0] * 5 and sorted_f.size == 0
    with pytest.raises(ValueError):
        O.dispatch(np.array([[0, 4]], np.int32), 4)


# --------------------------------------------------------------------------
# forward
# --------------------------------------------------------------------------

@pytest.mark.parametrize("act", ["silu", "gelu", "relu"])
@pytest.mark.parametrize("shape", [MoEShape(T=7, H=32, I=16, E=4, k=2),
                                   MoEShape(T=12, H=64, I=64, E=8, k=3),
                                   MoEShape(T=5, H=16, I=48, E=3, k=3)])
def test_forward_vs_brute_force(shape, act):
    logits, hidden, wgu, wd = _np_inputs(shape)
    idx, w = O.route(logits, shape.k)
    out = O.forward(hidden, idx, w, wgu, wd, act=act)
    ref = O.forward_brute(hidden, idx, w, wgu, wd, act=act)
    rms = np.sqrt(np.mean(ref ** 2))
    assert np.max(np.abs(out - ref)) / rms < 1e-10


# torch's CPU activations as the library routine the gated MLP reduces to
_TORCH_ACT = {"silu": torch.nn.functional.silu,
              "gelu": lambda x: torch.nn.functional.gelu(x, approximate="none"),
              "relu": torch.relu}


@pytest.mark.parametrize("act", ["silu", "gelu", "relu"])
def test_forward_single_expert_is_dense_glu(act):
    """E = 1, k = 1: the forward is one dense gated MLP (SwiGLU, GeGLU or
    ReGLU), computed here with torch's linear and activation on the CPU."""
    shape = MoEShape(T=33, H=64, I=96, E=1, k=1)
    logits, hidden, wgu, wd = _np_inputs(shape)
    idx, w = O.route(logits, 1)
    assert np.all(idx == 0) and np.allclose(w, 1.0)
    out = O.forward(hidden, idx, w, wgu, wd, dtype=np.float32, act=act)
    x = torch.from_numpy(hidden)
    g = torch.nn.functional.linear(x, torch.from_numpy(wgu[0, :96]))
    u = torch.nn.functional.linear(x, torch.from_numpy(wgu[0, 96:]))
    ref = torch.nn.functional.linear(_TORCH_ACT[act](g) * u,
                                     torch.from_numpy(wd[0])).numpy()
    assert O.rel_max_err(out, ref) < 1e-5


def test_gelu_closed_forms():
    """Exact GELU = x * Phi(x): Phi(1) = 0.8413447460685429 (normal table),
    gelu(x) - gelu(-x) = x (Phi(x) + Phi(-x) = 1), gelu(0) = 0, gelu(x) -> x
    and -> 0 in the tails; and torch's exact gelu in float64."""
    assert O.gelu(np.array([1.0]))[0] == pytest.approx(0.8413447460685429, rel=1e-15)
    assert O.gelu(np.array([-1.0]))[0] == pytest.approx(-0.15865525393145707, rel=1e-14)
    x = np.linspace(-9.0, 9.0, 1001)
    np.testing.assert_allclose(O.gelu(x) - O.gelu(-x), x, rtol=0, atol=1e-14)
    assert O.gelu(np.array([0.0]))[0] == 0.0
    assert abs(O.gelu(np.array([12.0]))[0] - 12.0) < 1e-15
    assert abs(O.gelu(np.array([-12.0]))[0]) < 1e-15
    ref = torch.nn.functional.gelu(torch.from_numpy(x), approximate="none").numpy()
    np.testing.assert_allclose(O.gelu(x), ref, rtol=1e-14, atol=1e-15)


def test_relu_and_silu_against_torch():
    x = np.linspace(-30.0, 30.0, 2001)
    np.testing.assert_array_equal(O.relu(x), torch.relu(torch.from_numpy(x)).numpy())
    np.testing.assert_allclose(O.silu(x), torch.nn.functional.silu(torch.from_numpy(x)).numpy(),
                               rtol=1e-14, atol=1e-300)


def test_forward_k_equals_E_uniform_is_mean_of_experts():
    shape = MoEShape(T=9, H=32, I=32, E=5, k=5)
    _, hidden, wgu, wd = _np_inputs(shape)
    logits = np.zeros((9, 5), np.float32)
    idx, w = O.route(logits, 5)
    out = O.forward(hidden, idx, w, wgu, wd)
    ref = np.mean([O.expert_mlp(hidden, wgu[e], wd[e]) for e in range(5)], axis=0)
    np.testing.assert_allclose(out, ref, rtol=1e-10, atol=1e-12)


def test_forward_token_permutation_equivariance():
    shape = MoEShape(T=40, H=64, I=32, E=6, k=2)
    logits, hidden, wgu, wd = _np_inputs(shape)
    idx, w = O.route(logits, 2)
    out = O.forward(hidden, idx, w, wgu, wd)
    perm = np.random.default_rng(5).permutation(40)
    idx_p, w_p = O.route(logits[perm], 2)
    out_p = O.forward(hidden[perm], idx_p, w_p, wgu, wd)
    np.testing.assert_allclose(out_p, out[perm], rtol=1e-10, atol=1e-12)


def test_forward_linear_in_routing_weights():
    shape = MoEShape(T=10, H=32, I=32, E=4, k=2)
    logits, hidden, wgu, wd = _np_inputs(shape)
    idx, w = O.route(logits, 2)
    w2 = w.copy()
    w2[3] *= 2.5
    w2[7, 1] = 0.0
    out = O.forward(hidden, idx, w, wgu, wd)
    out2 = O.forward(hidden, idx, w2, wgu, wd)
    np.testing.assert_allclose(out2[3], 2.5 * out[3], rtol=1e-10)
    y0 = O.expert_mlp(hidden[7:8], wgu[idx[7, 0]], wd[idx[7, 0]])[0]
    np.testing.assert_allclose(out2[7], w[7, 0] * y0, rtol=1e-10)
    keep = [t for t in range(10) if t not in (3, 7)]
    np.testing.assert_array_equal(out2[keep], out[keep])


def test_round_to_bf16_matches_torch():
    rng = np.random.default_rng(7)
    x = (rng.standard_normal(100000) * np.exp(rng.uniform(-30, 30, 100000))).astype(np.float32)
    x[:4] = [0.0, -0.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8]     # ties to even
    ref = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    np.testing.assert_array_equal(O.round_to_bf16(x).view(np.uint32), ref.view(np.uint32))


# --------------------------------------------------------------------------
# FP8 e4m3 and block scales
# --------------------------------------------------------------------------

def test_e4m3_special_values():
    # OCP FP8 e4m3fn: max normal 448 = 0x7E, min normal 2^-6 = 0x08,
    # min subnormal 2^-9 = 0x01, 1.0 = 0x38, NaN = 0x7F (no infinities)
    vals = np.array([448.0, 2.0 ** -6, 2.0 ** -9, 1.0, -1.0, 0.0, -0.0, 1e30, -1e30,
                     2.0 ** -10, 3 * 2.0 ** -10, 1.0 + 1 / 16, 1.0 + 3 / 16], np.float32)
    codes = O.e4m3_encode(vals)
    assert codes.tolist() == [0x7E, 0x08, 0x01, 0x38, 0xB8, 0x00, 0x80, 0x7E, 0xFE,
                              0x00, 0x02, 0x38, 0x3A]
    dec = O.e4m3_decode(np.arange(256, dtype=np.uint8))
    assert dec[0x7E] == 448.0 and dec[0x01] == 2.0 ** -9 and np.isnan(dec[0x7F])
    assert np.isnan(dec[0xFF]) and dec[0xFE] == -448.0


def test_e4m3_matches_ml_dtypes_exhaustive_window():
    ml = pytest.importorskip("ml_dtypes")
    # every fp32 bit pattern with |x| in [2^-12, 2^10): all the values whose
    # rounding is not a plain flush to zero or a saturation, both signs
    lo = np.uint32((127 - 12) << 23)
    hi = np.uint32((127 + 10) << 23)
    step = 1 << 22
    for start in range(int(lo), int(hi), step):
        bits = np.arange(start, min(start + step, int(hi)), dtype=np.uint32)
        for sgn in (0, 0x80000000):
            x = (bits | np.uint32(sgn)).view(np.float32)
            mine = O.e4m3_encode(x)
            ref = np.asarray(x.astype(ml.float8_e4m3fn)).view(np.uint8)
            over = (ref & 0x7F) == 0x7F       # ml_dtypes overflows to NaN
            assert np.array_equal(mine[~over], ref[~over])
            assert np.all((mine[over] & 0x7F) == 0x7E)
    dec_ref = np.arange(256, dtype=np.uint8).view(ml.float8_e4m3fn).astype(np.float32)
    dec = O.e4m3_decode(np.arange(256, dtype=np.uint8))
    fin = ~np.isnan(dec_ref)
    assert np.array_equal(dec[fin], dec_ref[fin]) and np.all(np.isnan(dec[~fin]))


def test_e4m3_outside_window_saturates_or_flushes():
    rng = np.random.default_rng(11)
    big = np.ldexp(1.0 + rng.random(10000), rng.integers(10, 127, 10000)).astype(np.float32)
    assert np.all(O.e4m3_encode(big) == 0x7E) and np.all(O.e4m3_encode(-big) == 0xFE)
    tiny = np.ldexp(1.0 + rng.random(10000), rng.integers(-126, -12, 10000)).astype(np.float32)
    assert np.all(O.e4m3_encode(tiny) == 0x00) and np.all(O.e4m3_encode(-tiny) == 0x80)


@pytest.mark.parametrize("fmt", ["f32", "ue8m0"])
def test_block_quantiser_bounds(fmt):
    rng = np.random.default_rng(13)
    x = (rng.standard_normal((6, 512)) * np.exp(rng.uniform(-8, 8, (6, 1)))).astype(np.float32)
    x[2, 128:256] = 0.0                                  # amax = 0 block
    codes, stored, s = O.quantize_blocks(x, 1, 128, fmt)
    amax = np.abs(x.reshape(6, 4, 128)).max(-1)
    q = (amax / np.float32(448)).astype(np.float32)
    nz = amax > 0
    if fmt == "ue8m0":
        m, _ = np.frexp(s)
        assert np.all(m == 0.5)                            # powers of two
        assert np.all(s[nz] >= q[nz]) and np.all(s[nz] < 2 * q[nz])
        np.testing.assert_array_equal(O.scale_values(stored, fmt), s)
    else:
        np.testing.assert_array_equal(s[nz], q[nz])
    assert np.all(s[~nz] == 1.0)
    dec = O.e4m3_decode(codes)
    assert np.all(np.abs(dec) <= 448)
    back = O.dequantize_blocks(codes, s, 1, 128)
    # relative error of a normal-range e4m3 value is at most 2^-4
    xs = np.abs(x) / np.repeat(s, 128, axis=1)
    normal = xs >= 2.0 ** -6
    err = np.abs(back - x)
    assert np.all(err[normal] <= 2.0 ** -4 * np.abs(x[normal]) * (1 + 1e-6))
    assert np.all(back[2, 128:256] == 0.0)


def test_weight_block_quantiser_128x128_layout():
    rng = np.random.default_rng(17)
    w = (rng.standard_normal((2, 256, 384)) * 0.02).astype(np.float32)
    w[1, 128:, 256:] *= 1000.0
    codes, stored, s = O.quantize_blocks(w, 128, 128, "f32")
    assert stored.shape == (2, 2, 3)
    for e in range(2):
        for i in range(2):
            for j in range(3):
                blk = w[e, i * 128:(i + 1) * 128, j * 128:(j + 1) * 128]
                assert s[e, i, j] == np.float32(np.abs(blk).max()) / np.float32(448)


def _fp8_weights(wgu, wd, fmt):
    qgu, sgu, _ = O.quantize_blocks(wgu, 128, 128, fmt)
    qd, sd, _ = O.quantize_blocks(wd, 128, 128, fmt)
    return qgu, sgu, qd, sd


@pytest.mark.parametrize("fmt,act", [("f32", "silu"), ("ue8m0", "silu"), ("f32", "gelu"),
                                     ("ue8m0", "relu")])
def test_fp8_forward_without_act_quant_is_bf16_oracle_on_dequantised_weights(fmt, act):
    shape = MoEShape(T=24, H=256, I=128, E=4, k=2)
    logits, hidden, wgu, wd = _np_inputs(shape)
    idx, w = O.route(logits, 2)
    qgu, sgu, qd, sd = _fp8_weights(wgu, wd, fmt)
    out8 = O.forward_fp8(hidden, idx, w, qgu, sgu, qd, sd, fmt,
                         quantize_act=False, quantize_h=False, act=act)
    wgu_d = O.dequantize_blocks(qgu, O.scale_values(sgu, fmt), 128, 128)
    wd_d = O.dequantize_blocks(qd, O.scale_values(sd, fmt), 128, 128)
    ref = O.forward(hidden, idx, w, wgu_d, wd_d, act=act)
    np.testing.assert_allclose(out8, ref, rtol=1e-12, atol=1e-14)


def test_fp8_forward_activation_quant_lossless_on_grid_inputs():
    """Rows whose 1x128 blocks already sit on the e4m3 grid times a power of
    two (with 448 * 2^j present, so the UE8M0 scale is exactly 2^j) quantise
    without loss: the activation quantiser must then be the identity."""
    shape = MoEShape(T=16, H=256, I=128, E=4, k=2)
    logits, _, wgu, wd = _np_inputs(shape)
    rng = np.random.default_rng(19)
    codes = rng.integers(0, 0x7E, (16, 256)).astype(np.uint8)
    codes |= (rng.integers(0, 2, (16, 256)) << 7).astype(np.uint8)
    codes[:, ::128] = 0x7E                                      # amax = 448 per block
    hidden = O.e4m3_decode(codes) * np.float32(2.0 ** -5)
    idx, w = O.route(logits, 2)
    qgu, sgu, qd, sd = _fp8_weights(wgu, wd, "ue8m0")
    a = O.forward_fp8(hidden, idx, w, qgu, sgu, qd, sd, "ue8m0",
                      quantize_act=True, quantize_h=False)
    b = O.forward_fp8(hidden, idx, w, qgu, sgu, qd, sd, "ue8m0",
                      quantize_act=False, quantize_h=False)
    np.testing.assert_array_equal(a, b)


def test_fp8_forward_close_to_bf16_forward():
    """Sanity of scale placement: an FP8 forward that dropped or misplaced a
    scale would be off by orders of magnitude; the real quantisation error of
    e4m3 (about 2-4 % per element) keeps the result within 25 %."""
    shape = MoEShape(T=32, H=256, I=256, E=4, k=2)
    logits, hidden, wgu, wd = _np_inputs(shape)
    idx, w = O.route(logits, 2)
    ref = O.forward(hidden, idx, w, wgu, wd)
    for fmt in ("f32", "ue8m0"):
        qgu, sgu, qd, sd = _fp8_weights(wgu, wd, fmt)
        out = O.forward_fp8(hidden, idx, w, qgu, sgu, qd, sd, fmt)
        rel_rms = np.sqrt(np.mean((out - ref) ** 2) / np.mean(ref ** 2))
        assert rel_rms < 0.25, rel_rms


# --------------------------------------------------------------------------
# FP4 (e2m1) experts: the oracle parts written ahead of their kernel
# --------------------------------------------------------------------------

def test_e2m1_code_table_closed_form():
    """Code s|e e|m: (-1)^s * m/2 for e = 0, else (-1)^s * 2^(e-1) * (1 + m/2)."""
    c = np.arange(16, dtype=np.uint8)
    e = (c.astype(np.int64) >> 1) & 3
    m = c.astype(np.int64) & 1
    mag = np.where(e == 0, m / 2.0, np.ldexp(1.0 + m / 2.0, e - 1))
    ref = np.where(c & 8, -mag, mag)
    np.testing.assert_array_equal(O.e2m1_decode(c), ref.astype(np.float32))
    np.testing.assert_array_equal(O.e2m1_encode(O.e2m1_decode(c)), c)


def test_e2m1_ties_to_even_and_saturation():
    x = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.5, 1e9, -0.0, -5.5, 0.2, 0.3],
                 np.float32)
    want = np.array([0, 2, 2, 4, 4, 6, 6, 7, 7, 8, 15, 0, 1], np.uint8)
    np.testing.assert_array_equal(O.e2m1_encode(x), want)


def test_e2m1_nearest_value_brute_force():
    x = np.random.default_rng(9).uniform(-7.0, 7.0, 200000).astype(np.float32)
    got = O.e2m1_decode(O.e2m1_encode(x)).astype(np.float64)
    grid = O.e2m1_decode(np.arange(8, dtype=np.uint8)).astype(np.float64)
    a = np.minimum(np.abs(x.astype(np.float64)), 6.0)
    best = np.abs(a[:, None] - grid[None, :]).min(axis=1)
    assert np.all(np.abs(np.abs(got) - a) == best)
    assert np.all((got == 0) | (np.sign(got) == np.sign(x)))


def test_e2m1_matches_ml_dtypes():
    ml = pytest.importorskip("ml_dtypes")
    if not hasattr(ml, "float4_e2m1fn"):
        pytest.skip("ml_dtypes without float4_e2m1fn")
    # every fp32 pattern with |x| in [2^-4, 2^4), both signs, thinned 1:64
    bits = np.arange((127 - 4) << 23, (127 + 4) << 23, 64, dtype=np.uint32)
    for sgn in (0, 0x80000000):
        x = (bits | np.uint32(sgn)).view(np.float32)
        ref = np.asarray(x.astype(ml.float4_e2m1fn)).view(np.uint8) & 0xF
        np.testing.assert_array_equal(O.e2m1_encode(x), ref)


def test_fp4_pack_unpack_round_trip():
    c = np.random.default_rng(3).integers(0, 16, size=(5, 64)).astype(np.uint8)
    p = O.pack_e2m1(c)
    assert p.shape == (5, 32)
    np.testing.assert_array_equal(p[:, 0] & 0xF, c[:, 0])
    np.testing.assert_array_equal(p[:, 0] >> 4, c[:, 1])
    np.testing.assert_array_equal(O.unpack_e2m1(p), c)


def test_fp4_block_quantiser_bounds():
    rng = np.random.default_rng(4)
    x = (rng.standard_normal((6, 256)) * np.exp(rng.uniform(-8, 8, (6, 1)))).astype(np.float32)
    x[2, 32:64] = 0.0                                     # an all-zero block
    packed, stored, s = O.quantize_fp4_blocks(x, 32)
    assert packed.shape == (6, 128) and stored.shape == (6, 8)
    np.testing.assert_array_equal(O.scale_values(stored, "ue8m0"), s)
    amax = np.abs(x.reshape(6, 8, 32)).max(axis=-1)
    nz = amax > 0
    assert np.all(np.frexp(s)[0] == 0.5)                 # powers of two
    assert np.all(s[nz] >= amax[nz] / 6.0) and np.all(s[nz] < 2.0 * amax[nz] / 6.0)
    assert s[2, 1] == 1.0 and stored[2, 1] == 127
    deq = O.dequantize_fp4_blocks(packed, s, 32)
    # error within half the widest spacing (2) of the grid at the block scale
    err = np.abs(deq - x.astype(np.float64)).reshape(6, 8, 32).max(axis=-1)
    assert np.all(err <= 1.0 * s + 1e-30)


def test_fp4_forward_without_act_quant_is_bf16_oracle_on_dequantised_weights():
    shape = MoEShape(T=20, H=128, I=64, E=4, k=2)
    logits, hidden, wgu, wd = _np_inputs(shape)
    idx, w = O.route(logits, 2)
    qgu, bgu, _ = O.quantize_fp4_blocks(wgu, 32)
    qd, bd, _ = O.quantize_fp4_blocks(wd, 32)
    out4 = O.forward_fp4(hidden, idx, w, qgu, bgu, qd, bd, 32,
                         quantize_act=False, quantize_h=False, act="silu")
    ref = O.forward(hidden, idx, w, O.dequantize_fp4_blocks(qgu, O.scale_values(bgu, "ue8m0")),
                    O.dequantize_fp4_blocks(qd, O.scale_values(bd, "ue8m0")))
    np.testing.assert_allclose(out4, ref, rtol=1e-12, atol=1e-14)
    # with the activations and h quantised it stays near the bf16 forward:
    # e2m1 carries ~10-20 % relative error per weight, so the rms error of
    # the output is a fraction of its rms
    q = O.forward_fp4(hidden, idx, w, qgu, bgu, qd, bd, 32)
    ref32 = O.forward(hidden, idx, w, wgu, wd)
    assert np.sqrt(np.mean((q - ref32) ** 2)) < 0.5 * np.sqrt(np.mean(ref32 ** 2))
