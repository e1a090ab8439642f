"""FP8 e4m3 block-scaled variant: the CUDA path (through the C ABI) against
the CPU oracle.

* The weight quantiser must reproduce the oracle's e4m3 codes and block
  scales bit for bit, for float32 and UE8M0 scales.
* The forward is compared with the mirrored oracle (same dequantised weights,
  same dynamic 1x128 activation quantisation of the hidden rows and of h):
  max|err| / rms(ref) <= 6e-2, the FP8 tolerance of the workload definition.
  Remaining differences come from accumulation order flipping a rounding of h
  before it is re-quantised.
"""
import numpy as np
import pytest
import torch

import oracle as O
from workloads import MoEShape, make_inputs, shape_for

pytestmark = pytest.mark.gpu

FP8_TOL = 6e-2


@pytest.fixture(scope="module")
def moe():
    import mixture_experts_routed_top_gb300 as m
    m.lib()
    return m


@pytest.mark.parametrize("fmt", ["f32", "ue8m0"])
def test_weight_quantiser_bit_exact(moe, fmt):
    g = torch.Generator().manual_seed(11)
    w = torch.randn(3, 256, 384, generator=g) * 0.02
    w[0, :128, :128] = 0.0                                   # amax = 0 block
    w[1, 128:, 256:] *= 3000.0                               # wide dynamic range
    w[2, :128, 128:256] *= 1e-6
    wb = w.to(torch.bfloat16)
    q, s = moe.quantize_fp8_blocks(wb.cuda(), fmt)
    rq, rs, _ = O.quantize_blocks(wb.float().numpy(), 128, 128, fmt)
    assert np.array_equal(q.cpu().numpy(), rq)
    if fmt == "f32":
        assert np.array_equal(s.cpu().numpy().view(np.uint32), rs.view(np.uint32))
    else:
        assert np.array_equal(s.cpu().numpy(), rs)


@pytest.mark.parametrize("fmt", ["f32", "ue8m0"])
def test_quantiser_every_bf16_value_at_scale_one(moe, fmt):
    """Every finite bf16 value with |x| <= 448, through the device quantiser
    (the hardware e4m3 conversion) at block scale exactly 1: each 128x128
    block also holds 448, so amax = 448 and s = 448/448 = 1 (float32) or
    2^0 (UE8M0).  The codes must be the oracle encoder's codes of the values
    themselves, bit for bit."""
    bits = np.arange(65536, dtype=np.uint32) << np.uint32(16)
    vals = bits.view(np.float32)
    vals = vals[np.isfinite(vals) & (np.abs(vals) <= 448.0)]
    per = 128 * 128 - 1
    nblk = -(-vals.size // per)
    arr = np.zeros((nblk, 128 * 128), np.float32)
    arr[:, 0] = 448.0
    for b in range(nblk):
        chunk = vals[b * per:(b + 1) * per]
        arr[b, 1:1 + chunk.size] = chunk
    arr = arr.reshape(nblk, 128, 128)
    q, sc = moe.quantize_fp8_blocks(torch.from_numpy(arr).to(torch.bfloat16).cuda(), fmt)
    sc = sc.cpu().numpy()
    if fmt == "f32":
        assert np.all(sc == 1.0)
    else:
        assert np.all(sc == 127)
    assert np.array_equal(q.cpu().numpy(), O.e4m3_encode(arr))


def _fp8_case(moe, shape, fmt, seed=0, logit_bias=None, act="silu"):
    d = make_inputs(shape, seed=seed, device="cpu")
    logits = d["logits"] if logit_bias is None else d["logits"] + logit_bias
    idx, w = O.route(logits.numpy(), shape.k)
    w = w.astype(np.float32)
    qgu, sgu, _ = O.quantize_blocks(d["w_gate_up"].float().numpy(), 128, 128, fmt)
    qd, sd, _ = O.quantize_blocks(d["w_down"].float().numpy(), 128, 128, fmt)
    out = moe.experts_forward(d["hidden"].cuda(), torch.from_numpy(idx).cuda(),
                              torch.from_numpy(w).cuda(), torch.from_numpy(qgu).cuda(),
                              torch.from_numpy(qd).cuda(), scale_gate_up=torch.from_numpy(sgu).cuda(),
                              scale_down=torch.from_numpy(sd).cuda(), scale_fmt=fmt,
                              activation=act)
    moe.workspace_status(moe.default_workspace())
    hid = d["hidden"].float().numpy()
    ref = O.forward_fp8(hid, idx, w, qgu, sgu, qd, sd, fmt, act=act)
    plain = O.forward(hid, idx, w, d["w_gate_up"].float().numpy(), d["w_down"].float().numpy(),
                      act=act)
    return out.float().cpu().numpy(), ref, plain


@pytest.mark.parametrize("fmt", ["f32", "ue8m0"])
@pytest.mark.parametrize("shape", [
    MoEShape(T=64, H=256, I=256, E=8, k=2),
    MoEShape(T=300, H=512, I=384, E=6, k=3),       # ragged m-tiles, 3 I-blocks
    MoEShape(T=129, H=256, I=128, E=4, k=2),       # one K-block in the down GEMM
    MoEShape(T=1, H=256, I=256, E=16, k=4),
    MoEShape(T=40, H=1024, I=512, E=64, k=6),
])
def test_forward_fp8_parity(moe, shape, fmt):
    out, ref, plain = _fp8_case(moe, shape, fmt)
    assert np.all(np.isfinite(out))
    assert O.rel_max_err(out, ref) <= FP8_TOL
    # sanity, not a gate: the FP8 result stays near the unquantised forward
    assert O.rel_max_err(out, plain) < 0.5


def test_forward_fp8_f32_phases_groups_l2_hints(moe):
    """Float32-scale kernel with its down GEMM's output columns in four
    slices (accumulator reductions under the L2 policy) and gate/up m-tiles
    in groups of two (an expert with 5 m-tiles): every tile runs once."""
    shape = MoEShape(T=700, H=1024, I=256, E=2, k=2)
    moe.set_down_phases(4)
    moe.set_tile_group(2)
    moe.set_down_l2_hints(1)
    try:
        out, ref, _ = _fp8_case(moe, shape, "f32")
    finally:
        moe.set_down_phases(-1)
        moe.set_tile_group(-1)
        moe.set_down_l2_hints(-1)
    assert O.rel_max_err(out, ref) <= FP8_TOL


@pytest.mark.parametrize("fmt,act", [("f32", "gelu"), ("ue8m0", "relu")])
@pytest.mark.parametrize("shape", [MoEShape(T=300, H=512, I=384, E=6, k=3),
                                   MoEShape(T=40, H=1024, I=512, E=64, k=6)])
def test_forward_fp8_geglu_reglu(moe, shape, fmt, act):
    out, ref, plain = _fp8_case(moe, shape, fmt, act=act)
    assert O.rel_max_err(out, ref) <= FP8_TOL
    assert O.rel_max_err(out, plain) < 0.5


@pytest.mark.parametrize("fmt", ["f32", "ue8m0"])
def test_forward_fp8_one_expert_takes_all(moe, fmt):
    shape = MoEShape(T=600, H=256, I=256, E=8, k=2)
    bias = torch.zeros(8)
    bias[2] = 30.0
    out, ref, _ = _fp8_case(moe, shape, fmt, logit_bias=bias)
    assert O.rel_max_err(out, ref) <= FP8_TOL


def test_forward_fp8_rejects_missing_scales(moe):
    d = make_inputs(MoEShape(T=4, H=256, I=128, E=2, k=1), seed=0, device="cuda")
    idx, w = moe.route(d["logits"], 1)
    q, s = moe.quantize_fp8_blocks(d["w_gate_up"], "f32")
    qd, sd = moe.quantize_fp8_blocks(d["w_down"], "f32")
    with pytest.raises(moe.MoEError) as ei:
        moe.experts_forward(d["hidden"], idx, w, q, qd)
    assert ei.value.status == 1


@pytest.mark.parametrize("T,fmt", [(64, "f32"), (64, "ue8m0"), (16384, "f32"), (16384, "ue8m0")])
def test_forward_fp8_full_size_every_tile(moe, T, fmt):
    """Full FP8 workload size on the GPU.  At T = 64 every token is checked.
    At T = 16384 the oracle recomputes the tokens at the edges of every
    grouped-GEMM tile of the busiest expert (125 tiles of 128 rows) and the
    first and last token of the other popular experts, using only tokens
    whose eight experts are all among the 16 most popular (more if some tile
    has no such token), so that few experts are dequantised on the host."""
    from full_size_sampling import (check_accumulator, fp8_expert_fn, oracle_on_tokens,
                                    probe_tokens, tile_count)
    shape = shape_for("dsv3_fp8", T)
    d = make_inputs(shape, seed=0, device="cuda")
    qgu, sgu = moe.quantize_fp8_blocks(d["w_gate_up"], fmt)
    qd, sd = moe.quantize_fp8_blocks(d["w_down"], fmt)
    del d["w_gate_up"], d["w_down"]
    idx, w = moe.route(d["logits"], shape.k)
    out = moe.experts_forward(d["hidden"], idx, w, qgu, qd, scale_gate_up=sgu, scale_down=sd,
                              scale_fmt=fmt)
    moe.workspace_status(moe.default_workspace())
    ref_idx, ref_w = O.route(d["logits"].cpu().numpy(), shape.k)
    assert np.array_equal(idx.cpu().numpy(), ref_idx)
    if T <= 64:
        toks = np.arange(T)
    else:
        counts = np.bincount(ref_idx.ravel(), minlength=shape.E)
        order = np.argsort(-counts, kind="stable")
        for n_cheap in (16, 24, 32, 48):          # widen until every hot tile is reached
            cheap = set(order[:n_cheap].tolist())
            toks, counts, hot, reached = probe_tokens(ref_idx, shape.E, shape.k, cheap=cheap)
            if reached == tile_count(int(counts[hot])):
                break
        assert hot in cheap and reached == tile_count(int(counts[hot]))
    tt = torch.from_numpy(toks).cuda()
    ref = oracle_on_tokens(toks, ref_idx, ref_w, d["hidden"][tt].float().cpu().numpy(),
                           fp8_expert_fn(qgu, sgu, qd, sd, fmt))
    check_accumulator(moe, out, toks, ref, shape, moe.W_FP8_E4M3, FP8_TOL)
