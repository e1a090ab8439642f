"""FP4 (e2m1) experts: the CUDA path (through the C ABI) against the CPU
oracle.

* The weight quantiser must reproduce the oracle's packed e2m1 codes and
  UE8M0 bytes bit for bit.
* The forward is compared with the mirrored oracle (the same packed weights
  and scales, the same dynamic 1x32 e4m3 quantisation of the hidden rows
  and of h): max|err| / rms(ref) <= 6e-2, the tolerance used for the FP8
  experts.  Remaining differences come from fp32 accumulation order
  flipping an e4m3 rounding (or a block scale) of h.
* These shapes run on the small-token GEMVs (threshold set to 64 routed
  rows here); by default FP4 runs on the block-scaled tensor-core GEMMs
  (tests/test_gpu_block_scaled.py).
"""
import numpy as np
import pytest
import torch

import oracle as O
from workloads import MoEShape, make_inputs, shape_for

pytestmark = pytest.mark.gpu

FP4_TOL = 6e-2


@pytest.fixture(scope="module")
def moe():
    """The library with the FP4 GEMV threshold at its maximum (64 routed
    rows), so these small batches exercise the CUDA-core GEMVs; the default
    sends them to the block-scaled GEMMs (tests/test_gpu_block_scaled.py)."""
    import mixture_experts_routed_top_gb300 as m
    m.lib()
    m.set_fp4_gemv_rows(64)
    yield m
    m.set_fp4_gemv_rows(-1)


def test_weight_quantiser_bit_exact(moe):
    g = torch.Generator().manual_seed(5)
    w = torch.randn(3, 64, 96, generator=g) * 0.02
    w[0, :4, :32] = 0.0                                     # amax = 0 blocks
    w[1, 8:16] *= 3000.0                                    # wide dynamic range
    w[2, :8, 32:64] *= 1e-6
    # every rounding tie and the saturation edge at scale 1 (block amax = 6)
    ties = torch.tensor([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, 0.5, 1.5, 3.0, 4.0,
                         0.0, -0.0, 5.5, 0.125])
    w[2, 20, :16] = ties
    w[2, 20, 16:32] = -ties
    wb = w.to(torch.bfloat16)
    q, s = moe.quantize_fp4_blocks(wb.cuda())
    rq, rs, _ = O.quantize_fp4_blocks(wb.float().numpy())
    assert np.array_equal(s.cpu().numpy(), rs)
    assert np.array_equal(q.cpu().numpy(), rq)


def test_quantiser_every_bf16_value_at_scale_one(moe):
    """Every finite bf16 value with |x| <= 6, each 1x32 block also holding 6
    so that amax/6 = 1 and the scale is 2^0: the device codes must be the
    oracle encoder's codes of the values themselves."""
    bits = np.arange(65536, dtype=np.uint32) << np.uint32(16)
    vals = bits.view(np.float32)
    vals = vals[np.isfinite(vals) & (np.abs(vals) <= 6.0)]
    per = 31
    nblk = -(-vals.size // per)
    arr = np.zeros((nblk, 32), np.float32)
    arr[:, 0] = 6.0
    flat = np.zeros(nblk * per, np.float32)
    flat[:vals.size] = vals
    arr[:, 1:] = flat.reshape(nblk, per)
    q, s = moe.quantize_fp4_blocks(torch.from_numpy(arr).to(torch.bfloat16).cuda())
    assert np.all(s.cpu().numpy() == 127)
    assert np.array_equal(O.unpack_e2m1(q.cpu().numpy()), O.e2m1_encode(arr))


def _fp4_inputs(shape, seed=0, logit_bias=None):
    d = make_inputs(shape, seed=seed, device="cpu")
    logits = d["logits"] if logit_bias is None else d["logits"] + logit_bias
    idx, w = O.route(logits.numpy(), shape.k)
    qgu, sgu, _ = O.quantize_fp4_blocks(d["w_gate_up"].float().numpy())
    qd, sd, _ = O.quantize_fp4_blocks(d["w_down"].float().numpy())
    return d, idx, w.astype(np.float32), qgu, sgu, qd, sd


def _fp4_case(moe, shape, seed=0, logit_bias=None, act="silu"):
    d, idx, w, qgu, sgu, qd, sd = _fp4_inputs(shape, seed, logit_bias)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    out = moe.experts_forward(d["hidden"].cuda(), dev(idx), dev(w), dev(qgu), dev(qd),
                              scale_gate_up=dev(sgu), scale_down=dev(sd), scale_fmt="ue8m0",
                              activation=act)
    moe.workspace_status(moe.default_workspace())
    hid = d["hidden"].float().numpy()
    ref = O.forward_fp4(hid, idx, w, qgu, sgu, qd, sd, act=act)
    plain = O.forward(hid, idx, w, d["w_gate_up"].float().numpy(), d["w_down"].float().numpy(),
                      act=act)
    return out.float().cpu().numpy(), ref, plain


def _rel_rms(out, ref):
    return float(np.sqrt(np.mean((out - ref) ** 2)) / np.sqrt(np.mean(ref ** 2)))


@pytest.mark.parametrize("shape", [
    MoEShape(T=1, H=256, I=256, E=16, k=4),
    MoEShape(T=3, H=512, I=384, E=8, k=2),          # token chunks of 2 with a ragged tail
    MoEShape(T=8, H=1024, I=512, E=32, k=8),        # T*k = 64, the largest batch
    MoEShape(T=16, H=256, I=128, E=4, k=4),         # 16 rows per expert: chunks of 8
    MoEShape(T=5, H=2048, I=1408, E=4, k=2),        # Qwen widths: 44 blocks along I
    MoEShape(T=2, H=7168, I=256, E=4, k=2),         # DeepSeek-V3 width: 224 blocks along H
])
def test_forward_fp4_parity(moe, shape):
    out, ref, plain = _fp4_case(moe, shape)
    assert np.all(np.isfinite(out))
    assert O.rel_max_err(out, ref) <= FP4_TOL
    # sanity, not a gate: FP4 weights stay near the unquantised forward
    assert _rel_rms(out, plain) < 0.5


@pytest.mark.parametrize("act", ["gelu", "relu"])
@pytest.mark.parametrize("shape", [MoEShape(T=3, H=512, I=384, E=8, k=2),
                                   MoEShape(T=4, H=512, I=256, E=16, k=4)])
def test_forward_fp4_geglu_reglu(moe, shape, act):
    out, ref, plain = _fp4_case(moe, shape, act=act)
    assert O.rel_max_err(out, ref) <= FP4_TOL
    assert _rel_rms(out, plain) < 0.5


def test_forward_fp4_one_expert_takes_all(moe):
    shape = MoEShape(T=32, H=256, I=256, E=8, k=2)
    bias = torch.zeros(8)
    bias[2] = 30.0
    out, ref, _ = _fp4_case(moe, shape, logit_bias=bias)
    assert O.rel_max_err(out, ref) <= FP4_TOL


def test_forward_fp4_full_qwen_width(moe):
    """Full Qwen expert count and widths (E=60, H=2048, I=1408), T=2 and its
    first token alone.  The oracle quantises only the touched experts; the
    other experts' slots hold zero codes, which a kernel that read them would
    turn into a wrong output."""
    shape = shape_for("qwen", 2)
    d = make_inputs(shape, seed=0, device="cpu")
    idx, w = O.route(d["logits"].numpy(), shape.k)
    w = w.astype(np.float32)
    experts = np.unique(idx)
    E, I, H = shape.E, shape.I, shape.H
    qgu = np.zeros((E, 2 * I, H // 2), np.uint8)
    sgu = np.zeros((E, 2 * I, H // 32), np.uint8)
    qd = np.zeros((E, H, I // 2), np.uint8)
    sd = np.zeros((E, H, I // 32), np.uint8)
    for e in experts:
        qgu[e], sgu[e], _ = O.quantize_fp4_blocks(d["w_gate_up"][e].float().numpy())
        qd[e], sd[e], _ = O.quantize_fp4_blocks(d["w_down"][e].float().numpy())
    del d["w_gate_up"], d["w_down"]
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    W = dict(w_gate_up=dev(qgu), w_down=dev(qd), scale_gate_up=dev(sgu), scale_down=dev(sd),
             scale_fmt="ue8m0")
    remap = np.full(E, -1, np.int64)
    remap[experts] = np.arange(len(experts))
    hid = d["hidden"].float().numpy()
    for T in (2, 1):
        out = moe.experts_forward(d["hidden"][:T].cuda(), dev(idx[:T]), dev(w[:T]), **W)
        moe.workspace_status(moe.default_workspace())
        ref = O.forward_fp4(hid[:T], remap[idx[:T]].astype(np.int32), w[:T],
                            qgu[experts], sgu[experts], qd[experts], sd[experts])
        assert O.rel_max_err(out.float().cpu().numpy(), ref) <= FP4_TOL


def test_forward_fp4_rejections(moe):
    shape = MoEShape(T=4, H=256, I=128, E=4, k=2)
    d = make_inputs(shape, seed=0, device="cuda")
    idx, w = moe.route(d["logits"], shape.k)
    qgu, sgu = moe.quantize_fp4_blocks(d["w_gate_up"])
    qd, sd = moe.quantize_fp4_blocks(d["w_down"])
    with pytest.raises(moe.MoEError) as ei:                 # float32 scale format
        moe.experts_forward(d["hidden"], idx, w, qgu, qd, scale_gate_up=sgu, scale_down=sd,
                            scale_fmt="f32")
    assert ei.value.status == 1
    with pytest.raises(moe.MoEError) as ei:                 # scales missing
        moe.experts_forward(d["hidden"], idx, w, qgu, qd)
    assert ei.value.status == 1
    # above 64 routed rows the block-scaled GEMMs run; their 256-wide down
    # tiles need H % 256 == 0
    narrow = MoEShape(T=40, H=128, I=128, E=4, k=2)
    big = make_inputs(narrow, seed=1, device="cuda")
    bidx, bw = moe.route(big["logits"], 2)
    nq, ns = moe.quantize_fp4_blocks(big["w_gate_up"])
    nqd, nsd = moe.quantize_fp4_blocks(big["w_down"])
    with pytest.raises(moe.MoEError) as ei:                 # T*k = 80 > 64, H = 128
        moe.experts_forward(big["hidden"], bidx, bw, nq, nqd, scale_gate_up=ns, scale_down=nsd)
    assert ei.value.status == 2


def test_forward_fp4_reports_bad_expert_index(moe):
    shape = MoEShape(T=4, H=256, I=128, E=4, k=2)
    d = make_inputs(shape, seed=0, device="cuda")
    idx, w = moe.route(d["logits"], shape.k)
    qgu, sgu = moe.quantize_fp4_blocks(d["w_gate_up"])
    qd, sd = moe.quantize_fp4_blocks(d["w_down"])
    idx[1, 0] = shape.E                                     # out of range: skipped, reported
    ws = moe.Workspace(idx.device)
    moe.experts_forward(d["hidden"], idx, w, qgu, qd, scale_gate_up=sgu, scale_down=sd,
                        workspace=ws)
    with pytest.raises(moe.MoEError) as ei:
        moe.workspace_status(ws)
    assert ei.value.status == 1
