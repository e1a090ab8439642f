"""Block-scaled tensor-core GEMMs (tcgen05.mma kind::mxf8f6f4 with UE8M0
scale factors) against the CPU oracle, through the C ABI.

* FP4 (e2m1) experts, which take these GEMMs at every batch size by
  default: the mirrored FP4 oracle (same packed weights and 1x32 scales,
  same dynamic 1x32 e4m3 quantisation of the hidden rows and of h),
  max|err| / rms(ref) <= 6e-2.
* FP8 experts with UE8M0 scales on the hardware block scaling and on the
  software promotion kernel: both against the mirrored FP8 oracle.
* Scales spread over a wide range of powers of two, per 32-wide sub-block
  of rows and columns, so that a scale applied to the wrong row, column or
  sub-block changes the result by orders of magnitude instead of a few per
  cent.

Source: Hugging Face Transformers "Experts backends" page, "FP8 and FP4
quantized experts" section (UE8M0 scales on Blackwell; FP4 weights packed in
int8) and the paragraph after the backends table.
"""
import numpy as np
import pytest
import torch

import oracle as O
from workloads import MoEShape, make_inputs

pytestmark = pytest.mark.gpu

TOL = 6e-2


@pytest.fixture(scope="module")
def moe():
    import mixture_experts_routed_top_gb300 as m
    m.lib()
    yield m
    m.set_fp4_gemv_rows(-1)
    m.set_block_scaled_mma(True)


def _spread(x, block, rng, lo=-6, hi=6):
    """Multiply each 1 x block group along the last axis by its own power of
    two drawn from [2^lo, 2^hi]."""
    *lead, C = x.shape
    e = rng.integers(lo, hi + 1, size=(*lead, C // block)).astype(np.float32)
    return (x.reshape(*lead, C // block, block) * np.exp2(e)[..., None]).reshape(x.shape)


def _inputs(shape, seed, spread=None, logit_bias=None):
    d = make_inputs(shape, seed=seed, device="cpu")
    logits = d["logits"] if logit_bias is None else d["logits"] + logit_bias
    idx, w = O.route(logits.numpy(), shape.k)
    hid = d["hidden"].float().numpy()
    wgu = d["w_gate_up"].float().numpy()
    wd = d["w_down"].float().numpy()
    if spread:
        rng = np.random.default_rng(seed + 100)
        hid = _spread(hid, spread, rng)
        wgu = _spread(wgu, spread, rng)
        wd = _spread(wd, spread, rng)
        # back to bf16-representable values (the device reads bf16 hidden rows)
        hid = torch.from_numpy(hid).to(torch.bfloat16).float().numpy()
    return hid, idx, w.astype(np.float32), wgu, wd


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _run_fp4(moe, shape, seed=0, spread=None, act="silu", logit_bias=None):
    hid, idx, w, wgu, wd = _inputs(shape, seed, spread, logit_bias)
    qgu, sgu, _ = O.quantize_fp4_blocks(wgu)
    qd, sd, _ = O.quantize_fp4_blocks(wd)
    n0 = moe.launch_count()
    out = moe.experts_forward(_dev(hid).to(torch.bfloat16), _dev(idx), _dev(w), _dev(qgu), _dev(qd),
                              scale_gate_up=_dev(sgu), scale_down=_dev(sd), scale_fmt="ue8m0",
                              activation=act)
    moe.workspace_status(moe.default_workspace())
    launches = moe.launch_count() - n0
    ref = O.forward_fp4(hid, idx, w, qgu, sgu, qd, sd, act=act)
    return out.float().cpu().numpy(), ref, launches


def _run_fp8(moe, shape, seed=0, spread=None, act="silu", logit_bias=None):
    hid, idx, w, wgu, wd = _inputs(shape, seed, spread, logit_bias)
    qgu, sgu, _ = O.quantize_blocks(wgu, 128, 128, "ue8m0")
    qd, sd, _ = O.quantize_blocks(wd, 128, 128, "ue8m0")
    out = moe.experts_forward(_dev(hid).to(torch.bfloat16), _dev(idx), _dev(w), _dev(qgu), _dev(qd),
                              scale_gate_up=_dev(sgu), scale_down=_dev(sd), scale_fmt="ue8m0",
                              activation=act)
    moe.workspace_status(moe.default_workspace())
    ref = O.forward_fp8(hid, idx, w, qgu, sgu, qd, sd, "ue8m0", act=act)
    return out.float().cpu().numpy(), ref


FP4_SHAPES = [
    MoEShape(T=40, H=256, I=128, E=4, k=2),         # 80 routed rows: just above the GEMVs
    MoEShape(T=300, H=512, I=384, E=6, k=3),        # ragged m-tiles, 3 feature blocks
    MoEShape(T=129, H=256, I=256, E=4, k=2),        # one 128-wide K block in the down GEMM
    MoEShape(T=100, H=2048, I=1408, E=60, k=4),     # Qwen widths
    MoEShape(T=48, H=7168, I=256, E=8, k=4),        # DeepSeek-V3 width along K
]


@pytest.mark.parametrize("shape", FP4_SHAPES)
def test_fp4_block_scaled_parity(moe, shape):
    moe.set_fp4_gemv_rows(-1)
    out, ref, launches = _run_fp4(moe, shape)
    assert launches >= 5          # dispatch, gather, zero, two GEMMs, output: not the GEMVs
    assert np.all(np.isfinite(out))
    assert O.rel_max_err(out, ref) <= TOL


@pytest.mark.parametrize("shape", [MoEShape(T=1, H=256, I=256, E=16, k=4),
                                   MoEShape(T=8, H=1024, I=512, E=32, k=8)])
def test_fp4_block_scaled_small_batches(moe, shape):
    """Small batches take the GEMMs by default (threshold 0)."""
    moe.set_fp4_gemv_rows(-1)
    assert moe.get_fp4_gemv_rows() == 0
    out, ref, launches = _run_fp4(moe, shape)
    assert launches >= 5
    assert O.rel_max_err(out, ref) <= TOL


def test_fp4_narrow_hidden_small_batch_takes_the_gemvs(moe):
    """H % 256 != 0: the GEMMs' 256-wide down tiles do not fit, so a batch of
    at most 64 routed rows runs on the GEMVs (three launches)."""
    out, ref, launches = _run_fp4(moe, MoEShape(T=4, H=384, I=256, E=8, k=2))
    assert launches == 3
    assert O.rel_max_err(out, ref) <= TOL


@pytest.mark.parametrize("shape", [MoEShape(T=300, H=512, I=384, E=6, k=3),
                                   MoEShape(T=64, H=256, I=256, E=4, k=2)])
def test_fp4_block_scaled_wide_scale_range(moe, shape):
    """Every 1x32 block of the hidden rows and weights scaled by its own
    power of two in [2^-6, 2^6]: a scale factor read for the wrong row,
    column or 32-wide sub-block shows as an error of order one."""
    moe.set_fp4_gemv_rows(-1)
    out, ref, _ = _run_fp4(moe, shape, seed=3, spread=32)
    assert O.rel_max_err(out, ref) <= TOL


@pytest.mark.parametrize("act", ["gelu", "relu"])
def test_fp4_block_scaled_geglu_reglu(moe, act):
    out, ref, _ = _run_fp4(moe, MoEShape(T=300, H=512, I=384, E=6, k=3), act=act)
    assert O.rel_max_err(out, ref) <= TOL


def test_fp4_block_scaled_one_expert_takes_all(moe):
    bias = torch.zeros(8)
    bias[5] = 30.0
    out, ref, _ = _run_fp4(moe, MoEShape(T=700, H=256, I=256, E=8, k=2), logit_bias=bias)
    assert O.rel_max_err(out, ref) <= TOL


def test_fp4_gemv_and_gemm_paths_agree(moe):
    """The same 64-row FP4 batch through the GEMVs and through the GEMMs."""
    shape = MoEShape(T=16, H=512, I=256, E=8, k=4)
    moe.set_fp4_gemv_rows(64)
    try:
        a, ref, la = _run_fp4(moe, shape, seed=7)
    finally:
        moe.set_fp4_gemv_rows(-1)
    b, _, lb = _run_fp4(moe, shape, seed=7)
    assert la == 3 and lb >= 5
    assert O.rel_max_err(a, ref) <= TOL and O.rel_max_err(b, ref) <= TOL


@pytest.mark.parametrize("fmt", ["fp4", "fp8"])
def test_block_scaled_down_gemm_phases_and_groups(moe, fmt):
    """Down GEMM output columns in four slices (with L2 policies on its
    accumulator reductions and weight loads) and gate/up m-tiles in groups of
    two (an expert with 5 m-tiles): every tile still runs exactly once."""
    shape = MoEShape(T=700, H=1024, I=256, E=2, k=2)
    moe.set_down_phases(4)
    moe.set_tile_group(2)
    moe.set_down_l2_hints(3)
    try:
        if fmt == "fp4":
            out, ref, _ = _run_fp4(moe, shape)
        else:
            out, ref = _run_fp8(moe, shape)
    finally:
        moe.set_down_phases(-1)
        moe.set_tile_group(-1)
        moe.set_down_l2_hints(-1)
    assert O.rel_max_err(out, ref) <= TOL


FP8_SHAPES = [
    MoEShape(T=64, H=256, I=256, E=8, k=2),
    MoEShape(T=300, H=512, I=384, E=6, k=3),
    MoEShape(T=129, H=256, I=128, E=4, k=2),
    MoEShape(T=40, H=1024, I=512, E=64, k=6),
]


@pytest.mark.parametrize("hw", [True, False], ids=["block_scaled_mma", "promotion"])
@pytest.mark.parametrize("shape", FP8_SHAPES)
def test_fp8_ue8m0_both_kernels(moe, shape, hw):
    moe.set_block_scaled_mma(hw)
    try:
        out, ref = _run_fp8(moe, shape)
    finally:
        moe.set_block_scaled_mma(True)
    assert O.rel_max_err(out, ref) <= TOL


@pytest.mark.parametrize("shape", [MoEShape(T=300, H=512, I=384, E=6, k=3)])
def test_fp8_ue8m0_wide_scale_range(moe, shape):
    """128x128 weight blocks and 1x128 activation blocks (here every 1x32
    group) spread over [2^-6, 2^6]."""
    out, ref = _run_fp8(moe, shape, seed=4, spread=32)
    assert O.rel_max_err(out, ref) <= TOL
