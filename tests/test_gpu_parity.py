"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Routing indices, counts, offsets and the permutation must match bit for bit;
routing weights within 2e-6 relative; the bf16 forward within
max|err| / rms(ref) <= 2e-2 (the float tolerance the workload definition
states).  Sizes span several 128-row tiles with ragged tails, empty experts,
one overloaded expert, T = 1, and the full workload sizes on sampled tokens.
"""
import numpy as np
import pytest
import torch

import oracle as O
from workloads import MoEShape, make_inputs, shape_for

pytestmark = pytest.mark.gpu

BF16_TOL = 2e-2


@pytest.fixture(scope="module")
def moe():
    import mixture_experts_routed_top_gb300 as m
    m.lib()
    return m


def _to_np(t):
    return t.detach().cpu().float().numpy() if t.dtype == torch.bfloat16 else t.detach().cpu().numpy()


# ----------------------------------------------------------------- router
@pytest.mark.parametrize("T,E,k", [(64, 8, 2), (4096, 60, 4), (1000, 256, 8), (3, 1024, 32),
                                   (33, 33, 32), (5, 1, 1), (17, 40, 7)])
def test_route_parity(moe, T, E, k):
    g = torch.Generator().manual_seed(T * 7 + E)
    logits = torch.randn(T, E, generator=g)
    logits[: T // 3, E // 2] = logits[: T // 3, 0]          # exact ties
    if T > 2:
        logits[1] = 0.25                                    # all equal
        logits[2, : max(1, E - k)] = float("-inf")          # -inf entries
    idx, w = moe.route(logits.cuda(), k)
    ref_idx, ref_w = O.route(logits.numpy(), k)
    assert np.array_equal(idx.cpu().numpy(), ref_idx)
    np.testing.assert_allclose(w.cpu().numpy(), ref_w, rtol=2e-6, atol=1e-7)


def test_route_all_neg_inf_row(moe):
    logits = torch.full((2, 6), float("-inf"))
    logits[1, 4] = 1.0
    idx, w = moe.route(logits.cuda(), 3)
    ref_idx, ref_w = O.route(logits.numpy(), 3)
    assert np.array_equal(idx.cpu().numpy(), ref_idx)
    np.testing.assert_allclose(w.cpu().numpy(), ref_w, rtol=1e-6)


def test_route_empty(moe):
    idx, w = moe.route(torch.empty(0, 8, device="cuda"), 2)
    assert idx.shape == (0, 2)


# ----------------------------------------------------------------- dispatch
@pytest.mark.parametrize("T,E,k", [(64, 8, 2), (4096, 60, 4), (5000, 256, 8), (1, 4, 4),
                                   (700, 1024, 3), (2049, 2, 1)])
def test_dispatch_parity(moe, T, E, k):
    g = torch.Generator().manual_seed(T + E + k)
    logits = torch.randn(T, E, generator=g)
    logits[:, 0] += 2.0                                      # one popular expert
    if E > 3:
        logits[:, 3] -= 50.0                                 # one empty expert
    ref_idx, _ = O.route(logits.numpy(), k)
    idx = torch.from_numpy(ref_idx).cuda()
    counts, offsets, sorted_f, row_of = moe.dispatch(idx, E)
    rc, ro, rs, rr = O.dispatch(ref_idx, E)
    assert np.array_equal(counts.cpu().numpy(), rc)
    assert np.array_equal(offsets.cpu().numpy(), ro)
    assert np.array_equal(sorted_f.cpu().numpy(), rs)
    assert np.array_equal(row_of.cpu().numpy(), rr)


def test_dispatch_empty(moe):
    counts, offsets, sorted_f, row_of = moe.dispatch(torch.empty(0, 2, dtype=torch.int32,
                                                                 device="cuda"), 5)
    assert counts.cpu().tolist() == [0] * 5 and offsets.cpu().tolist() == [0] * 6


def test_dispatch_out_of_range_index_is_reported(moe):
    idx = torch.tensor([[0, 1], [7, 2]], dtype=torch.int32, device="cuda")
    with pytest.raises(moe.MoEError) as ei:
        moe.dispatch(idx, 4)
    assert ei.value.status == 1


# ----------------------------------------------------------------- forward
# (decode-path row threshold, swap-AB rows-per-expert threshold, CTA-pair mask)
PATHS = {"rows": (0, 0, 0), "swap": (0, 1 << 20, 0), "decode": (2048, -1, 0),
         "pair": (0, -1, 3)}


@pytest.fixture
def path(moe, request):
    """Force one of the bf16 paths: grouped GEMMs with token rows as the
    MMA's M side, grouped GEMMs with weight rows as M (swap-AB), both grouped
    GEMMs on CTA pairs (weight rows as M, cta_group::2), or the decode
    GEMVs."""
    dec, swap, pair = PATHS[request.param]
    moe.set_decode_rows(dec)
    moe.set_swap_rows(swap)
    moe.set_pair_gemm(pair)
    yield request.param
    moe.set_decode_rows(-1)
    moe.set_swap_rows(-1)
    moe.set_pair_gemm(-1)


def _forward_case(moe, shape, seed=0, logit_bias=None, device_inputs=None, act="silu"):
    d = make_inputs(shape, seed=seed, device="cpu") if device_inputs is None else device_inputs
    logits = d["logits"]
    if logit_bias is not None:
        logits = logits + logit_bias
    idx, w = O.route(logits.numpy(), shape.k)
    dev = {n: d[n].cuda() for n in ("hidden", "w_gate_up", "w_down")}
    out = moe.experts_forward(dev["hidden"], torch.from_numpy(idx).cuda(),
                              torch.from_numpy(w.astype(np.float32)).cuda(),
                              dev["w_gate_up"], dev["w_down"], activation=act)
    moe.workspace_status(moe.default_workspace())
    ref = O.forward(d["hidden"].float().numpy(), idx, w.astype(np.float32),
                    d["w_gate_up"].float().numpy(), d["w_down"].float().numpy(), act=act)
    return _to_np(out), ref


SMALL_SHAPES = [
    shape_for("tiny"),
    MoEShape(T=300, H=256, I=384, E=6, k=3),        # ragged m-tiles, several n-tiles
    MoEShape(T=129, H=384, I=128, E=4, k=2),        # down GEMM with 128-wide n-tiles
    MoEShape(T=1, H=512, I=256, E=16, k=4),         # a single token
    MoEShape(T=40, H=1024, I=512, E=64, k=6),       # most experts get 1-10 rows
    MoEShape(T=3, H=128, I=128, E=2, k=2),          # k = E
    MoEShape(T=64, H=128, I=128, E=1024, k=32),     # E and k at their limits, 2048 rows
]


def _random_shapes(n, seed):
    """Seeded random shapes over the library's path boundaries: H and I
    multiples of 128 (H with and without H % 256 == 0, which the CTA-pair
    down GEMM needs), E up to 96, k up to 8, and T so that the
    routed rows per expert run from under one (decode GEMVs) to a few
    hundred (token-row and CTA-pair GEMMs, several ragged tiles)."""
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        E = int(rng.integers(1, 97))
        k = int(rng.integers(1, min(E, 8) + 1))
        per_expert = float(rng.choice([0.5, 2.0, 9.0, 40.0, 150.0, 320.0]))
        T = max(1, min(700, int(round(per_expert * E / k))))
        H = int(rng.choice([128, 256, 384, 512, 768, 1024]))
        I = int(rng.choice([128, 256, 384, 512]))
        out.append(MoEShape(T=T, H=H, I=I, E=E, k=k))
    return out


RANDOM_SHAPES = _random_shapes(16, seed=20261203)


@pytest.mark.parametrize("shape", RANDOM_SHAPES, ids=lambda s: f"T{s.T}_H{s.H}_I{s.I}_E{s.E}_k{s.k}")
def test_forward_bf16_random_shapes_default_paths(moe, shape):
    """The library's own path choice (decode GEMVs, swap-AB, token-row or
    CTA-pair GEMMs for either GEMM) on seeded random shapes, every output
    against the oracle.  Above 100 k outputs the grouped paths are checked
    on their fp32 accumulator, the bf16 output its exact RNE image: at that
    many outputs the bf16 rounding of the largest ones alone approaches the
    tolerance (see tests/full_size_sampling.py)."""
    from full_size_sampling import check_accumulator
    out, ref = _forward_case(moe, shape, seed=shape.T + shape.E)
    assert np.all(np.isfinite(out))
    grouped = shape.T * shape.k > moe.get_decode_rows()
    if grouped and shape.T * shape.H > 100_000:
        out_t = torch.from_numpy(out).to(torch.bfloat16).cuda()
        check_accumulator(moe, out_t, np.arange(shape.T), ref, shape, moe.W_BF16, BF16_TOL)
    else:
        err = O.rel_max_err(out, ref)
        assert err <= BF16_TOL, (shape, err)


@pytest.mark.parametrize("pair", [0, 3], ids=["one_cta", "cta_pairs"])
def test_forward_bf16_random_shape_both_down_kernels_agree(moe, pair):
    """The largest random shape through the one-CTA and the CTA-pair down
    GEMMs: both within the tolerance on the fp32 accumulator."""
    from full_size_sampling import check_accumulator
    shape = max(RANDOM_SHAPES, key=lambda s: s.T * s.k * s.H)
    moe.set_pair_gemm(pair)
    try:
        out, ref = _forward_case(moe, shape, seed=shape.T + shape.E)
    finally:
        moe.set_pair_gemm(-1)
    out_t = torch.from_numpy(out).to(torch.bfloat16).cuda()
    check_accumulator(moe, out_t, np.arange(shape.T), ref, shape, moe.W_BF16, BF16_TOL)


@pytest.mark.parametrize("path", ["rows", "swap", "pair", "decode"], indirect=True)
@pytest.mark.parametrize("shape", SMALL_SHAPES)
def test_forward_bf16_parity(moe, shape, path):
    out, ref = _forward_case(moe, shape)
    err = O.rel_max_err(out, ref)
    assert err <= BF16_TOL, err
    assert np.all(np.isfinite(out))


@pytest.mark.parametrize("pair", [0, 3], ids=["swap_down", "pair_down"])
@pytest.mark.parametrize("phases", [2, 4])
def test_forward_bf16_down_gemm_phases(moe, phases, pair):
    """The down GEMM's output columns in 2 or 4 slices run one after the
    other (the order used when the fp32 accumulator exceeds L2), on the
    one-CTA swap-AB kernel and on CTA pairs: every tile still runs exactly
    once."""
    from full_size_sampling import check_accumulator
    shape = MoEShape(T=300, H=1024, I=384, E=6, k=3)
    moe.set_down_phases(phases)
    moe.set_pair_gemm(pair)
    try:
        out, ref = _forward_case(moe, shape)
    finally:
        moe.set_down_phases(-1)
        moe.set_pair_gemm(-1)
    # 307 k outputs: checked on the fp32 accumulator, the bf16 output its
    # exact RNE image (see tests/full_size_sampling.py)
    out_t = torch.from_numpy(out).to(torch.bfloat16).cuda()
    check_accumulator(moe, out_t, np.arange(shape.T), ref, shape, moe.W_BF16, BF16_TOL)


@pytest.mark.parametrize("bits", [1, 2, 3])
def test_forward_bf16_down_l2_hints(moe, bits):
    """Down GEMM with L2 policies on the accumulator reductions and/or the
    weight loads: the same result, checked like any forward."""
    from full_size_sampling import check_accumulator
    shape = MoEShape(T=300, H=1024, I=384, E=6, k=3)
    moe.set_down_l2_hints(bits)
    try:
        out, ref = _forward_case(moe, shape)
    finally:
        moe.set_down_l2_hints(-1)
    out_t = torch.from_numpy(out).to(torch.bfloat16).cuda()
    check_accumulator(moe, out_t, np.arange(shape.T), ref, shape, moe.W_BF16, BF16_TOL)


@pytest.mark.parametrize("mask", [1, 2, 3])
@pytest.mark.parametrize("group", [0, 1, 2])
@pytest.mark.parametrize("shape", [
    MoEShape(T=1200, H=512, I=256, E=2, k=1),     # 600 rows per expert: three 200-token pair tiles
    MoEShape(T=700, H=256, I=384, E=8, k=3),      # 262 rows per expert on average: ragged pair tiles
    MoEShape(T=37, H=768, I=128, E=16, k=4),      # 9 rows per expert: 16-column tiles, one half-step
])
def test_forward_bf16_pair_gemms(moe, mask, group, shape):
    """Gate/up (mask 1), down (mask 2) or both on CTA pairs, with the token
    tiles of an expert in groups of 0 (all), 1 or 2: every tile runs once,
    both CTAs' halves of the tokens and of the weight rows land in place."""
    from full_size_sampling import check_accumulator
    moe.set_decode_rows(0)
    moe.set_pair_gemm(mask)
    moe.set_tile_group(group)
    try:
        out, ref = _forward_case(moe, shape)
    finally:
        moe.set_decode_rows(-1)
        moe.set_pair_gemm(-1)
        moe.set_tile_group(-1)
    out_t = torch.from_numpy(out).to(torch.bfloat16).cuda()
    check_accumulator(moe, out_t, np.arange(shape.T), ref, shape, moe.W_BF16, BF16_TOL)


@pytest.mark.parametrize("path", ["rows", "swap", "pair"], indirect=True)
def test_forward_bf16_parity_qwen_shape_520_tokens(moe, path):
    out, ref = _forward_case(moe, MoEShape(T=520, H=2048, I=1408, E=60, k=4))
    assert O.rel_max_err(out, ref) <= BF16_TOL


@pytest.mark.parametrize("path", ["rows", "swap", "pair", "decode"], indirect=True)
def test_forward_bf16_one_expert_takes_all(moe, path):
    shape = MoEShape(T=700 if path != "decode" else 90, H=256, I=256, E=8, k=2)
    bias = torch.zeros(8)
    bias[5] = 30.0                                  # every token routes to expert 5
    out, ref = _forward_case(moe, shape, logit_bias=bias)
    assert O.rel_max_err(out, ref) <= BF16_TOL


@pytest.mark.parametrize("path", ["decode"], indirect=True)
@pytest.mark.parametrize("shape", [
    MoEShape(T=2, H=7168, I=256, E=8, k=8),        # DeepSeek-V3 width, every expert touched
    MoEShape(T=16, H=256, I=128, E=4, k=1),        # several tokens per expert
    MoEShape(T=16, H=128, I=256, E=1, k=1),        # 16 tokens on one expert: 2 token chunks
    MoEShape(T=4, H=2048, I=1408, E=60, k=4),      # Qwen width at the default threshold
    MoEShape(T=8, H=256, I=2048, E=8, k=4),        # the widest h rows (2048) at 8 tokens per expert
])
@pytest.mark.parametrize("single", [True, False], ids=["one_kernel", "two_kernels"])
def test_forward_bf16_fused_decode(moe, shape, path, single):
    """Few routed rows: the routing table is rebuilt inside the kernels, so
    no dispatch or combine kernel runs: one cooperative kernel (gate/up,
    then down + combine) or the two fused kernels, including the widest
    rows and the most tokens per expert they see."""
    moe.set_decode_single(single)
    try:
        n0 = moe.launch_count()
        out, ref = _forward_case(moe, shape)
        launches = moe.launch_count() - n0
    finally:
        moe.set_decode_single(False)
    assert launches == (1 if single else 2)
    assert O.rel_max_err(out, ref) <= BF16_TOL


@pytest.mark.parametrize("act", ["gelu", "relu"])
@pytest.mark.parametrize("path", ["rows", "swap", "decode"], indirect=True)
@pytest.mark.parametrize("shape", [
    shape_for("tiny"),
    MoEShape(T=300, H=256, I=384, E=6, k=3),
    MoEShape(T=3, H=128, I=128, E=2, k=2),         # fused decode kernels
])
def test_forward_bf16_geglu_reglu(moe, shape, path, act):
    """GeGLU (exact GELU) and ReGLU experts on every bf16 path."""
    out, ref = _forward_case(moe, shape, act=act)
    assert O.rel_max_err(out, ref) <= BF16_TOL


def test_forward_rejects_unknown_activation(moe):
    d = make_inputs(MoEShape(T=4, H=128, I=128, E=2, k=1), seed=0, device="cuda")
    idx, w = moe.route(d["logits"], 1)
    with pytest.raises(ValueError):
        moe.experts_forward(d["hidden"], idx, w, d["w_gate_up"], d["w_down"], activation="tanh")


def test_profile_read_after_graph_replays(moe):
    """Stage events captured in a CUDA graph report each replay's stage
    times through profile_read; eager profiling sums every launch."""
    shape = MoEShape(T=256, H=256, I=256, E=8, k=2)
    d = make_inputs(shape, seed=2, device="cuda")
    idx, w = moe.route(d["logits"], shape.k)
    out = torch.empty(shape.T, shape.H, dtype=torch.bfloat16, device="cuda")
    ws = moe.Workspace("cuda")
    run = lambda: moe.experts_forward(d["hidden"], idx, w, d["w_gate_up"], d["w_down"],
                                      out=out, workspace=ws)
    run()
    torch.cuda.synchronize()
    moe.profile_begin()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run()
    for _ in range(3):
        g.replay()
        torch.cuda.synchronize()
        st = moe.profile_read()
        assert all(st[k][1] == 1 and st[k][0] > 0 for k in ("dispatch", "gemm1", "gemm2", "finish"))
    moe.profile_end()
    moe.profile_begin()
    run()
    run()
    st = moe.profile_end()
    assert st["gemm1"][1] == 2 and st["gemm2"][1] == 2
    moe.workspace_status(ws)


def test_all_paths_agree(moe):
    shape = MoEShape(T=96, H=512, I=384, E=16, k=4)
    d = make_inputs(shape, seed=5, device="cuda")
    idx, w = moe.route(d["logits"], shape.k)
    outs = []
    for dec, swap, pair in PATHS.values():
        moe.set_decode_rows(dec)
        moe.set_swap_rows(swap)
        moe.set_pair_gemm(pair)
        outs.append(moe.experts_forward(d["hidden"], idx, w, d["w_gate_up"], d["w_down"]).float())
    moe.set_decode_rows(-1)
    moe.set_swap_rows(-1)
    moe.set_pair_gemm(-1)
    # every path is within BF16_TOL * rms of the oracle, so two paths agree
    # within twice that (triangle inequality); in practice they differ by a
    # one-ulp bf16 flip at the largest outputs, about 2 % of rms
    ref = outs[0].pow(2).mean().sqrt().item()
    for o in outs[1:]:
        assert (outs[0] - o).abs().max().item() <= 2 * BF16_TOL * ref


@pytest.mark.parametrize("T", [1, 8, 32, 128])
def test_forward_bf16_decode_workloads_full(moe, T):
    """The Qwen-shaped decode workloads at their full size, every token
    checked against the oracle, through the default path choice."""
    shape = shape_for("qwen", T)
    d = make_inputs(shape, seed=0, device="cuda")
    idx, w = moe.route(d["logits"], shape.k)
    out = moe.experts_forward(d["hidden"], idx, w, d["w_gate_up"], d["w_down"])
    moe.workspace_status(moe.default_workspace())
    ref_idx, ref_w = O.route(d["logits"].cpu().numpy(), shape.k)
    assert np.array_equal(idx.cpu().numpy(), ref_idx)
    experts = np.unique(ref_idx)
    remap = np.full(shape.E, -1, np.int64)
    remap[experts] = np.arange(len(experts))
    ex_t = torch.from_numpy(experts).long().cuda()
    ref = O.forward(d["hidden"].float().cpu().numpy(), remap[ref_idx].astype(np.int32),
                    w.cpu().numpy(), d["w_gate_up"].index_select(0, ex_t).float().cpu().numpy(),
                    d["w_down"].index_select(0, ex_t).float().cpu().numpy())
    assert O.rel_max_err(out.float().cpu().numpy(), ref) <= BF16_TOL


def test_forward_bf16_zero_tokens(moe):
    h = torch.empty(0, 128, dtype=torch.bfloat16, device="cuda")
    out = moe.experts_forward(h, torch.empty(0, 2, dtype=torch.int32, device="cuda"),
                              torch.empty(0, 2, device="cuda"),
                              torch.zeros(4, 256, 128, dtype=torch.bfloat16, device="cuda"),
                              torch.zeros(4, 128, 128, dtype=torch.bfloat16, device="cuda"))
    assert out.shape == (0, 128)


def test_forward_bf16_repeatable_and_token_order_equivariant(moe):
    shape = MoEShape(T=256, H=256, I=256, E=8, k=2)
    d = make_inputs(shape, seed=3)
    idx, w = O.route(d["logits"].numpy(), 2)
    args = [torch.from_numpy(idx).cuda(), torch.from_numpy(w.astype(np.float32)).cuda(),
            d["w_gate_up"].cuda(), d["w_down"].cuda()]
    h = d["hidden"].cuda()
    a = moe.experts_forward(h, *args).float()
    perm = torch.randperm(256, generator=torch.Generator().manual_seed(1))
    b = moe.experts_forward(h[perm.cuda()].contiguous(), args[0][perm.cuda()].contiguous(),
                            args[1][perm.cuda()].contiguous(), args[2], args[3]).float()
    ref = a[perm.cuda()]
    # fp32 atomics may add the k terms in another order: tiny differences only
    assert (b - ref).abs().max().item() <= 1e-2 * ref.pow(2).mean().sqrt().item()


@pytest.mark.parametrize("name,T,pair", [("qwen", 4096, -1), ("dsv3", 8192, -1),
                                         ("qwen", 4096, 3), ("dsv3", 8192, 3)])
def test_forward_bf16_full_size_every_tile(moe, name, T, pair):
    """Full workload size on the GPU, through the default path choice; the
    oracle recomputes the tokens at the edges of every grouped-GEMM tile of
    the busiest expert (63 tiles of 128 rows for the skewed DeepSeek-V3
    layer) and the first and last token of every other touched expert.  The
    fp32 accumulator is checked against it, and the bf16 output against the
    accumulator (bit for bit)."""
    from full_size_sampling import (bf16_expert_fn, check_accumulator, oracle_on_tokens,
                                    probe_tokens, tile_count)
    shape = shape_for(name, T)
    d = make_inputs(shape, seed=0, device="cuda")
    idx, w = moe.route(d["logits"], shape.k)
    moe.set_pair_gemm(pair)       # -1: the library's default kernels; 3: both GEMMs on CTA pairs
    try:
        out = moe.experts_forward(d["hidden"], idx, w, d["w_gate_up"], d["w_down"])
        moe.workspace_status(moe.default_workspace())
    finally:
        moe.set_pair_gemm(-1)
    ref_idx, ref_w = O.route(d["logits"].cpu().numpy(), shape.k)
    assert np.array_equal(idx.cpu().numpy(), ref_idx)
    np.testing.assert_allclose(w.cpu().numpy(), ref_w, rtol=2e-6, atol=1e-7)
    toks, counts, hot, reached = probe_tokens(ref_idx, shape.E, shape.k)
    assert reached == tile_count(int(counts[hot]))
    tt = torch.from_numpy(toks).cuda()
    ref = oracle_on_tokens(toks, ref_idx, ref_w, d["hidden"][tt].float().cpu().numpy(),
                           bf16_expert_fn(d["w_gate_up"], d["w_down"]))
    check_accumulator(moe, out, toks, ref, shape, moe.W_BF16, BF16_TOL)


def _replay_case(moe, shape, seeds, fp8=None):
    """Router + experts_forward captured once as a CUDA graph on fixed device
    buffers; every replay follows a copy of new logits and hidden rows into
    those buffers.  Yields (out after the replay, oracle output)."""
    base = make_inputs(shape, seed=seeds[0], device="cpu")
    wgu, wd = base["w_gate_up"].cuda(), base["w_down"].cuda()
    kw = dict(w_gate_up=wgu, w_down=wd)
    if fp8 is not None:
        qgu, sgu = moe.quantize_fp8_blocks(wgu, fp8)
        qd, sd = moe.quantize_fp8_blocks(wd, fp8)
        kw = dict(w_gate_up=qgu, w_down=qd, scale_gate_up=sgu, scale_down=sd, scale_fmt=fp8)
    logits = base["logits"].cuda()
    hidden = base["hidden"].cuda()
    out = torch.empty(shape.T, shape.H, dtype=torch.bfloat16, device="cuda")
    ws = moe.Workspace("cuda")

    def step():
        idx, w = moe.route(logits, shape.k)
        moe.experts_forward(hidden, idx, w, out=out, workspace=ws, **kw)

    step()                                       # lazy set-up outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for seed in seeds[1:]:
        d = make_inputs(shape, seed=seed, device="cpu")
        logits.copy_(d["logits"].cuda())
        hidden.copy_(d["hidden"].cuda())
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        moe.workspace_status(ws)
        ref_idx, ref_w = O.route(d["logits"].numpy(), shape.k)
        hid = d["hidden"].float().numpy()
        if fp8 is None:
            ref = O.forward(hid, ref_idx, ref_w, base["w_gate_up"].float().numpy(),
                            base["w_down"].float().numpy())
        else:
            ref = O.forward_fp8(hid, ref_idx, ref_w, qgu.cpu().numpy(), sgu.cpu().numpy(),
                                qd.cpu().numpy(), sd.cpu().numpy(), fp8)
        yield out.float().cpu().numpy(), ref


@pytest.mark.parametrize("path,shape", [
    ("rows", MoEShape(T=300, H=256, I=384, E=6, k=3)),
    ("swap", MoEShape(T=300, H=256, I=384, E=6, k=3)),
    ("pair", MoEShape(T=300, H=256, I=384, E=6, k=3)),
    ("decode", MoEShape(T=4, H=512, I=256, E=16, k=4)),      # the two fused decode kernels
    ("decode", MoEShape(T=40, H=512, I=256, E=16, k=4)),     # dispatch, two GEMVs, combine
], indirect=["path"])
def test_graph_replay_matches_oracle(moe, shape, path):
    """What the benchmark times: the whole step as a replayed CUDA graph,
    every kernel chained by programmatic dependent launch (the small decode
    batch as one cooperative kernel).  Each replay's output (after new
    inputs were copied into the captured buffers) must match the oracle on
    those inputs."""
    n = 0
    for got, ref in _replay_case(moe, shape, seeds=(20, 21, 22)):
        assert O.rel_max_err(got, ref) <= BF16_TOL
        n += 1
    assert n == 2


def test_decode_single_kernel_repeats_and_recovers(moe):
    """The one-kernel decode path synchronises its CTAs through two counters
    in the workspace head, which every launch leaves at zero: many launches
    in a row on one workspace (eager and replayed) all give the oracle's
    output, and the counters read zero afterwards."""
    shape = MoEShape(T=1, H=2048, I=1408, E=60, k=4)
    d = make_inputs(shape, seed=9, device="cuda")
    idx, w = moe.route(d["logits"], shape.k)
    ws = moe.Workspace("cuda")
    moe.set_decode_single(True)
    out = torch.empty(1, shape.H, dtype=torch.bfloat16, device="cuda")
    run = lambda: moe.experts_forward(d["hidden"], idx, w, d["w_gate_up"], d["w_down"], out=out,
                                      workspace=ws)
    outs = []
    for _ in range(20):
        run()
        outs.append(out.clone())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run()
    for _ in range(20):
        g.replay()
    torch.cuda.synchronize()
    moe.set_decode_single(False)
    moe.workspace_status(ws)
    head = ws.buf[:16].view(torch.int32).cpu().tolist()
    assert head[:3] == [0, 0, 0]
    ref_idx, ref_w = O.route(d["logits"].cpu().numpy(), shape.k)
    experts = np.unique(ref_idx)
    remap = np.full(shape.E, -1, np.int64)
    remap[experts] = np.arange(len(experts))
    et = torch.from_numpy(experts).long().cuda()
    ref = O.forward(d["hidden"].float().cpu().numpy(), remap[ref_idx].astype(np.int32), ref_w,
                    d["w_gate_up"].index_select(0, et).float().cpu().numpy(),
                    d["w_down"].index_select(0, et).float().cpu().numpy())
    for o in outs + [out]:
        assert torch.equal(o, outs[0])               # fixed summation order: bit-identical
    assert O.rel_max_err(out.float().cpu().numpy(), ref) <= BF16_TOL


@pytest.mark.parametrize("fmt", ["f32", "ue8m0"])
def test_graph_replay_matches_oracle_fp8(moe, fmt):
    shape = MoEShape(T=300, H=512, I=384, E=6, k=3)
    for got, ref in _replay_case(moe, shape, seeds=(30, 31, 32), fp8=fmt):
        assert O.rel_max_err(got, ref) <= 6e-2


# ----------------------------------------------------------------- error paths
def test_forward_rejects_unsupported(moe):
    h = torch.zeros(4, 100, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(moe.MoEError) as ei:
        moe.experts_forward(h, torch.zeros(4, 2, dtype=torch.int32, device="cuda"),
                            torch.zeros(4, 2, device="cuda"),
                            torch.zeros(4, 256, 100, dtype=torch.bfloat16, device="cuda"),
                            torch.zeros(4, 100, 128, dtype=torch.bfloat16, device="cuda"))
    assert ei.value.status == 2


@pytest.mark.parametrize("path", ["rows", "swap", "decode"], indirect=True)
def test_forward_bad_expert_index_reported(moe, path):
    shape = MoEShape(T=16, H=128, I=128, E=4, k=2)
    d = make_inputs(shape, seed=1, device="cuda")
    idx = torch.zeros(16, 2, dtype=torch.int32, device="cuda")
    idx[:, 1] = 1
    idx[5, 1] = 9
    ws = moe.Workspace("cuda")
    moe.experts_forward(d["hidden"], idx, torch.full((16, 2), 0.5, device="cuda"),
                        d["w_gate_up"], d["w_down"], workspace=ws)
    with pytest.raises(moe.MoEError) as ei:
        moe.workspace_status(ws)
    assert ei.value.status == 1
    moe.workspace_status(ws)          # cleared


def test_device_wait_timeout_is_reported_not_hung(moe):
    st = moe.selftest_wait_timeout(limit_us=5000)
    assert st == 4
    # the context is still usable
    x = torch.ones(10, device="cuda")
    assert float(x.sum()) == 10.0
