"""Host-side arithmetic of bench.py that every reported roofline fraction
depends on: algorithmic flops and bytes of a step, the peak table and the
ncu traffic lookup.  CPU only."""
import json
import os

import numpy as np
import pytest

import bench
from workloads import shape_for


def _w(name, T, wfmt="bf16", sfmt=None):
    return {"shape": shape_for(name, T), "wfmt": wfmt, "sfmt": sfmt}


def test_algorithmic_bf16_counts_routed_rows_and_touched_experts():
    w = _w("qwen", 4096)
    s = w["shape"]
    counts = np.full(s.E, 4096 * 4 // s.E)
    counts[7] = 0                                   # one expert untouched
    flops, wbytes, io, touched = bench.algorithmic(w, counts)
    assert flops == 6.0 * 2048 * 1408 * 4096 * 4    # 6 H I per routed row
    assert touched == s.E - 1
    assert wbytes == (s.E - 1) * 3 * 2048 * 1408 * 2
    assert io == 4096 * 2048 * 2 * 2 + 4096 * 60 * 4


@pytest.mark.parametrize("sfmt,per", [("f32", 4), ("ue8m0", 1)])
def test_algorithmic_fp8_weight_bytes_include_block_scales(sfmt, per):
    w = _w("dsv3_fp8", 64, "fp8", sfmt)
    s = w["shape"]
    counts = np.zeros(s.E, np.int64)
    counts[:10] = 1
    _, wbytes, _, touched = bench.algorithmic(w, counts)
    scales = (2 * s.I // 128) * (s.H // 128) * per + (s.H // 128) * (s.I // 128) * per
    assert touched == 10
    assert wbytes == 10 * (3 * s.H * s.I + scales)


def test_peaks_have_both_denominators():
    peaks, src = bench.load_peaks()
    assert src in ("measured", "fallback")
    assert peaks["hbm_gbs"] > 1000 and peaks["bf16_tflops"] > 100


def test_traffic_lookup_follows_the_kernel_source():
    assert bench.traffic_for("gemm1:no-such-workload") is None
    d = json.load(open(os.path.join(bench.ROOT, "profiles", "traffic.json")))
    for key, ent in d.items():
        if key.startswith("_"):
            continue
        got = bench.traffic_for(key)
        # either the kernel source still hashes as captured, or the entry is ignored
        assert got in (None, ent["bytes_per_launch"])
        assert ent["bytes_per_launch"] == ent["read"] + ent["write"]


def test_algorithmic_fp4_weight_bytes_are_half_bytes_plus_block_scales():
    w = _w("qwen", 1, "fp4", "ue8m0")
    s = w["shape"]
    counts = np.zeros(s.E, np.int64)
    counts[[3, 9, 17, 40]] = 1
    flops, wbytes, _, touched = bench.algorithmic(w, counts)
    assert touched == 4
    assert flops == 6.0 * s.H * s.I * 4
    # 4 bits per weight and one UE8M0 byte per 32 weights
    assert wbytes == 4 * (3 * s.H * s.I / 2 + 3 * s.H * s.I / 32)


def test_fp4_workloads_fit_their_path():
    """FP4 workloads use UE8M0 scales; those above 64 routed rows run on the
    block-scaled GEMMs, whose 256-wide down tiles need H % 256 == 0."""
    for name, (sname, T, wfmt, sfmt) in bench.WORKLOADS.items():
        if wfmt == "fp4":
            s = shape_for(sname, T)
            assert sfmt == "ue8m0", name
            assert s.T * s.k <= 64 or s.H % 256 == 0, name


@pytest.mark.parametrize("wfmt", ["bf16", "fp8", "fp4"])
def test_oracle_sample_runs_on_every_weight_format(wfmt):
    """The CPU legs of bench.py (cpu_baseline and the reference arm) on a
    tiny workload held in host memory, with the quantised weights made by
    the oracle's quantisers: the sample selects tokens, copies their experts
    and runs the matching oracle forward."""
    import torch
    import oracle as O
    from workloads import MoEShape, make_inputs
    s = MoEShape(T=8, H=256, I=128, E=4, k=2)
    d = make_inputs(s, seed=0, device="cpu")
    w = {"shape": s, "wfmt": wfmt, "sfmt": {"bf16": None, "fp8": "f32", "fp4": "ue8m0"}[wfmt],
         "logits": d["logits"], "hidden": d["hidden"], "w_gate_up": d["w_gate_up"],
         "w_down": d["w_down"]}
    if wfmt == "fp8":
        q, sc, _ = O.quantize_blocks(d["w_gate_up"].float().numpy(), 128, 128, "f32")
        qd, sd, _ = O.quantize_blocks(d["w_down"].float().numpy(), 128, 128, "f32")
    elif wfmt == "fp4":
        q, sc, _ = O.quantize_fp4_blocks(d["w_gate_up"].float().numpy())
        qd, sd, _ = O.quantize_fp4_blocks(d["w_down"].float().numpy())
    if wfmt != "bf16":
        w.update(q_gate_up=torch.from_numpy(q), s_gate_up=torch.from_numpy(sc),
                 q_down=torch.from_numpy(qd), s_down=torch.from_numpy(sd))
    smp = bench.OracleSample(w, 4)
    assert smp.n == 4
    assert smp.run() > 0.0


def test_dominant_roof_is_the_one_that_binds():
    """The roofline time is max(flops / tensor peak, bytes / HBM bandwidth):
    the Qwen-shaped gate/up GEMM (E=60, every expert touched) moves more
    bytes than its flops take at the tensor peak, the DeepSeek-V3-shaped one
    the reverse; decode batches stream weights.  The tensor peak is the
    sustained measurement (the timed loops run back to back)."""
    peaks = {"hbm_gbs": 6705.2, "bf16_tflops": 1886.7, "bf16_tflops_sustained": 1737.5}

    def roof(sname, T, wfmt, sfmt, dominant, touched):
        w = _w(sname, T, wfmt, sfmt)
        s = w["shape"]
        counts = np.zeros(s.E, np.int64)
        counts[:touched] = 1
        flops, wbytes, _, _ = bench.algorithmic(w, counts)
        return bench.dominant_roof(w, dominant, flops, wbytes, peaks), w["shape"]

    (f, b, wb, pk, hbm), s = roof("qwen", 4096, "bf16", None, "gemm1", 60)
    assert f == 4.0 * s.H * s.I * s.T * s.k
    # weights (gate and up rows of 60 experts), X rows in, h rows out
    assert b == 60 * 2 * s.H * s.I * 2 + s.T * s.k * (s.H + s.I) * 2
    assert hbm and pk == 1737.5
    (f, b, wb, pk, hbm), s = roof("dsv3", 8192, "bf16", None, "gemm1", 192)
    assert not hbm
    (f, b, wb, pk, hbm), s = roof("dsv3", 8192, "bf16", None, "gemm2", 192)
    assert b == 192 * s.H * s.I * 2 + s.T * s.k * s.I * 2 + s.T * s.H * 4
    (f, b, wb, pk, hbm), s = roof("qwen", 32, "bf16", None, "gemm1", 50)
    assert hbm
    (f, b, wb, pk, hbm), s = roof("dsv3_fp8", 16384, "fp8", "f32", "gemm1", 214)
    assert not hbm and pk == 2 * 1737.5


def test_roof_entry_reports_sustained_and_burst_fractions():
    """Tensor-bound lines: achieved = flops per launch / launch time, against
    the sustained rate, with the burst fraction beside it (x2 for the
    FP8-rate MMAs); HBM-bound lines against the copy bandwidth."""
    peaks = {"hbm_gbs": 6705.2, "bf16_tflops": 1886.7, "bf16_tflops_sustained": 1737.5}
    w = _w("dsv3", 8192, "bf16", None)
    s = w["shape"]
    counts = np.zeros(s.E, np.int64)
    counts[:194] = 1                 # the bench workload's touched experts
    flops, wbytes, _, _ = bench.algorithmic(w, counts)
    f, b, _, pk, hbm = bench.dominant_roof(w, "gemm1", flops, wbytes, peaks)
    r = bench.roof_entry(w, hbm, f, b, 3.364e-3, pk, peaks)
    assert r["bound"] == "tensor" and r["peak"] == 1737.5 and r["peak_burst"] == 1886.7
    assert abs(r["achieved"] - f / 3.364e-3 / 1e12) < 0.06
    assert abs(r["frac"] - r["achieved"] / 1737.5) < 1e-4
    assert abs(r["frac_of_burst"] - r["achieved"] / 1886.7) < 1e-4
    w8 = _w("dsv3_fp8", 16384, "fp8", "ue8m0")
    c8 = np.zeros(w8["shape"].E, np.int64)
    c8[:205] = 1
    f8, wb8, _, _ = bench.algorithmic(w8, c8)
    f, b, _, pk, hbm = bench.dominant_roof(w8, "gemm1", f8, wb8, peaks)
    r = bench.roof_entry(w8, hbm, f, b, 3.76e-3, pk, peaks)
    assert r["peak"] == 2 * 1737.5 and r["peak_burst"] == 2 * 1886.7
    wq = _w("qwen", 4096, "bf16", None)
    cq = np.ones(wq["shape"].E, np.int64)
    fq, wbq, _, _ = bench.algorithmic(wq, cq)
    f, b, _, pk, hbm = bench.dominant_roof(wq, "gemm1", fq, wbq, peaks)
    r = bench.roof_entry(wq, hbm, f, b, 0.195e-3, pk, peaks)
    assert hbm and r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert abs(r["frac"] - b / 0.195e-3 / 1e9 / 6705.2) < 1e-4
    assert "frac_of_burst" not in r
