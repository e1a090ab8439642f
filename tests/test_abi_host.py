"""Host-side checks of the C ABI that need no GPU: the library builds for
sm_103a, loads, exports every function include/moe_experts.h declares, and
rejects bad arguments before touching the device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_experts.h")


@pytest.fixture(scope="module")
def L():
    from mixture_experts_routed_top_gb300 import build, lib
    build.build()
    return lib()


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)))


def test_header_declares_the_entry_points():
    names = _declared()
    for n in ("moe_route", "moe_dispatch", "moe_experts_forward", "moe_workspace_size",
              "moe_quantize_fp8_blocks", "moe_quantize_fp4_blocks", "moe_last_error"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    for n in _declared():
        assert hasattr(L, n), n


def test_version_and_sizes(L):
    assert L.moe_version() >= 100
    a = L.moe_workspace_size(64, 128, 256, 8, 2, 0)
    b = L.moe_workspace_size(4096, 2048, 1408, 60, 4, 0)
    assert 0 < a < b
    # x_perm (T*k*H bf16) + h (T*k*I bf16) + fp32 accumulator dominate
    assert b >= 4096 * 4 * (2048 + 1408) * 2 + 4096 * 2048 * 4
    f8 = L.moe_workspace_size(4096, 2048, 1408, 60, 4, 1)
    assert f8 < b
    assert L.moe_workspace_size(-1, 128, 128, 8, 2, 0) == 0


def test_argument_errors_without_device(L):
    nul = ctypes.c_void_p(0)
    assert L.moe_route(nul, 4, 0, 1, nul, nul, nul) == 2          # E < 1
    assert L.moe_route(nul, 4, 8, 9, nul, nul, nul) == 2          # k > E
    assert L.moe_route(nul, 4, 2000, 2, nul, nul, nul) == 2       # E > 1024
    assert L.moe_route(nul, 4, 8, 2, nul, nul, nul) == 1          # null pointers
    assert b"null" in L.moe_last_error()
    assert L.moe_route(nul, 0, 8, 2, nul, nul, nul) == 0          # T = 0 no-op
    f = L.moe_experts_forward
    # H not a multiple of 128
    assert f(nul, 4, 100, nul, nul, 8, 2, 128, nul, nul, 0, nul, nul, 0, nul, nul, 0, nul) == 2
    # FP8 weights without a scale format
    assert f(nul, 4, 128, nul, nul, 8, 2, 128, nul, nul, 1, nul, nul, 0, nul, nul, 0, nul) == 1
    # bf16 weights with a scale format
    assert f(nul, 4, 128, nul, nul, 8, 2, 128, nul, nul, 0, nul, nul, 1, nul, nul, 0, nul) == 1
    # workspace too small (checked before any launch); fake aligned pointers
    p = ctypes.c_void_p(1 << 20)
    assert f(p, 4, 128, p, p, 8, 2, 128, p, p, 0, nul, nul, 0, p, p, 16, nul) == 5
    fa = L.moe_experts_forward_act
    # unknown gate activation (checked first); the three named ones pass that check
    assert fa(p, 4, 128, p, p, 8, 2, 128, p, p, 0, nul, nul, 0, 3, p, p, 16, nul) == 1
    assert b"activation" in L.moe_last_error()
    for act in (0, 1, 2):
        assert fa(p, 4, 128, p, p, 8, 2, 128, p, p, 0, nul, nul, 0, act, p, p, 16, nul) == 5
    assert L.moe_quantize_fp8_blocks(nul, 1, 100, 128, 1, nul, nul, nul) == 2
    assert L.moe_quantize_fp8_blocks(nul, 1, 128, 128, 0, nul, nul, nul) == 1


def test_fp4_argument_errors_without_device(L):
    nul = ctypes.c_void_p(0)
    p = ctypes.c_void_p(1 << 20)
    f = L.moe_experts_forward
    # FP4 weights (wdtype 2) take UE8M0 scales only
    for sf in (0, 1):
        assert f(p, 4, 128, p, p, 8, 2, 128, p, p, 2, p, p, sf, p, p, 1 << 30, nul) == 1
    assert b"UE8M0" in L.moe_last_error()
    # ... and need both scale buffers
    assert f(p, 4, 128, p, p, 8, 2, 128, p, p, 2, nul, p, 2, p, p, 1 << 30, nul) == 1
    # above 64 routed rows FP4 runs on the block-scaled tensor-core GEMMs,
    # whose 256-wide down tiles need H % 256 == 0 ...
    assert f(p, 33, 128, p, p, 8, 2, 128, p, p, 2, p, p, 2, p, p, 1 << 30, nul) == 2
    assert b"H % 256" in L.moe_last_error()
    # ... and 32-byte aligned packed weights (TMA of packed e2m1)
    p16 = ctypes.c_void_p((1 << 20) + 16)
    assert f(p, 33, 256, p, p, 8, 2, 128, p16, p, 2, p, p, 2, p, p, 1 << 30, nul) == 1
    assert b"32-byte" in L.moe_last_error()
    assert f(p, 33, 256, p, p, 8, 2, 128, p, p, 2, p, p, 2, p, p, 16, nul) == 5
    # by default even one routed row takes the GEMMs (alignment checked) ...
    assert L.moe_get_fp4_gemv_rows() == 0
    assert f(p, 1, 256, p, p, 8, 1, 128, p16, p, 2, p, p, 2, p, p, 1 << 30, nul) == 1
    # ... unless the GEMV threshold covers the batch (then no alignment rule)
    L.moe_set_fp4_gemv_rows(64)
    try:
        assert L.moe_get_fp4_gemv_rows() == 64
        assert f(p, 1, 256, p, p, 8, 1, 128, p16, p, 2, p, p, 2, p, p, 16, nul) == 5
    finally:
        L.moe_set_fp4_gemv_rows(-1)
    L.moe_set_fp4_gemv_rows(1000)
    assert L.moe_get_fp4_gemv_rows() == 64            # clamped
    L.moe_set_fp4_gemv_rows(-1)
    # T*k = 64 passes those checks and stops at the workspace size
    assert f(p, 32, 128, p, p, 8, 2, 128, p, p, 2, p, p, 2, p, p, 16, nul) == 5
    need = L.moe_workspace_size(32, 128, 128, 8, 2, 2)
    # quantised activations [T, H] and h [T*k, I] are kept in fp32
    assert need >= 32 * 128 * 4 + 64 * 128 * 4
    assert L.moe_quantize_fp4_blocks(nul, 1, 4, 48, nul, nul, nul) == 2    # cols % 32
    assert L.moe_quantize_fp4_blocks(nul, 1, 4, 64, nul, nul, nul) == 1    # null pointers
    assert L.moe_quantize_fp4_blocks(nul, 0, 4, 64, nul, nul, nul) == 0    # empty


def test_block_scaled_mma_setting_and_accumulator_offset(L):
    assert L.moe_get_block_scaled_mma() == 1
    L.moe_set_block_scaled_mma(0)
    assert L.moe_get_block_scaled_mma() == 0
    L.moe_set_block_scaled_mma(1)
    for wd in (0, 1, 2):
        off = L.moe_workspace_accumulator_offset(300, 256, 128, 8, 2, wd)
        assert off % 1024 == 0 and 0 < off
        assert off + 300 * 256 * 4 <= L.moe_workspace_size(300, 256, 128, 8, 2, wd)
    assert L.moe_workspace_accumulator_offset(-1, 256, 128, 8, 2, 0) == 0


def test_decode_rows_setting(L):
    L.moe_set_decode_rows(77)
    assert L.moe_get_decode_rows() == 77
    L.moe_set_decode_rows(-1)


def test_pair_gemm_setting(L):
    assert L.moe_get_pair_gemm() == -1          # the library default
    for m in (0, 1, 2, 3):
        L.moe_set_pair_gemm(m)
        assert L.moe_get_pair_gemm() == m
    L.moe_set_pair_gemm(7)
    assert L.moe_get_pair_gemm() == 3           # two bits only
    L.moe_set_pair_gemm(-5)
    assert L.moe_get_pair_gemm() == -1


def test_down_l2_hints_setting(L):
    assert L.moe_get_down_l2_hints() == 1       # accumulator evict_last by default
    L.moe_set_down_l2_hints(2)
    assert L.moe_get_down_l2_hints() == 2
    L.moe_set_down_l2_hints(0)
    assert L.moe_get_down_l2_hints() == 0
    L.moe_set_down_l2_hints(-1)
    assert L.moe_get_down_l2_hints() == 1
