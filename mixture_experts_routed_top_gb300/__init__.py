"""Routed top-k Mixture-of-Experts experts forward for GB300 (sm_103a).

Thin ctypes binding over the C ABI declared in include/moe_experts.h.  It
only checks and marshals arguments: every step of the forward runs in the
library's CUDA kernels.  PyTorch provides device memory and the current
stream.  There is no CPU or eager fallback: if the library is missing or no
CUDA device is present the calls raise.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import torch

from . import build as _build

__all__ = [
    "MoEError", "lib", "route", "dispatch", "dispatch_workspace_size", "workspace_size",
    "experts_forward", "quantize_fp8_blocks", "quantize_fp4_blocks", "workspace_status", "set_decode_rows",
    "get_decode_rows", "set_swap_rows", "get_swap_rows", "profile_begin", "profile_end", "profile_read",
    "selftest_wait_timeout", "launch_count", "accumulator", "set_block_scaled_mma",
    "get_block_scaled_mma", "set_fp4_gemv_rows", "get_fp4_gemv_rows", "set_decode_single",
    "get_decode_single", "set_tile_group", "get_tile_group", "set_pair_gemm", "get_pair_gemm", "set_down_l2_hints", "get_down_l2_hints", "set_down_phases",
    "get_down_phases",
    "Workspace", "STATUS", "STAGES", "W_BF16", "W_FP8_E4M3", "W_FP4_E2M1", "SCALE_NONE", "SCALE_F32",
    "SCALE_UE8M0", "ACTIVATIONS",
]

STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_CUDA",
          4: "MOE_ERR_TIMEOUT", 5: "MOE_ERR_WORKSPACE"}
STAGES = ("dispatch", "gemm1", "gemm2", "finish")
W_BF16, W_FP8_E4M3, W_FP4_E2M1 = 0, 1, 2
SCALE_NONE, SCALE_F32, SCALE_UE8M0 = 0, 1, 2
_SCALE_BY_NAME = {None: SCALE_NONE, "none": SCALE_NONE, "f32": SCALE_F32, "float": SCALE_F32,
                  "ue8m0": SCALE_UE8M0}


class MoEError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS.get(status, status)}: {msg}")
        self.status = status


_LIB = None
_P, _I, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
_SIGS = {
    "moe_version": ([], _I),
    "moe_last_error": ([], ctypes.c_char_p),
    "moe_route": ([_P, _I, _I, _I, _P, _P, _P], _I),
    "moe_dispatch_workspace_size": ([_I, _I, _I], _SZ),
    "moe_dispatch": ([_P, _I, _I, _I, _P, _P, _P, _P, _P, _SZ, _P], _I),
    "moe_workspace_size": ([_I, _I, _I, _I, _I, _I], _SZ),
    "moe_experts_forward": ([_P, _I, _I, _P, _P, _I, _I, _I, _P, _P, _I, _P, _P, _I, _P, _P,
                             _SZ, _P], _I),
    "moe_experts_forward_act": ([_P, _I, _I, _P, _P, _I, _I, _I, _P, _P, _I, _P, _P, _I, _I, _P,
                                 _P, _SZ, _P], _I),
    "moe_quantize_fp8_blocks": ([_P, _I, _I, _I, _I, _P, _P, _P], _I),
    "moe_quantize_fp4_blocks": ([_P, _I, _I, _I, _P, _P, _P], _I),
    "moe_workspace_status": ([_P, _P], _I),
    "moe_set_decode_rows": ([_I], None),
    "moe_get_decode_rows": ([], _I),
    "moe_set_swap_rows": ([_I], None),
    "moe_get_swap_rows": ([], _I),
    "moe_profile_begin": ([], _I),
    "moe_profile_end": ([ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_int), _I], _I),
    "moe_profile_read": ([ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_int), _I], _I),
    "moe_selftest_wait_timeout": ([_P, _SZ, _I, _P], _I),
    "moe_launch_count": ([], ctypes.c_longlong),
    "moe_workspace_accumulator_offset": ([_I, _I, _I, _I, _I, _I], _SZ),
    "moe_set_block_scaled_mma": ([_I], None),
    "moe_get_block_scaled_mma": ([], _I),
    "moe_set_down_l2_hints": ([_I], None),
    "moe_get_down_l2_hints": ([], _I),
    "moe_set_pair_gemm": ([_I], None),
    "moe_get_pair_gemm": ([], _I),
    "moe_set_down_phases": ([_I], None),
    "moe_get_down_phases": ([], _I),
    "moe_set_tile_group": ([_I], None),
    "moe_get_tile_group": ([], _I),
    "moe_set_decode_single": ([_I], None),
    "moe_get_decode_single": ([], _I),
    "moe_set_fp4_gemv_rows": ([_I], None),
    "moe_get_fp4_gemv_rows": ([], _I),
}


def lib_path() -> str:
    return _build.LIB_PATH


def lib(build_if_missing: bool = True):
    """Load libmoe_gb300.so (building it in-tree first if it is absent)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = lib_path()
    if not os.path.isfile(path):
        if not build_if_missing:
            raise RuntimeError(f"CUDA library {path} is not built")
        _build.build()
    L = ctypes.CDLL(path)
    for name, (args, res) in _SIGS.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = res
    _LIB = L
    return L


def _check(status: int):
    if status != 0:
        raise MoEError(status, lib().moe_last_error().decode())


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _need_cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")


# ------------------------------------------------------------------ router
def route(logits: torch.Tensor, k: int, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Top-k routing of fp32 logits [T, E] -> (topk_idx int32 [T,k], topk_w fp32 [T,k])."""
    _need_cuda(logits)
    if logits.dtype != torch.float32 or logits.dim() != 2:
        raise ValueError("logits must be fp32 [T, E]")
    T, E = logits.shape
    idx = torch.empty(T, k, dtype=torch.int32, device=logits.device)
    w = torch.empty(T, k, dtype=torch.float32, device=logits.device)
    _check(lib().moe_route(_ptr(logits), T, E, k, _ptr(idx), _ptr(w), _stream(stream)))
    return idx, w


# ------------------------------------------------------------------ dispatch
def dispatch_workspace_size(T: int, E: int, k: int) -> int:
    return int(lib().moe_dispatch_workspace_size(T, E, k))


def dispatch(topk_idx: torch.Tensor, E: int, stream=None):
    """Expert-contiguous ordering -> (counts [E], offsets [E+1], sorted_f [T*k], row_of [T*k])."""
    _need_cuda(topk_idx)
    if topk_idx.dtype != torch.int32 or topk_idx.dim() != 2:
        raise ValueError("topk_idx must be int32 [T, k]")
    T, k = topk_idx.shape
    dev = topk_idx.device
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    sorted_f = torch.empty(T * k, dtype=torch.int32, device=dev)
    row_of = torch.empty(T * k, dtype=torch.int32, device=dev)
    nbytes = dispatch_workspace_size(T, E, k)
    ws = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=dev)
    _check(lib().moe_dispatch(_ptr(topk_idx), T, E, k, _ptr(counts), _ptr(offsets),
                              _ptr(sorted_f), _ptr(row_of), _ptr(ws), nbytes, _stream(stream)))
    _check(lib().moe_workspace_status(_ptr(ws), _stream(stream)))
    return counts, offsets, sorted_f, row_of


# ------------------------------------------------------------------ forward
def workspace_size(T: int, H: int, I: int, E: int, k: int, wdtype: int = W_BF16) -> int:
    """Bytes of workspace experts_forward needs for these sizes and weight
    type (W_BF16, W_FP8_E4M3 or W_FP4_E2M1)."""
    return int(lib().moe_workspace_size(T, H, I, E, k, wdtype))


class Workspace:
    """Caller-owned device scratch for experts_forward, grown on demand.
    The first 256 bytes hold the device error word; they start zeroed."""

    def __init__(self, device="cuda"):
        self.device = torch.device(device)
        self.buf = None

    def get(self, nbytes: int) -> torch.Tensor:
        if self.buf is None or self.buf.numel() < nbytes:
            self.buf = torch.zeros(max(nbytes, 1024), dtype=torch.uint8, device=self.device)
        return self.buf


_DEFAULT_WS = {}

# moe_activation values
ACTIVATIONS = {"silu": 0, "gelu": 1, "relu": 2}


def experts_forward(hidden: torch.Tensor, topk_idx: torch.Tensor, topk_w: torch.Tensor,
                    w_gate_up: torch.Tensor, w_down: torch.Tensor,
                    scale_gate_up: Optional[torch.Tensor] = None,
                    scale_down: Optional[torch.Tensor] = None, scale_fmt=None,
                    out: Optional[torch.Tensor] = None, workspace: Optional[Workspace] = None,
                    stream=None, activation: str = "silu") -> torch.Tensor:
    """Routed experts forward -> bf16 [T, H].

    hidden bf16 [T,H]; topk_idx int32 [T,k]; topk_w fp32 [T,k];
    w_gate_up [E,2I,H] and w_down [E,H,I], bf16 or e4m3 bytes (uint8 or
    float8_e4m3fn) with 128x128 block scales (scale_fmt 'f32' or 'ue8m0'),
    or packed e2m1 bytes (uint8 or int8) [E,2I,H/2] and [E,H,I/2] with 1x32
    UE8M0 scales from quantize_fp4_blocks; activation: the gate activation,
    'silu' (SwiGLU), 'gelu' (GeGLU, exact erf GELU) or 'relu' (ReGLU)."""
    _need_cuda(hidden, topk_idx, topk_w, w_gate_up, w_down, scale_gate_up, scale_down, out)
    T, H = hidden.shape
    k = topk_idx.shape[1]
    E, twoI, H2 = w_gate_up.shape
    I = twoI // 2
    fp4 = w_gate_up.dtype in (torch.uint8, torch.int8) and 2 * H2 == H
    if fp4:
        if tuple(w_down.shape) != (E, H, I // 2):
            raise ValueError("packed FP4 weight shapes must be [E, 2I, H/2] and [E, H, I/2]")
        if scale_fmt is None:
            scale_fmt = "ue8m0"
    elif H2 != H or tuple(w_down.shape) != (E, H, I):
        raise ValueError("weight shapes must be [E, 2I, H] and [E, H, I]")
    if hidden.dtype != torch.bfloat16 or topk_idx.dtype != torch.int32 or topk_w.dtype != torch.float32:
        raise ValueError("hidden bf16, topk_idx int32, topk_w fp32 expected")
    fp8 = not fp4 and w_gate_up.dtype in (torch.uint8, torch.float8_e4m3fn)
    wdtype = W_FP4_E2M1 if fp4 else W_FP8_E4M3 if fp8 else W_BF16
    if not (fp4 or fp8) and w_gate_up.dtype != torch.bfloat16:
        raise ValueError("weights must be bf16, e4m3 bytes or packed e2m1 bytes")
    sf = _SCALE_BY_NAME[scale_fmt] if not isinstance(scale_fmt, int) else scale_fmt
    if out is None:
        out = torch.empty(T, H, dtype=torch.bfloat16, device=hidden.device)
    nbytes = workspace_size(T, H, I, E, k, wdtype)
    if workspace is None:
        key = hidden.device
        workspace = _DEFAULT_WS.get(key)
        if workspace is None:
            workspace = _DEFAULT_WS.setdefault(key, Workspace(key))
    ws = workspace.get(nbytes)
    if activation not in ACTIVATIONS:
        raise ValueError(f"activation must be one of {sorted(ACTIVATIONS)}")
    _check(lib().moe_experts_forward_act(
        _ptr(hidden), T, H, _ptr(topk_idx), _ptr(topk_w), E, k, I, _ptr(w_gate_up),
        _ptr(w_down), wdtype, _ptr(scale_gate_up), _ptr(scale_down), sf, ACTIVATIONS[activation],
        _ptr(out), _ptr(ws), ws.numel(), _stream(stream)))
    return out


def workspace_status(workspace, stream=None):
    """Synchronise and raise MoEError if a kernel flagged an error in ws."""
    ws = workspace.buf if isinstance(workspace, Workspace) else workspace
    _check(lib().moe_workspace_status(_ptr(ws), _stream(stream)))


def accumulator(workspace, T: int, H: int, I: int, E: int, k: int,
                wdtype: int = W_BF16) -> torch.Tensor:
    """fp32 [T, H] view of the workspace's output accumulator: after a
    grouped-path forward with these sizes it holds the un-rounded output
    (see moe_workspace_accumulator_offset)."""
    ws = workspace.buf if isinstance(workspace, Workspace) else workspace
    off = int(lib().moe_workspace_accumulator_offset(T, H, I, E, k, wdtype))
    if off == 0 or off + T * H * 4 > ws.numel():
        raise ValueError("workspace too small for these sizes")
    return ws[off:off + T * H * 4].view(torch.float32).view(T, H)


def default_workspace(device="cuda") -> Workspace:
    d = torch.device(device)
    if d.index is None:
        d = torch.device("cuda", torch.cuda.current_device())
    return _DEFAULT_WS.setdefault(d, Workspace(d))


# ------------------------------------------------------------------ FP8
def quantize_fp8_blocks(w: torch.Tensor, scale_fmt: str = "f32", stream=None):
    """bf16 [..., R, C] -> (e4m3 codes uint8 [..., R, C], scales [..., R/128, C/128]
    as fp32 ('f32') or uint8 exponent bytes ('ue8m0'))."""
    _need_cuda(w)
    if w.dtype != torch.bfloat16:
        raise ValueError("w must be bf16")
    *lead, R, C = w.shape
    nmat = 1
    for d in lead:
        nmat *= d
    q = torch.empty(w.shape, dtype=torch.uint8, device=w.device)
    sf = _SCALE_BY_NAME[scale_fmt]
    sdt = torch.uint8 if sf == SCALE_UE8M0 else torch.float32
    s = torch.empty(*lead, R // 128 if R % 128 == 0 else 0, C // 128 if C % 128 == 0 else 0,
                    dtype=sdt, device=w.device)
    _check(lib().moe_quantize_fp8_blocks(_ptr(w), nmat, R, C, sf, _ptr(q), _ptr(s),
                                         _stream(stream)))
    return q, s


def quantize_fp4_blocks(w: torch.Tensor, stream=None):
    """bf16 [..., R, C] -> (packed e2m1 codes uint8 [..., R, C/2], two per
    byte with the even element in the low nibble; UE8M0 exponent bytes
    uint8 [..., R, C/32], one per 1x32 block)."""
    _need_cuda(w)
    if w.dtype != torch.bfloat16:
        raise ValueError("w must be bf16")
    *lead, R, C = w.shape
    nmat = 1
    for d in lead:
        nmat *= d
    q = torch.empty(*lead, R, C // 2, dtype=torch.uint8, device=w.device)
    s = torch.empty(*lead, R, C // 32, dtype=torch.uint8, device=w.device)
    _check(lib().moe_quantize_fp4_blocks(_ptr(w), nmat, R, C, _ptr(q), _ptr(s), _stream(stream)))
    return q, s


# ------------------------------------------------------------------ control
def set_decode_rows(rows: int):
    lib().moe_set_decode_rows(int(rows))


def get_decode_rows() -> int:
    return int(lib().moe_get_decode_rows())


def set_swap_rows(rows_per_expert: int):
    """Mean rows per expert at or below which the bf16 GEMMs use the swap-AB
    orientation (< 0: default, 0: never)."""
    lib().moe_set_swap_rows(int(rows_per_expert))


def get_swap_rows() -> int:
    return int(lib().moe_get_swap_rows())


def set_block_scaled_mma(on: bool):
    """UE8M0 FP8 experts on the tensor core's block scaling (True, default)
    or on the software-promotion kernel (False)."""
    lib().moe_set_block_scaled_mma(1 if on else 0)


def get_block_scaled_mma() -> bool:
    return bool(lib().moe_get_block_scaled_mma())


def set_down_l2_hints(bits: int):
    """L2 policies of the down GEMMs: bit 0 accumulator evict_last, bit 1
    W_down loads evict_first (< 0: the default, 1)."""
    lib().moe_set_down_l2_hints(int(bits))


def get_down_l2_hints() -> int:
    return int(lib().moe_get_down_l2_hints())


def set_pair_gemm(mask: int):
    """bf16 grouped GEMMs on CTA pairs: bit 0 gate/up, bit 1 down (< 0: the
    default, gate/up on pairs where H >= 4096)."""
    lib().moe_set_pair_gemm(int(mask))


def get_pair_gemm() -> int:
    return int(lib().moe_get_pair_gemm())


def set_down_phases(phases: int):
    """Output-column slices of the down GEMMs run one after the other (< 0:
    automatic, the default; 0 or 1: one)."""
    lib().moe_set_down_phases(int(phases))


def get_down_phases() -> int:
    return int(lib().moe_get_down_phases())


def set_tile_group(m_tiles: int):
    """m-tiles per tile group of the token-row gate/up GEMM (0: all)."""
    lib().moe_set_tile_group(int(m_tiles))


def get_tile_group() -> int:
    return int(lib().moe_get_tile_group())


def set_decode_single(on: bool):
    """Small bf16 decode batches (<= 64 routed rows) as one cooperative
    kernel (True) or as two kernels (False, default)."""
    lib().moe_set_decode_single(1 if on else 0)


def get_decode_single() -> bool:
    return bool(lib().moe_get_decode_single())


def set_fp4_gemv_rows(rows: int):
    """FP4 forwards with T*k <= rows use the CUDA-core GEMVs, larger ones the
    block-scaled tensor-core GEMMs (< 0: the default, 0 = GEMMs always; at
    most 64)."""
    lib().moe_set_fp4_gemv_rows(int(rows))


def get_fp4_gemv_rows() -> int:
    return int(lib().moe_get_fp4_gemv_rows())


def profile_begin():
    _check(lib().moe_profile_begin())


def profile_end():
    """-> {stage: (total_ms, launches)} for the forwards since profile_begin()."""
    n = len(STAGES)
    ms = (ctypes.c_float * n)()
    cnt = (ctypes.c_int * n)()
    lib().moe_profile_end(ms, cnt, n)
    return {STAGES[i]: (float(ms[i]), int(cnt[i])) for i in range(n)}


def profile_read():
    """-> {stage: (total_ms, launches)} of the forwards recorded so far, without
    ending the session (after a CUDA-graph replay: that replay's times)."""
    n = len(STAGES)
    ms = (ctypes.c_float * n)()
    cnt = (ctypes.c_int * n)()
    lib().moe_profile_read(ms, cnt, n)
    return {STAGES[i]: (float(ms[i]), int(cnt[i])) for i in range(n)}


def launch_count() -> int:
    """Kernels launched by the library so far in this process."""
    return int(lib().moe_launch_count())


def selftest_wait_timeout(limit_us: int = 2000, stream=None) -> int:
    """Run the bounded-wait self-test; returns the status that
    moe_workspace_status reports afterwards (expected MOE_ERR_TIMEOUT)."""
    ws = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    _check(lib().moe_selftest_wait_timeout(_ptr(ws), ws.numel(), int(limit_us), _stream(stream)))
    return int(lib().moe_workspace_status(_ptr(ws), _stream(stream)))
