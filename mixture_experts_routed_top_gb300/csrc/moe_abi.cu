// C-ABI entry points: argument validation, workspace layout, tensor-map
// construction and the launch sequence of the routed experts forward.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "moe_internal.h"

using namespace moe;

namespace moe {
static std::atomic<long long> g_launches{0};
void count_launches(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }
}  // namespace moe

namespace {

thread_local std::string g_last_error;

moe_status fail(moe_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

}  // namespace

moe_status moe::set_last_error(moe_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

namespace {

moe_status cuda_fail(cudaError_t e, const char* what) {
  return fail(MOE_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Process-wide path thresholds (< 0: default); atomic, since any host
// thread may set them while others launch forwards.
std::atomic<int> g_decode_rows{-1};
std::atomic<int> g_swap_rows{-1};
std::atomic<int> g_block_scaled_mma{1};   // UE8M0 FP8 experts on the tensor core's block scaling
std::atomic<int> g_fp4_gemv_rows{-1};     // FP4: CUDA-core GEMVs up to this many routed rows
std::atomic<int> g_decode_single{0};      // small decode batches as one cooperative launch
std::atomic<int> g_tile_group{-1};        // token-row gate/up GEMM: m-tiles per tile group
std::atomic<int> g_down_phases{-1};       // down GEMMs: accumulator slices (< 0: automatic)
std::atomic<int> g_down_l2{kDownL2Default};  // down GEMMs: L2 policy bits (accumulator, weights)
std::atomic<int> g_pair_gemm{-1};         // bf16 grouped GEMMs on CTA pairs (bit mask, < 0: default)

// ----------------------------------------------------------- workspace map
struct WsLayout {
  size_t counts, offsets, tile_pref, touched, sorted_f, row_of, blk_counts;
  size_t xa, xa_scale, hb, hb_scale, out32, ydec;
  size_t total;
};

WsLayout ws_layout(long T, long H, long I, long E, long k, moe_wdtype wd) {
  WsLayout L{};
  const bool fp8 = wd == MOE_W_FP8_E4M3;
  const bool fp4 = wd == MOE_W_FP4_E2M1;
  const long n = T * k;
  const long nchunks = n ? (n + dispatch_chunk(n) - 1) / dispatch_chunk(n) : 0;
  size_t off = sizeof(WsHeader);
  auto take = [&](size_t bytes) {
    size_t at = align_up(off, 1024);
    off = at + bytes;
    return at;
  };
  L.counts = take(E * 4);
  L.offsets = take((E + 1) * 4);
  L.tile_pref = take((E + 1) * 4);
  L.touched = take((E + 1) * 4);
  L.sorted_f = take(n * 4);
  L.row_of = take(n * 4);
  L.blk_counts = take(nchunks * E * 4);
  // activations and h: e4m3 codes (FP8), bf16, or the quantised values in
  // fp32 (FP4, which keeps one row per token for the activations)
  // (FP4 keeps both forms: fp32 values for the small-token GEMVs, e4m3
  // codes with K-block-major scale words for the block-scaled GEMMs)
  const size_t esz = fp8 ? 1 : fp4 ? 4 : 2;
  L.xa = take(fp4 ? std::max(T * H * 4, n * H) : n * H * esz);
  L.xa_scale = take(fp8 ? n * scale_stride(H / 128) * 4 : fp4 ? n * (H / 128) * 4 : 0);
  L.hb = take(n * I * esz);
  L.hb_scale = take(fp8 ? n * scale_stride(I / 128) * 4 : fp4 ? n * (I / 128) * 4 : 0);
  L.out32 = take(T * H * 4);
  L.ydec = take(n <= kDecodeRowsMax ? n * H * 4 : 0);
  L.total = align_up(off, 1024);
  return L;
}

size_t dispatch_ws_bytes(long T, long E, long k) {
  const long n = T * k;
  const long nchunks = n ? (n + dispatch_chunk(n) - 1) / dispatch_chunk(n) : 0;
  size_t off = align_up(sizeof(WsHeader), 1024);
  off = align_up(off + (E + 1) * 4, 1024);  // tile prefix
  off = align_up(off + (E + 1) * 4, 1024);  // touched list
  off = align_up(off + nchunks * E * 4, 1024);
  return off;
}

// ----------------------------------------------------------- tensor maps
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D row-major [outer, inner] matrix, box = box_rows rows x row_bytes
// (128 or 64) bytes, swizzled at the same width, out-of-range rows read as
// zero.
moe_status make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int esize,
                    uint64_t inner, uint64_t outer, uint32_t box_rows = 128,
                    uint32_t row_bytes = 128) {
  auto fn = encode_fn();
  if (!fn) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * esize};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(row_bytes / esize), box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE,
                  row_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return MOE_OK;
}

// Gate/up weights [E, 2I, K] viewed as 3-D [2E, I, K] (plane 2e = the gate
// rows of expert e, plane 2e+1 its up rows): a box {row_bytes / esize
// elements, box_rows, 2} brings box_rows gate rows and then the matching up
// rows, swizzled at 128 bytes.  For packed e2m1 (dt 16U4_ALIGN16B) K counts
// elements and a row holds K/2 bytes.
moe_status make_map_gate_up(CUtensorMap* m, const void* base, CUtensorMapDataType dt,
                            uint64_t K, uint64_t I, uint64_t E, uint32_t box_rows,
                            uint32_t box_elems, uint64_t row_bytes) {
  auto fn = encode_fn();
  if (!fn) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[3] = {K, I, 2 * E};
  cuuint64_t strides[2] = {row_bytes, row_bytes * I};
  cuuint32_t box[3] = {box_elems, box_rows, 2};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled (gate/up view) failed (%d)", (int)r);
  return MOE_OK;
}

// bf16 operand of the CTA-pair kernel, whose stages cover 128 of K as two
// 64-wide slices: the matrix [.., K] viewed with the 64-wide K slice index as
// the outermost coordinate (stride 128 bytes), so one box of
// {64, rows, (2 planes,) 2 slices} lands as the two swizzled slices one after
// the other.  rows_dim = the row count, planes = 0 for a plain [rows, K]
// matrix or 2E for the gate/up weights' [2E, I, K] view (rows_dim = I).
moe_status make_map_k2(CUtensorMap* m, const void* base, uint64_t K, uint64_t rows_dim,
                       uint64_t planes, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  const uint64_t row_bytes = K * 2;
  cuuint64_t dims[4] = {64, rows_dim, planes ? planes : K / 64, K / 64};
  cuuint64_t strides[3] = {row_bytes, planes ? row_bytes * rows_dim : 128, 128};
  cuuint32_t box[4] = {64, box_rows, 2, 2};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  const cuuint32_t rank = planes ? 4 : 3;
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled (128-wide K stages) failed (%d)", (int)r);
  return MOE_OK;
}

// 2-D packed e2m1 matrix [rows, k_elems] (two codes per byte, row stride
// k_elems/2 bytes), box 128 elements x box_rows rows, expanded by TMA into the
// one-byte-per-element-slot shared-memory form (16 codes in 8 bytes, 8 bytes
// of padding) and swizzled at 128 bytes.
moe_status make_map_e2m1(CUtensorMap* m, const void* base, uint64_t k_elems, uint64_t rows,
                         uint32_t box_rows = 128) {
  auto fn = encode_fn();
  if (!fn) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[2] = {k_elems, rows};
  cuuint64_t strides[1] = {k_elems / 2};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 2, const_cast<void*>(base), dims,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled (packed e2m1) failed (%d)", (int)r);
  return MOE_OK;
}

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 148;
  return n;
}

// ----------------------------------------------------------- stage timing
struct Profiler {
  bool on = false;
  struct Rec {
    int stage;
    cudaEvent_t a, b;
  };
  std::vector<Rec> recs;
  std::vector<cudaEvent_t> pool;
  cudaEvent_t get() {
    if (!pool.empty()) {
      cudaEvent_t e = pool.back();
      pool.pop_back();
      return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
  }
};
Profiler g_prof;
std::mutex g_prof_mu;

// Records a CUDA event pair around one stage of a forward.  Inside a stream
// capture the events are recorded as external event nodes, so that after a
// replay of the graph they hold that replay's times.
struct StageScope {
  cudaStream_t s;
  int stage;
  cudaEvent_t b = nullptr;
  unsigned flags = cudaEventRecordDefault;
  StageScope(cudaStream_t s_, int st) : s(s_), stage(st) {
    if (!g_prof.on) return;
    std::lock_guard<std::mutex> g(g_prof_mu);
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusActive)
      flags = cudaEventRecordExternal;
    cudaEvent_t a = g_prof.get();
    b = g_prof.get();
    cudaEventRecordWithFlags(a, s, flags);
    g_prof.recs.push_back({stage, a, b});
  }
  ~StageScope() {
    if (b) cudaEventRecordWithFlags(b, s, flags);
  }
};

}  // namespace

// =========================================================== exported API
extern "C" {

int moe_version(void) { return 100; }

long long moe_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

const char* moe_last_error(void) { return g_last_error.c_str(); }

void moe_set_decode_rows(int rows) {
  g_decode_rows = rows < 0 ? -1 : (rows > kDecodeRowsMax ? kDecodeRowsMax : rows);
}
int moe_get_decode_rows(void) {
  const int r = g_decode_rows.load(std::memory_order_relaxed);
  return r < 0 ? kDecodeRowsDefault : r;
}

void moe_set_swap_rows(int rows_per_expert) { g_swap_rows = rows_per_expert < 0 ? -1 : rows_per_expert; }
int moe_get_swap_rows(void) {
  const int r = g_swap_rows.load(std::memory_order_relaxed);
  return r < 0 ? kSwapRowsDefault : r;
}

void moe_set_down_l2_hints(int bits) { g_down_l2 = bits < 0 ? kDownL2Default : (bits & 3); }
int moe_get_down_l2_hints(void) { return g_down_l2.load(std::memory_order_relaxed); }

void moe_set_pair_gemm(int mask) { g_pair_gemm = mask < 0 ? -1 : (mask & 3); }
int moe_get_pair_gemm(void) { return g_pair_gemm.load(std::memory_order_relaxed); }

void moe_set_down_phases(int phases) { g_down_phases = phases < 0 ? -1 : phases; }
int moe_get_down_phases(void) { return g_down_phases.load(std::memory_order_relaxed); }

void moe_set_tile_group(int m_tiles) { g_tile_group = m_tiles < 0 ? -1 : m_tiles; }
int moe_get_tile_group(void) {
  const int g = g_tile_group.load(std::memory_order_relaxed);
  return g < 0 ? kTileGroupDefault : g;
}

void moe_set_decode_single(int on) { g_decode_single = on ? 1 : 0; }
int moe_get_decode_single(void) { return g_decode_single.load(std::memory_order_relaxed); }

void moe_set_block_scaled_mma(int on) { g_block_scaled_mma = on ? 1 : 0; }
int moe_get_block_scaled_mma(void) { return g_block_scaled_mma.load(std::memory_order_relaxed); }

void moe_set_fp4_gemv_rows(int rows) {
  g_fp4_gemv_rows = rows < 0 ? -1 : (rows > kFusedDecodeRows ? kFusedDecodeRows : rows);
}
int moe_get_fp4_gemv_rows(void) {
  const int r = g_fp4_gemv_rows.load(std::memory_order_relaxed);
  return r < 0 ? kFp4GemvRowsDefault : r;
}

moe_status moe_route(const float* logits, int T, int E, int k, int32_t* topk_idx, float* topk_w,
                     void* stream) {
  if (T < 0) return fail(MOE_ERR_INVALID_ARG, "moe_route: T < 0");
  if (E < 1 || E > kMaxE) return fail(MOE_ERR_UNSUPPORTED, "moe_route: E must be in [1, %d]", kMaxE);
  if (k < 1 || k > E || k > kMaxK)
    return fail(MOE_ERR_UNSUPPORTED, "moe_route: k must be in [1, min(E, %d)]", kMaxK);
  if (T == 0) return MOE_OK;
  if (!logits || !topk_idx || !topk_w) return fail(MOE_ERR_INVALID_ARG, "moe_route: null pointer");
  if (!aligned(logits, 4) || !aligned(topk_idx, 4) || !aligned(topk_w, 4))
    return fail(MOE_ERR_INVALID_ARG, "moe_route: misaligned pointer");
  cudaError_t e = launch_route(logits, T, E, k, topk_idx, topk_w, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "moe_route launch");
  return MOE_OK;
}

size_t moe_dispatch_workspace_size(int T, int E, int k) {
  if (T < 0 || E < 1 || k < 1) return 0;
  return dispatch_ws_bytes(T, E, k);
}

moe_status moe_dispatch(const int32_t* topk_idx, int T, int E, int k, int32_t* counts,
                        int32_t* offsets, int32_t* sorted_f, int32_t* row_of, void* ws,
                        size_t ws_bytes, void* stream) {
  if (T < 0) return fail(MOE_ERR_INVALID_ARG, "moe_dispatch: T < 0");
  if (E < 1 || E > kMaxE) return fail(MOE_ERR_UNSUPPORTED, "moe_dispatch: E must be in [1, %d]", kMaxE);
  if (k < 1 || k > E || k > kMaxK)
    return fail(MOE_ERR_UNSUPPORTED, "moe_dispatch: k must be in [1, min(E, %d)]", kMaxK);
  if (static_cast<long>(T) * k > 0x7FFFFFFFL)
    return fail(MOE_ERR_UNSUPPORTED, "moe_dispatch: T*k exceeds int32");
  if (!counts || !offsets || !ws || (T > 0 && (!topk_idx || !sorted_f || !row_of)))
    return fail(MOE_ERR_INVALID_ARG, "moe_dispatch: null pointer");
  if (!aligned(ws, 256)) return fail(MOE_ERR_INVALID_ARG, "moe_dispatch: ws must be 256-byte aligned");
  const size_t need = dispatch_ws_bytes(T, E, k);
  if (ws_bytes < need)
    return fail(MOE_ERR_WORKSPACE, "moe_dispatch: workspace %zu < %zu bytes", ws_bytes, need);
  uint8_t* w = static_cast<uint8_t*>(ws);
  const long n = static_cast<long>(T) * k;
  DispatchBufs d;
  size_t off = align_up(sizeof(WsHeader), 1024);
  d.err = reinterpret_cast<int*>(w);
  d.counts = counts;
  d.offsets = offsets;
  d.tile_pref = reinterpret_cast<int*>(w + off);
  off = align_up(off + (E + 1) * 4, 1024);
  d.touched = reinterpret_cast<int*>(w + off);
  off = align_up(off + (E + 1) * 4, 1024);
  d.blk_counts = reinterpret_cast<int*>(w + off);
  d.sorted_f = sorted_f;
  d.row_of = row_of;
  (void)n;
  cudaError_t e = launch_dispatch(topk_idx, T, E, k, d, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "moe_dispatch launch");
  return MOE_OK;
}

size_t moe_workspace_size(int T, int H, int I, int E, int k, moe_wdtype wdtype) {
  if (T < 0 || H < 1 || I < 1 || E < 1 || k < 1) return 0;
  return ws_layout(T, H, I, E, k, wdtype).total;
}

size_t moe_workspace_accumulator_offset(int T, int H, int I, int E, int k, moe_wdtype wdtype) {
  if (T < 0 || H < 1 || I < 1 || E < 1 || k < 1) return 0;
  return ws_layout(T, H, I, E, k, wdtype).out32;
}

moe_status moe_experts_forward(const void* hidden, int T, int H, const int32_t* topk_idx,
                               const float* topk_w, int E, int k, int I, const void* w_gate_up,
                               const void* w_down, moe_wdtype wdtype, const void* scale_gate_up,
                               const void* scale_down, moe_scale_fmt sfmt, void* out, void* ws,
                               size_t ws_bytes, void* stream) {
  return moe_experts_forward_act(hidden, T, H, topk_idx, topk_w, E, k, I, w_gate_up, w_down,
                                 wdtype, scale_gate_up, scale_down, sfmt, MOE_ACT_SILU, out, ws,
                                 ws_bytes, stream);
}

moe_status moe_experts_forward_act(const void* hidden, int T, int H, const int32_t* topk_idx,
                                   const float* topk_w, int E, int k, int I,
                                   const void* w_gate_up, const void* w_down, moe_wdtype wdtype,
                                   const void* scale_gate_up, const void* scale_down,
                                   moe_scale_fmt sfmt, moe_activation act, void* out, void* ws,
                                   size_t ws_bytes, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (act != MOE_ACT_SILU && act != MOE_ACT_GELU && act != MOE_ACT_RELU)
    return fail(MOE_ERR_INVALID_ARG, "moe_experts_forward: unknown activation %d",
                static_cast<int>(act));
  if (T < 0 || H < 1 || I < 1) return fail(MOE_ERR_INVALID_ARG, "moe_experts_forward: bad sizes");
  if (E < 1 || E > kMaxE)
    return fail(MOE_ERR_UNSUPPORTED, "moe_experts_forward: E must be in [1, %d]", kMaxE);
  if (k < 1 || k > E || k > kMaxK)
    return fail(MOE_ERR_UNSUPPORTED, "moe_experts_forward: k must be in [1, min(E, %d)]", kMaxK);
  if (H % 128 || I % 128)
    return fail(MOE_ERR_UNSUPPORTED, "moe_experts_forward: H and I must be multiples of 128");
  if (static_cast<long>(T) * k > 0x7FFFFFFFL)
    return fail(MOE_ERR_UNSUPPORTED, "moe_experts_forward: T*k exceeds int32");
  const bool fp8 = wdtype == MOE_W_FP8_E4M3;
  const bool fp4 = wdtype == MOE_W_FP4_E2M1;
  if (wdtype != MOE_W_BF16 && !fp8 && !fp4)
    return fail(MOE_ERR_INVALID_ARG, "moe_experts_forward: unknown weight dtype %d", (int)wdtype);
  if (fp8) {
    if (sfmt != MOE_SCALE_F32 && sfmt != MOE_SCALE_UE8M0)
      return fail(MOE_ERR_INVALID_ARG,
                  "moe_experts_forward: FP8 weights need float32 or UE8M0 block scales");
    if (!scale_gate_up || !scale_down)
      return fail(MOE_ERR_INVALID_ARG, "moe_experts_forward: FP8 weights need scale buffers");
  } else if (fp4) {
    if (sfmt != MOE_SCALE_UE8M0)
      return fail(MOE_ERR_INVALID_ARG, "moe_experts_forward: FP4 weights need UE8M0 block scales");
    if (!scale_gate_up || !scale_down)
      return fail(MOE_ERR_INVALID_ARG, "moe_experts_forward: FP4 weights need scale buffers");
    if (static_cast<long>(T) * k > moe_get_fp4_gemv_rows() &&
        !(H % 256 && static_cast<long>(T) * k <= kFusedDecodeRows)) {
      if (H % 256)
        return fail(MOE_ERR_UNSUPPORTED,
                    "moe_experts_forward: FP4 weights above %d routed rows need H %% 256 == 0",
                    kFusedDecodeRows);
      if (!aligned(w_gate_up, 32) || !aligned(w_down, 32))
        return fail(MOE_ERR_INVALID_ARG,
                    "moe_experts_forward: FP4 weights must be 32-byte aligned (packed TMA loads)");
    }
  } else if (sfmt != MOE_SCALE_NONE || scale_gate_up || scale_down) {
    return fail(MOE_ERR_INVALID_ARG, "moe_experts_forward: bf16 weights take no scales");
  }
  if (T == 0) return MOE_OK;
  if (!hidden || !topk_idx || !topk_w || !w_gate_up || !w_down || !out || !ws)
    return fail(MOE_ERR_INVALID_ARG, "moe_experts_forward: null pointer");
  const void* ptrs[] = {hidden, topk_idx, topk_w, w_gate_up, w_down, out};
  for (const void* q : ptrs)
    if (!aligned(q, 16)) return fail(MOE_ERR_INVALID_ARG, "moe_experts_forward: buffers must be 16-byte aligned");
  if (!aligned(ws, 256))
    return fail(MOE_ERR_INVALID_ARG, "moe_experts_forward: ws must be 256-byte aligned");
  const WsLayout L = ws_layout(T, H, I, E, k, wdtype);
  if (ws_bytes < L.total)
    return fail(MOE_ERR_WORKSPACE, "moe_experts_forward: workspace %zu < %zu bytes", ws_bytes,
                L.total);
  if (fp8 && H % 256)
    return fail(MOE_ERR_UNSUPPORTED, "moe_experts_forward: FP8 weights need H % 256 == 0");
  if (fp8 && (!aligned(scale_gate_up, 4) || !aligned(scale_down, 4)))
    return fail(MOE_ERR_INVALID_ARG, "moe_experts_forward: scale buffers must be 4-byte aligned");

  uint8_t* w = static_cast<uint8_t*>(ws);
  const long n = static_cast<long>(T) * k;
  DispatchBufs d;
  d.err = reinterpret_cast<int*>(w);
  d.counts = reinterpret_cast<int*>(w + L.counts);
  d.offsets = reinterpret_cast<int*>(w + L.offsets);
  d.tile_pref = reinterpret_cast<int*>(w + L.tile_pref);
  d.touched = reinterpret_cast<int*>(w + L.touched);
  d.sorted_f = reinterpret_cast<int*>(w + L.sorted_f);
  d.row_of = reinterpret_cast<int*>(w + L.row_of);
  d.blk_counts = reinterpret_cast<int*>(w + L.blk_counts);
  void* xa = w + L.xa;
  void* hb = w + L.hb;
  float* out32 = reinterpret_cast<float*>(w + L.out32);

  const int sms = num_sms();
  cudaError_t e;
  // FP4: the block-scaled GEMMs above the GEMV threshold, except where their
  // 256-wide down tiles do not divide H and the GEMVs can take the batch
  const bool fp4_gemm = fp4 && n > moe_get_fp4_gemv_rows() && !(H % 256 && n <= kFusedDecodeRows);
  const bool mx = (fp8 && sfmt == MOE_SCALE_UE8M0 && moe_get_block_scaled_mma()) || fp4_gemm;
  if (mx) {
    // FP8 (UE8M0) or FP4 experts on the tensor core's block scaling:
    // dispatch, e4m3 quantisation of the rows in 1x128 (FP8) or 1x32 (FP4)
    // blocks written in expert order (accumulator zeroed in the same launch),
    // the two block-scaled grouped GEMMs, bf16 output
    uint8_t* xq = w + L.xa;
    uint32_t* xs = reinterpret_cast<uint32_t*>(w + L.xa_scale);
    uint8_t* hq = w + L.hb;
    uint32_t* hs = reinterpret_cast<uint32_t*>(w + L.hb_scale);
    CUtensorMap tm_x, tm_wgu, tm_h, tm_wd;
    moe_status st;
    if ((st = make_map(&tm_x, xq, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, H, n)) != MOE_OK) return st;
    if ((st = make_map(&tm_h, hq, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, I, n)) != MOE_OK) return st;
    // gate/up weights: the [2E, I, H] view, one box = 128 gate rows and
    // their up rows; down weights: 256-row boxes
    if (fp4) {
      if ((st = make_map_gate_up(&tm_wgu, w_gate_up, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, H, I,
                                 E, 128, 128, static_cast<uint64_t>(H) / 2)) != MOE_OK)
        return st;
      if ((st = make_map_e2m1(&tm_wd, w_down, I, static_cast<uint64_t>(E) * H, 256)) != MOE_OK)
        return st;
    } else {
      if ((st = make_map_gate_up(&tm_wgu, w_gate_up, CU_TENSOR_MAP_DATA_TYPE_UINT8, H, I, E, 128,
                                 128, H)) != MOE_OK)
        return st;
      if ((st = make_map(&tm_wd, w_down, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, I,
                         static_cast<uint64_t>(E) * H, 256)) != MOE_OK)
        return st;
    }
    {
      StageScope sc(s, MOE_STAGE_DISPATCH);
      e = n <= kSmallDispatchMax ? launch_dispatch_small(topk_idx, T, E, k, d, s)
                                 : launch_dispatch(topk_idx, T, E, k, d, s);
      if (e != cudaSuccess) return cuda_fail(e, "dispatch");
      if ((e = launch_scatter_quant_mx(hidden, H, T, k, d.row_of, static_cast<int>(n),
                                       fp4 ? 32 : 128, xq, xs, out32, s)) != cudaSuccess)
        return cuda_fail(e, "scatter_quant_mx");
    }
    GroupedGemmMxArgs g{};
    g.offsets = d.offsets;
    g.tile_pref = d.tile_pref;
    g.E = E;
    g.I = I;
    g.H = H;
    g.k = k;
    g.n_rows = static_cast<int>(n);
    g.err = d.err;
    g.hq = hq;
    g.hs = hs;
    g.out32 = out32;
    g.sorted_f = d.sorted_f;
    g.topk_w = topk_w;
    g.act = static_cast<int>(act);
    const long mtiles_max = n / kBM + E;
    g.tile_group = moe_get_tile_group();
    {
      StageScope sc(s, MOE_STAGE_GEMM1);
      g.tm_a = &tm_x;
      g.tm_b = &tm_wgu;
      g.K = H;
      g.a_sf = xs;
      g.w_sf = static_cast<const uint8_t*>(scale_gate_up);
      g.num_sms = static_cast<int>(std::min<long>(sms, mtiles_max * (I / 128)));
      if ((e = launch_gemm1_mx(g, fp4, s)) != cudaSuccess) return cuda_fail(e, "gemm1_mx");
    }
    {
      StageScope sc(s, MOE_STAGE_GEMM2);
      g.tm_a = &tm_h;
      g.tm_b = &tm_wd;
      g.K = I;
      g.a_sf = hs;
      g.w_sf = static_cast<const uint8_t*>(scale_down);
      g.num_sms = static_cast<int>(std::min<long>(sms, mtiles_max * (H / 256)));
      g.tile_group = 0;
      g.phases = down_phases(T, H, H / 256, g_down_phases.load(std::memory_order_relaxed));
      g.l2_hints = moe_get_down_l2_hints();
      if ((e = launch_gemm2_mx(g, fp4, s)) != cudaSuccess) return cuda_fail(e, "gemm2_mx");
    }
    {
      StageScope sc(s, MOE_STAGE_FINISH);
      if ((e = launch_to_bf16(out32, out, static_cast<long>(T) * H, s)) != cudaSuccess)
        return cuda_fail(e, "to_bf16");
    }
    return MOE_OK;
  }
  if (fp4) {
    // packed e2m1 weights, small-token path: the routing table is rebuilt
    // in the gate/up and down kernels, and the down kernel combines
    Fp4DecodeArgs a;
    a.hidden = hidden;
    a.w_gate_up = w_gate_up;
    a.w_down = w_down;
    a.scale_gate_up = scale_gate_up;
    a.scale_down = scale_down;
    a.topk_idx = topk_idx;
    a.topk_w = topk_w;
    a.xdq = reinterpret_cast<float*>(w + L.xa);
    a.hq = reinterpret_cast<float*>(w + L.hb);
    a.out = out;
    a.err = d.err;
    a.T = T;
    a.H = H;
    a.I = I;
    a.E = E;
    a.k = k;
    a.num_sms = sms;
    a.act = static_cast<int>(act);
    {
      StageScope sc(s, MOE_STAGE_DISPATCH);
      if ((e = launch_fp4_quant_x(a, s)) != cudaSuccess) return cuda_fail(e, "fp4_quant_x");
    }
    {
      StageScope sc(s, MOE_STAGE_GEMM1);
      if ((e = launch_fp4_gate_up(a, s)) != cudaSuccess) return cuda_fail(e, "fp4_gate_up");
    }
    {
      StageScope sc(s, MOE_STAGE_GEMM2);
      if ((e = launch_fp4_down(a, s)) != cudaSuccess) return cuda_fail(e, "fp4_down");
    }
    return MOE_OK;
  }
  if (!fp8 && n <= moe_get_decode_rows()) {
    // small-token path: stream the touched experts' weights once
    DecodeArgs a;
    a.hidden = hidden;
    a.w_gate_up = w_gate_up;
    a.w_down = w_down;
    a.topk_w = topk_w;
    a.offsets = d.offsets;
    a.touched = d.touched;
    a.sorted_f = d.sorted_f;
    a.row_of = d.row_of;
    a.h = hb;
    a.Y = reinterpret_cast<float*>(w + L.ydec);
    a.out = out;
    a.T = T;
    a.H = H;
    a.I = I;
    a.E = E;
    a.k = k;
    a.num_sms = sms;
    a.act = static_cast<int>(act);
    if (decode_fused_fits(a) && g_decode_single.load(std::memory_order_relaxed)) {
      // one cooperative kernel: gate/up, then down + combine, the down
      // weights streaming while the last h values are computed
      StageScope sc(s, MOE_STAGE_GEMM1);
      e = launch_decode_single(a, topk_idx, d.err, s);
      if (e == cudaSuccess) return MOE_OK;
      (void)cudaGetLastError();   // not launched (grid too large for this GPU): two kernels
    }
    if (decode_fused_fits(a)) {
      // routing table rebuilt inside both kernels; the down kernel combines
      {
        StageScope sc(s, MOE_STAGE_GEMM1);
        if ((e = launch_decode_fused_gate_up(a, topk_idx, d.err, s)) != cudaSuccess)
          return cuda_fail(e, "decode_fused_gate_up");
      }
      {
        StageScope sc(s, MOE_STAGE_GEMM2);
        if ((e = launch_decode_fused_down(a, topk_idx, d.err, s)) != cudaSuccess)
          return cuda_fail(e, "decode_fused_down");
      }
      return MOE_OK;
    }
    {
      StageScope sc(s, MOE_STAGE_DISPATCH);
      if ((e = launch_dispatch_small(topk_idx, T, E, k, d, s)) != cudaSuccess)
        return cuda_fail(e, "dispatch_small");
    }
    {
      StageScope sc(s, MOE_STAGE_GEMM1);
      if ((e = launch_decode_gate_up(a, s)) != cudaSuccess) return cuda_fail(e, "decode_gate_up");
    }
    {
      StageScope sc(s, MOE_STAGE_GEMM2);
      if ((e = launch_decode_down(a, s)) != cudaSuccess) return cuda_fail(e, "decode_down");
    }
    {
      StageScope sc(s, MOE_STAGE_FINISH);
      if ((e = launch_decode_combine(a, s)) != cudaSuccess) return cuda_fail(e, "decode_combine");
    }
    return MOE_OK;
  }

  if (fp8) {
    const bool ue = sfmt == MOE_SCALE_UE8M0;
    uint8_t* xq = w + L.xa;
    void* xs = w + L.xa_scale;
    uint8_t* hq = w + L.hb;
    void* hs = w + L.hb_scale;
    float* out32 = reinterpret_cast<float*>(w + L.out32);
    CUtensorMap tm_x, tm_wgu, tm_h, tm_wd;
    moe_status st;
    if ((st = make_map(&tm_x, xq, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, H, n)) != MOE_OK) return st;
    if ((st = make_map_gate_up(&tm_wgu, w_gate_up, CU_TENSOR_MAP_DATA_TYPE_UINT8, H, I, E, 128,
                               128, H)) != MOE_OK)
      return st;
    if ((st = make_map(&tm_h, hq, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, I, n)) != MOE_OK) return st;
    if ((st = make_map(&tm_wd, w_down, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, I,
                       static_cast<uint64_t>(E) * H, 256)) != MOE_OK)
      return st;
    {
      StageScope sc(s, MOE_STAGE_DISPATCH);
      e = n <= kSmallDispatchMax ? launch_dispatch_small(topk_idx, T, E, k, d, s)
                                 : launch_dispatch(topk_idx, T, E, k, d, s);
      if (e != cudaSuccess) return cuda_fail(e, "dispatch");
      if ((e = launch_scatter_fp8(hidden, H, T, k, d.row_of, ue, xq, xs, out32, s)) != cudaSuccess)
        return cuda_fail(e, "scatter_fp8");
    }
    GroupedGemmFp8Args g{};
    g.offsets = d.offsets;
    g.act = static_cast<int>(act);
    g.tile_pref = d.tile_pref;
    g.E = E;
    g.I = I;
    g.H = H;
    g.k = k;
    g.n_rows = static_cast<int>(n);
    g.err = d.err;
    g.ue8m0 = ue;
    g.hq = hq;
    g.hs = hs;
    g.out32 = out32;
    g.sorted_f = d.sorted_f;
    g.topk_w = topk_w;
    const long mtiles_max = n / kBM + E;
    {
      StageScope sc(s, MOE_STAGE_GEMM1);
      g.tm_a = &tm_x;
      g.tm_b = &tm_wgu;
      g.K = H;
      g.a_scale = xs;
      g.w_scale = scale_gate_up;
      g.num_sms = static_cast<int>(std::min<long>(sms, mtiles_max * (I / 128)));
      g.tile_group = moe_get_tile_group();
      if ((e = launch_gemm1_fp8(g, s)) != cudaSuccess) return cuda_fail(e, "gemm1_fp8");
    }
    {
      StageScope sc(s, MOE_STAGE_GEMM2);
      g.tm_a = &tm_h;
      g.tm_b = &tm_wd;
      g.K = I;
      g.a_scale = hs;
      g.w_scale = scale_down;
      g.num_sms = static_cast<int>(std::min<long>(sms, mtiles_max * (H / 256)));
      g.tile_group = 0;
      g.phases = down_phases(T, H, H / 256, g_down_phases.load(std::memory_order_relaxed));
      g.l2_hints = moe_get_down_l2_hints();
      if ((e = launch_gemm2_fp8(g, s)) != cudaSuccess) return cuda_fail(e, "gemm2_fp8");
    }
    {
      StageScope sc(s, MOE_STAGE_FINISH);
      if ((e = launch_to_bf16(out32, out, static_cast<long>(T) * H, s)) != cudaSuccess)
        return cuda_fail(e, "to_bf16");
    }
    return MOE_OK;
  }

  // Orientation of each grouped GEMM.  Gate/up: weight rows as the MMA's M
  // side (swap-AB) when experts get few rows, token rows as M otherwise.
  // Down: swap-AB (measured faster at every size) unless a threshold was set
  // explicitly, which then applies to both (0: token rows always).
  const int swap_rows = moe_get_swap_rows();
  const bool swap1 = n <= static_cast<long>(swap_rows) * E;
  const bool swap2 = g_swap_rows.load(std::memory_order_relaxed) >= 0 ? swap1 : true;
  // CTA-pair kernels (either GEMM, by the process-wide mask)
  const int pair_set = moe_get_pair_gemm();
  const int pair = pair_set < 0 ? pair_gemm_default(H, n, E) : pair_set;
  // the pair kernel takes 128 of K per stage (K = H for gate/up, I for
  // down; the forward already requires both to be multiples of 128) and
  // its down tiles are 256 output columns wide
  const bool pair1 = (pair & 1) && H % 128 == 0;
  const bool pair2 = (pair & 2) && H % 256 == 0 && I % 128 == 0;
  // swap-AB kernel: 128-byte rows, token boxes of 64 rows; token-row
  // kernel: rows of kRowsBK bf16, 128-row boxes for both operands; pair
  // kernel: 128-byte rows, 128-row token boxes, weight boxes of 64 rows
  // (gate/up) or 128 (down)
  const uint32_t rb = kRowsBK * 2;
  // gate/up weights: the [2E, I, H] view, one box = box rows of gate and the
  // matching up rows; down weights: 128-row boxes (swap-AB: 128 per M=128
  // MMA of the tile, so 256 where H % 256 == 0)
  const uint32_t xr1 = swap1 && !pair1 ? 64 : 128, wr1 = pair1 ? 64 : 128;
  const uint32_t xb1 = (pair1 || swap1) ? 128 : rb;
  const uint32_t xr2 = swap2 && !pair2 ? 64 : 128;
  const uint32_t wr2 = swap2 && !pair2 && H % 256 == 0 ? 256 : 128;
  const uint32_t xb2 = (pair2 || swap2) ? 128 : rb;
  CUtensorMap tm_x, tm_wgu, tm_h, tm_wd;
  moe_status st;
  if (pair1) {  // 128-wide K stages
    if ((st = make_map_k2(&tm_x, xa, H, n, 0, 128)) != MOE_OK) return st;
    if ((st = make_map_k2(&tm_wgu, w_gate_up, H, I, static_cast<uint64_t>(E) * 2, 64)) != MOE_OK)
      return st;
  } else {
    if ((st = make_map(&tm_x, xa, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, H, n, xr1, xb1)) != MOE_OK)
      return st;
    if ((st = make_map_gate_up(&tm_wgu, w_gate_up, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, H, I, E, wr1,
                               xb1 / 2, static_cast<uint64_t>(H) * 2)) != MOE_OK)
      return st;
  }
  if (pair2) {  // 128-wide K stages
    if ((st = make_map_k2(&tm_h, hb, I, n, 0, 128)) != MOE_OK) return st;
    if ((st = make_map_k2(&tm_wd, w_down, I, static_cast<uint64_t>(E) * H, 0, 128)) != MOE_OK)
      return st;
  } else {
    if ((st = make_map(&tm_h, hb, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, I, n, xr2, xb2)) != MOE_OK)
      return st;
    if ((st = make_map(&tm_wd, w_down, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, I,
                       static_cast<uint64_t>(E) * H, wr2, xb2)) != MOE_OK)
      return st;
  }

  {
    StageScope sc(s, MOE_STAGE_DISPATCH);
    e = n <= kSmallDispatchMax ? launch_dispatch_small(topk_idx, T, E, k, d, s)
                               : launch_dispatch(topk_idx, T, E, k, d, s);
    if (e != cudaSuccess) return cuda_fail(e, "dispatch");
    // expert-sorted rows written from the token side (hidden read once), the
    // fp32 accumulator zeroed in the same launch: at DeepSeek-V3 size 0.237
    // against 0.317 ms for a row-side gather plus a zeroing kernel
    if ((e = launch_scatter_rows_bf16(hidden, H, T, k, d.row_of, xa, out32, s)) != cudaSuccess)
      return cuda_fail(e, "scatter");
  }
  GroupedGemmArgs g{};
  g.offsets = d.offsets;
  g.act = static_cast<int>(act);
  g.tile_pref = d.tile_pref;
  g.E = E;
  g.I = I;
  g.H = H;
  g.k = k;
  g.err = d.err;
  g.h_out = hb;
  g.out32 = out32;
  g.sorted_f = d.sorted_f;
  g.topk_w = topk_w;
  // upper bound on tiles: sum_e ceil(M_e/128) <= n/128 + E
  const long mtiles_max = n / kBM + E;
  {
    StageScope sc(s, MOE_STAGE_GEMM1);
    g.tm_a = (swap1 || pair1) ? &tm_wgu : &tm_x;
    g.tm_b = (swap1 || pair1) ? &tm_x : &tm_wgu;
    g.K = H;
    g.num_sms = static_cast<int>(std::min<long>(sms, mtiles_max * (I / 128)));
    g.tile_group = moe_get_tile_group();
    e = pair1 ? launch_gemm1_bf16_pair(g, n, s)
              : swap1 ? launch_gemm1_bf16_swap(g, s) : launch_gemm1_bf16_rows(g, s);
    if (e != cudaSuccess) return cuda_fail(e, "gemm1");
  }
  {
    StageScope sc(s, MOE_STAGE_GEMM2);
    g.tm_a = (swap2 || pair2) ? &tm_wd : &tm_h;
    g.tm_b = (swap2 || pair2) ? &tm_h : &tm_wd;
    g.K = I;
    const int nf = (pair2 || H % 256 == 0) ? 256 : 128;
    g.num_sms = static_cast<int>(std::min<long>(sms, mtiles_max * (H / nf)));
    g.phases = down_phases(T, H, H / nf, g_down_phases.load(std::memory_order_relaxed));
    g.l2_hints = moe_get_down_l2_hints();
    e = pair2 ? launch_gemm2_bf16_pair(g, n, s)
              : swap2 ? launch_gemm2_bf16_swap(g, s) : launch_gemm2_bf16_rows(g, s);
    if (e != cudaSuccess) return cuda_fail(e, "gemm2");
  }
  {
    StageScope sc(s, MOE_STAGE_FINISH);
    if ((e = launch_to_bf16(out32, out, static_cast<long>(T) * H, s)) != cudaSuccess)
      return cuda_fail(e, "to_bf16");
  }
  return MOE_OK;
}

moe_status moe_quantize_fp8_blocks(const void* wsrc, int nmat, int rows, int cols,
                                   moe_scale_fmt sfmt, uint8_t* q, void* scale, void* stream) {
  if (nmat < 0 || rows < 0 || cols < 0)
    return fail(MOE_ERR_INVALID_ARG, "moe_quantize_fp8_blocks: negative size");
  if (rows % 128 || cols % 128)
    return fail(MOE_ERR_UNSUPPORTED, "moe_quantize_fp8_blocks: rows and cols must be multiples of 128");
  if (sfmt != MOE_SCALE_F32 && sfmt != MOE_SCALE_UE8M0)
    return fail(MOE_ERR_INVALID_ARG, "moe_quantize_fp8_blocks: scale format must be F32 or UE8M0");
  if (static_cast<long>(nmat) * rows * cols == 0) return MOE_OK;
  if (!wsrc || !q || !scale) return fail(MOE_ERR_INVALID_ARG, "moe_quantize_fp8_blocks: null pointer");
  if (!aligned(wsrc, 16) || !aligned(q, 16) || !aligned(scale, 4))
    return fail(MOE_ERR_INVALID_ARG, "moe_quantize_fp8_blocks: misaligned pointer");
  cudaError_t e = launch_quantize_blocks(wsrc, nmat, rows, cols, sfmt == MOE_SCALE_UE8M0, q, scale,
                                         static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "moe_quantize_fp8_blocks launch");
  return MOE_OK;
}

moe_status moe_quantize_fp4_blocks(const void* wsrc, int nmat, int rows, int cols, uint8_t* q,
                                   uint8_t* scale, void* stream) {
  if (nmat < 0 || rows < 0 || cols < 0)
    return fail(MOE_ERR_INVALID_ARG, "moe_quantize_fp4_blocks: negative size");
  if (cols % 32) return fail(MOE_ERR_UNSUPPORTED, "moe_quantize_fp4_blocks: cols must be a multiple of 32");
  if (static_cast<long>(nmat) * rows * cols == 0) return MOE_OK;
  if (!wsrc || !q || !scale) return fail(MOE_ERR_INVALID_ARG, "moe_quantize_fp4_blocks: null pointer");
  if (!aligned(wsrc, 16) || !aligned(q, 16))
    return fail(MOE_ERR_INVALID_ARG, "moe_quantize_fp4_blocks: misaligned pointer");
  cudaError_t e = launch_quantize_fp4(wsrc, static_cast<long>(nmat) * rows, cols, q, scale, num_sms(),
                                      static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "moe_quantize_fp4_blocks launch");
  return MOE_OK;
}

moe_status moe_workspace_status(void* ws, void* stream) {
  if (!ws) return fail(MOE_ERR_INVALID_ARG, "moe_workspace_status: null workspace");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int err = 0;
  cudaError_t e = cudaMemcpyAsync(&err, ws, sizeof(int), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return cuda_fail(e, "moe_workspace_status");
  if (err) {
    // the error word and the decode counters (which a timed-out launch may
    // have left non-zero) start again from zero
    const int zero[3] = {0, 0, 0};
    e = cudaMemcpyAsync(ws, zero, sizeof(zero), cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "moe_workspace_status clear");
    if (err & (ERR_TIMEOUT_PRODUCER | ERR_TIMEOUT_MMA | ERR_TIMEOUT_EPILOGUE | ERR_TIMEOUT_SELFTEST))
      return fail(MOE_ERR_TIMEOUT, "device wait timed out (error word 0x%x)", err);
    return fail(MOE_ERR_INVALID_ARG, "kernel met an out-of-range expert index (error word 0x%x)", err);
  }
  return MOE_OK;
}

moe_status moe_profile_begin(void) {
  std::lock_guard<std::mutex> g(g_prof_mu);
  for (auto& r : g_prof.recs) {
    g_prof.pool.push_back(r.a);
    g_prof.pool.push_back(r.b);
  }
  g_prof.recs.clear();
  g_prof.on = true;
  return MOE_OK;
}

// Sums the elapsed time of every recorded pair per stage (caller holds the lock).
static void profile_collect(float* stage_ms, int* stage_launches, int n) {
  std::vector<float> ms(MOE_STAGE_COUNT, 0.f);
  std::vector<int> cnt(MOE_STAGE_COUNT, 0);
  for (auto& r : g_prof.recs) {
    cudaEventSynchronize(r.b);
    float t = 0.f;
    if (cudaEventElapsedTime(&t, r.a, r.b) == cudaSuccess) {
      ms[r.stage] += t;
      cnt[r.stage] += 1;
    }
  }
  (void)cudaGetLastError();  // a pair that could not be timed leaves no pending error behind
  for (int i = 0; i < n && i < MOE_STAGE_COUNT; ++i) {
    if (stage_ms) stage_ms[i] = ms[i];
    if (stage_launches) stage_launches[i] = cnt[i];
  }
}

int moe_profile_end(float* stage_ms, int* stage_launches, int n) {
  std::lock_guard<std::mutex> g(g_prof_mu);
  g_prof.on = false;
  profile_collect(stage_ms, stage_launches, n);
  for (auto& r : g_prof.recs) {
    g_prof.pool.push_back(r.a);
    g_prof.pool.push_back(r.b);
  }
  g_prof.recs.clear();
  return MOE_STAGE_COUNT;
}

int moe_profile_read(float* stage_ms, int* stage_launches, int n) {
  std::lock_guard<std::mutex> g(g_prof_mu);
  profile_collect(stage_ms, stage_launches, n);
  return MOE_STAGE_COUNT;
}

moe_status moe_selftest_wait_timeout(void* ws, size_t ws_bytes, int limit_us, void* stream) {
  if (!ws || ws_bytes < sizeof(WsHeader) || !aligned(ws, 256))
    return fail(MOE_ERR_INVALID_ARG, "moe_selftest_wait_timeout: bad workspace");
  if (limit_us < 1 || limit_us > 1000000)
    return fail(MOE_ERR_INVALID_ARG, "moe_selftest_wait_timeout: limit_us must be in [1, 1e6]");
  cudaError_t e = launch_selftest_wait(static_cast<int*>(ws), limit_us, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "moe_selftest_wait_timeout launch");
  return MOE_OK;
}

}  // extern "C"
