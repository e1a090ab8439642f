// Host-side declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

#include "../../include/moe_experts.h"

namespace moe {

// Every kernel of the library is launched with programmatic stream
// serialisation allowed (programmatic dependent launch): its CTAs may be
// scheduled while the previous kernel on the stream is still finishing, and
// each kernel executes griddepcontrol.wait before its first global-memory
// access, which blocks until that previous grid has completed and its
// writes are visible.  What overlaps is launch latency and the shared-memory
// and TMEM set-up, never a data dependence.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, Args&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Error word bits written by kernels into the head of the workspace.
enum : int {
  ERR_TIMEOUT_PRODUCER = 1,
  ERR_TIMEOUT_MMA = 2,
  ERR_TIMEOUT_EPILOGUE = 4,
  ERR_TIMEOUT_SELFTEST = 8,
  ERR_BAD_INDEX = 16,
};

constexpr int kMaxE = 1024;
constexpr int kMaxK = 32;
// Routing entries per histogram/placement block: at least 256, and at most
// 128 blocks whatever T*k is (the scan walks the blocks serially).
inline long dispatch_chunk(long n) {
  const long c = (n + 127) / 128;
  return c <= 256 ? 256 : (c + 255) / 256 * 256;
}
constexpr int kSmallDispatchMax = 2048;  // T*k at or below: one-CTA dispatch
constexpr int kBM = 128;               // max token rows per grouped-GEMM tile

// Device-side word block at the head of every workspace: the error word,
// then the two counters the single-launch decode kernel synchronises its
// CTAs with (zero between launches; the last CTA of a launch resets them).
struct WsHeader {
  int err;
  int pad[63];
};
constexpr int kSyncArriveWord = 1;
constexpr int kSyncDoneWord = 2;

// Pointers into the dispatch part of a workspace.
struct DispatchBufs {
  int* err;
  int* counts;       // [E]
  int* offsets;      // [E+1]
  int* tile_pref;    // [E+1] prefix of ceil(count/128)
  int* sorted_f;     // [T*k]
  int* row_of;       // [T*k]
  int* blk_counts;   // [nchunks * E]
  int* touched;      // [E+1]: touched[0] = n, then expert ids ascending
};

// Records the message moe_last_error() returns on this host thread; returns st.
moe_status set_last_error(moe_status st, const char* fmt, ...);

// Counts every kernel launch the library makes (exported as moe_launch_count).
void count_launches(int n);

// Row stride (in scale entries) of the per-row 1x128 activation scales:
// the block count rounded up to a multiple of 4.
__host__ __device__ inline int scale_stride(int nblocks) { return (nblocks + 3) & ~3; }

inline int ceil_div(long a, long b) { return static_cast<int>((a + b - 1) / b); }

// Kernel launchers (return cudaGetLastError()).
cudaError_t launch_route(const float* logits, int T, int E, int k, int32_t* idx, float* w,
                         cudaStream_t s);
cudaError_t launch_dispatch(const int32_t* topk_idx, int T, int E, int k, const DispatchBufs& d,
                            cudaStream_t s);
// X_perm rows from the token side (row_of from the dispatch), and
// out32[0:T*H] = 0 in the same launch.
cudaError_t launch_scatter_rows_bf16(const void* hidden, int H, int T, int k, const int* row_of,
                                     void* x_perm, float* out32, cudaStream_t s);
// FP8 activations (1x128 blocks, scales row-major) from the token side,
// and out32[0:T*H] = 0 in the same launch.
cudaError_t launch_scatter_fp8(const void* hidden, int H, int T, int k, const int* row_of,
                               bool ue8m0, uint8_t* xq, void* xs, float* out32, cudaStream_t s);
cudaError_t launch_to_bf16(const float* src, void* dst, long n, cudaStream_t s);
cudaError_t launch_quantize_blocks(const void* w, int nmat, int rows, int cols, bool ue8m0,
                                   uint8_t* q, void* scale, cudaStream_t s);
cudaError_t launch_selftest_wait(int* err, int limit_us, cudaStream_t s);

// Grouped tensor-core GEMMs (bf16).  Two orientations: token rows as the
// MMA's M side (gemm_rows.cu: tm_a = activations, tm_b = weights, both
// 128-row boxes) for experts with many rows, and weight rows as M
// (gemm_swap.cu: tm_a = weights with 128-row boxes, tm_b = activations with
// 64-row boxes) for experts with few rows.  Both use tile_pref = prefix of
// ceil(M_e / 128).
struct GroupedGemmArgs {
  const CUtensorMap* tm_a;
  const CUtensorMap* tm_b;
  const int* offsets;        // [E+1]
  const int* tile_pref;      // [E+1]
  int E, K, I, H, k;
  int* err;
  // gate/up + SwiGLU epilogue
  void* h_out;               // bf16 [rows, I]
  // down + combine epilogue
  float* out32;              // [T, H]
  const int* sorted_f;
  const float* topk_w;
  int num_sms;
  int act;                   // moe_activation of the gate/up epilogue
  int tile_group = 0;        // token-row kernel: m-tiles per tile group (0: all)
  int phases = 1;            // swap-AB kernel: feature-block slices run in turn
  int l2_hints = 0;          // down GEMM: bit 0 accumulator evict_last, bit 1 weights evict_first
};
cudaError_t launch_gemm1_bf16_rows(const GroupedGemmArgs& a, cudaStream_t s);
cudaError_t launch_gemm2_bf16_rows(const GroupedGemmArgs& a, cudaStream_t s);
cudaError_t launch_gemm1_bf16_swap(const GroupedGemmArgs& a, cudaStream_t s);
cudaError_t launch_gemm2_bf16_swap(const GroupedGemmArgs& a, cudaStream_t s);
// The same GEMMs on CTA pairs (gemm_pair.cu: tcgen05.mma.cta_group::2,
// M = 256 weight rows, tokens as N <= 256; tm_a = weights, tm_b =
// activations with 64- (gate/up) or 128-row (down) weight boxes and 128-row
// token boxes; the tile prefix is built in the kernel; stages cover 128 of
// K, so K % 128 == 0, and down needs H % 256 == 0).  n_rows = routed rows
// (T*k).
cudaError_t launch_gemm1_bf16_pair(const GroupedGemmArgs& a, long n_rows, cudaStream_t s);
cudaError_t launch_gemm2_bf16_pair(const GroupedGemmArgs& a, long n_rows, cudaStream_t s);
// Default CTA-pair use (bit 0: gate/up, bit 1: down): gate/up on pairs for
// H >= kPairGateUpMinH, measured faster there (DeepSeek-V3 width) and
// slower at H = 2048 (Qwen width, whose ~140-token tiles leave the pair
// bound by L2 reads); the down GEMM on pairs from kPairDownMinRows routed
// rows per expert on average (measured faster at every prefill size and at
// 8.5 rows per expert, slower at 1.3 and 2.4, where the one-CTA swap-AB
// kernel's 16-wide token tiles fit the batch).
constexpr int kPairGateUpMinH = 4096;
constexpr int kPairDownMinRows = 8;
// Down GEMMs' L2 policies by default: the accumulator's reductions
// evict_last (measured 1-3 % faster at every prefill size; evict_first on
// the weight loads measured no faster and is off).
constexpr int kDownL2Default = 1;
inline int pair_gemm_default(int H, long n_rows, int E) {
  return (H >= kPairGateUpMinH ? 1 : 0) |
         (n_rows >= static_cast<long>(kPairDownMinRows) * E ? 2 : 0);
}
constexpr int kRowsBK = 64;  // K-block (bf16 elements) of the token-row kernel; 32 measured slower
constexpr int kSwapRowsDefault = 128;  // mean rows per expert at or below: swap-AB kernel (measured)
constexpr int kTileGroupDefault = 4;   // token-row gate/up: m-tiles per tile group (measured)
// Down GEMMs: the fp32 accumulator slice [T, H/phases] that one phase
// updates is kept at or below this many bytes (automatic phase count).
constexpr long kDownPhaseBytes = 40L << 20;   // measured: 7 slices at DeepSeek-V3 T=8192, 14 at T=16384
// Number of slices (a divisor of nblocks) that brings T*H*4/slices to at
// most kDownPhaseBytes; `forced` > 0 asks for that many (rounded up to a
// divisor).
inline int down_phases(long T, long H, int nblocks, int forced) {
  const long acc = T * H * 4;
  for (int d = 1; d <= nblocks; ++d) {
    if (nblocks % d) continue;
    if (forced > 0 ? d >= forced : acc / d <= kDownPhaseBytes) return d;
  }
  return nblocks;
}

// FP8 e4m3 block-scaled grouped GEMMs (scales applied per 128-wide K-block).
struct GroupedGemmFp8Args {
  const CUtensorMap* tm_a;   // e4m3 activations [n_rows, K], box 128 x 128 B
  const CUtensorMap* tm_b;   // e4m3 weights [E * Nw, K], box 128 x 128 B
  const int* offsets;
  const int* tile_pref;
  int E, K, I, H, k, n_rows;
  int* err;
  const void* a_scale;       // [n_rows, scale_stride(K/128)]
  const void* w_scale;       // [E, Nw/128, K/128]
  bool ue8m0;
  void* hq;                  // gate/up output codes [n_rows, I]
  void* hs;                  // gate/up output scales [n_rows, scale_stride(I/128)]
  float* out32;              // down output accumulator [T, H]
  const int* sorted_f;
  const float* topk_w;
  int num_sms;
  int act;                   // moe_activation of the gate/up epilogue
  int tile_group = 0;        // m-tiles per tile group (0: all)
  int phases = 1;            // n-tile slices run in turn
  int l2_hints = 0;          // as GroupedGemmArgs::l2_hints
};
cudaError_t launch_gemm1_fp8(const GroupedGemmFp8Args& a, cudaStream_t s);
cudaError_t launch_gemm2_fp8(const GroupedGemmFp8Args& a, cudaStream_t s);

// Block-scaled grouped GEMMs on the tensor core's UE8M0 block scaling
// (tcgen05.mma kind::mxf8f6f4, token rows as M, N = 256): FP8 experts with
// UE8M0 128x128 weight scales, and FP4 (e2m1) experts with 1x32 weight
// scales.  Activations are e4m3 with one 32-bit scale word per row and
// 128-wide K block (byte j = the exponent of 32-wide sub-block j), stored
// K-block-major: a_sf[kb * n_rows + row].
struct GroupedGemmMxArgs {
  const CUtensorMap* tm_a;   // e4m3 activations [n_rows, K], box 128 x 128 B
  const CUtensorMap* tm_b;   // weights [E * Nw, K]: e4m3 (uint8 map) or e2m1 (16U4_ALIGN16B map)
  const int* offsets;
  const int* tile_pref;
  int E, K, I, H, k, n_rows;
  int* err;
  const uint32_t* a_sf;      // [K/128][n_rows]
  const uint8_t* w_sf;       // FP8: [E, Nw/128, K/128]; FP4: [E * Nw, K/32]
  uint8_t* hq;               // gate/up output codes [n_rows, I]
  uint32_t* hs;              // gate/up output scale words [I/128][n_rows]
  float* out32;              // down output accumulator [T, H]
  const int* sorted_f;
  const float* topk_w;
  int num_sms;
  int act;
  int tile_group = 0;        // m-tiles per tile group (0: all)
  int phases = 1;            // n-tile slices run in turn
  int l2_hints = 0;          // as GroupedGemmArgs::l2_hints
};
cudaError_t launch_gemm1_mx(const GroupedGemmMxArgs& a, bool fp4, cudaStream_t s);
cudaError_t launch_gemm2_mx(const GroupedGemmMxArgs& a, bool fp4, cudaStream_t s);
// e4m3 quantisation of the routed rows in 1 x block UE8M0 blocks (block 128
// or 32), written from the token side, scale words K-block-major as above;
// out32[0:T*H] = 0 in the same launch.
cudaError_t launch_scatter_quant_mx(const void* hidden, int H, int T, int k, const int* row_of,
                                    int rows, int block, uint8_t* xq, uint32_t* xs, float* out32,
                                    cudaStream_t s);

// Small-token decode path.
struct DecodeArgs {
  const void* hidden;        // bf16 [T, H]
  const void* w_gate_up;     // bf16 [E, 2I, H]
  const void* w_down;        // bf16 [E, H, I]
  const float* topk_w;       // [T, k]
  const int* offsets;        // [E+1]
  const int* touched;        // [E+1]
  const int* sorted_f;       // [T*k]
  const int* row_of;         // [T*k]
  void* h;                   // bf16 [T*k, I]
  float* Y;                  // fp32 [T*k, H], weighted rows
  void* out;                 // bf16 [T, H]
  int T, H, I, E, k, num_sms;
  int act;                   // moe_activation of the gate/up GEMV
};
constexpr int kDecodeRowsDefault = 16;    // T*k at or below: decode path (measured crossover)
constexpr int kDecodeRowsMax = 2048;      // the decode path's workspace is sized up to this
constexpr int kFusedDecodeRows = 64;      // T*k at or below: two fused decode kernels
constexpr int kFp4GemvRowsDefault = 0;    // FP4: block-scaled GEMMs at every size (measured faster)
cudaError_t launch_dispatch_small(const int32_t* topk_idx, int T, int E, int k,
                                  const DispatchBufs& d, cudaStream_t s);
cudaError_t launch_decode_gate_up(const DecodeArgs& a, cudaStream_t s);
cudaError_t launch_decode_down(const DecodeArgs& a, cudaStream_t s);
cudaError_t launch_decode_combine(const DecodeArgs& a, cudaStream_t s);
// True when the two fused decode kernels apply (T*k <= kFusedDecodeRows).
bool decode_fused_fits(const DecodeArgs& a);
cudaError_t launch_decode_fused_gate_up(const DecodeArgs& a, const int32_t* topk_idx, int* err,
                                       cudaStream_t s);
cudaError_t launch_decode_fused_down(const DecodeArgs& a, const int32_t* topk_idx, int* err,
                                     cudaStream_t s);
// Both fused decode kernels as one cooperative launch (phase B's W_down
// stream overlaps phase A); head = the workspace's word block.  Returns an
// error without launching when the GPU cannot hold the grid at once.
cudaError_t launch_decode_single(const DecodeArgs& a, const int32_t* topk_idx, int* head,
                                 cudaStream_t s);

// FP4 (e2m1, 1x32 UE8M0 blocks) experts, small-token path only:
// T*k <= kFusedDecodeRows.  Three kernels: activation quantisation, gate/up
// with the h quantisation, down with the combine.
struct Fp4DecodeArgs {
  const void* hidden;          // bf16 [T, H]
  const void* w_gate_up;       // packed e2m1 [E, 2I, H/2]
  const void* w_down;          // packed e2m1 [E, H, I/2]
  const void* scale_gate_up;   // UE8M0 [E, 2I, H/32]
  const void* scale_down;      // UE8M0 [E, H, I/32]
  const int32_t* topk_idx;     // [T, k]
  const float* topk_w;         // [T, k]
  float* xdq;                  // fp32 [T, H], quantised activations (scratch)
  float* hq;                   // fp32 [T*k, I], quantised h (scratch)
  void* out;                   // bf16 [T, H]
  int* err;                    // device error word
  int T, H, I, E, k, num_sms;
  int act;                     // moe_activation
};
cudaError_t launch_fp4_quant_x(const Fp4DecodeArgs& a, cudaStream_t s);
cudaError_t launch_fp4_gate_up(const Fp4DecodeArgs& a, cudaStream_t s);
cudaError_t launch_fp4_down(const Fp4DecodeArgs& a, cudaStream_t s);
// bf16 [rows, cols] -> packed e2m1 [rows, cols/2] + UE8M0 bytes [rows, cols/32]
cudaError_t launch_quantize_fp4(const void* w, long rows, int cols, uint8_t* q, uint8_t* scale,
                                int num_sms, cudaStream_t s);

}  // namespace moe
