// Router, dispatch, the expert-sorted row copies (bf16, or e4m3 with their
// block scales; each also zeroes the fp32 accumulator), output conversion
// and FP8 weight quantisation kernels (everything except the grouped
// tensor-core GEMMs and the decode GEMVs).
#include <cuda_fp8.h>
#include <float.h>
#include <limits.h>
#include <math.h>

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {

// ============================================================== router
// One warp per token.  Lane l holds logits l, l+32, ... in registers; k
// rounds of a warp-wide arg-max pick the experts in slot order (descending
// logit, ties to the lower expert index), then the kept logits go through a
// softmax relative to the largest one.  Selection uses only comparisons of
// the fp32 logits, so the chosen indices are exact.
template <int NPL>
__global__ void __launch_bounds__(256) route_kernel(const float* __restrict__ logits, int T, int E,
                                                    int k, int32_t* __restrict__ topk_idx,
                                                    float* __restrict__ topk_w) {
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const long t = (static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  if (t >= T) return;
  const float* row = logits + t * E;
  float v[NPL];
  uint32_t used = 0;
#pragma unroll
  for (int i = 0; i < NPL; ++i) {
    const int e = lane + 32 * i;
    v[i] = (e < E) ? __ldg(row + e) : -INFINITY;
    if (e >= E) used |= 1u << i;
  }
  float my_v = 0.f;
  int my_e = 0;
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int be = INT_MAX;  // INT_MAX = no candidate
#pragma unroll
    for (int i = 0; i < NPL; ++i) {
      if (!((used >> i) & 1u) && (be == INT_MAX || v[i] > bv)) {
        bv = v[i];
        be = lane + 32 * i;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oe = __shfl_xor_sync(0xffffffffu, be, off);
      const bool take = (oe != INT_MAX) &&
                        (be == INT_MAX || ov > bv || (ov == bv && oe < be));
      if (take) {
        bv = ov;
        be = oe;
      }
    }
    if ((be & 31) == lane) used |= 1u << (be >> 5);
    if (lane == j) {
      my_v = bv;
      my_e = be;
    }
  }
  const float top = __shfl_sync(0xffffffffu, my_v, 0);
  const bool dead = isinf(top) && top < 0.f;
  float ex = (lane < k && !dead) ? expf(my_v - top) : 0.f;
  float sum = ex;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  if (lane < k) {
    topk_idx[t * k + lane] = my_e;
    topk_w[t * k + lane] = dead ? 1.0f / static_cast<float>(k) : ex / sum;
  }
}

cudaError_t launch_route(const float* logits, int T, int E, int k, int32_t* idx, float* w,
                         cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int npl = ceil_div(E, 32);
  dim3 block(256), grid(ceil_div(static_cast<long>(T) * 32, 256));
  if (npl <= 1) launch_pdl(route_kernel<1>, grid, block, 0, s, logits, T, E, k, idx, w);
  else if (npl <= 2) launch_pdl(route_kernel<2>, grid, block, 0, s, logits, T, E, k, idx, w);
  else if (npl <= 4) launch_pdl(route_kernel<4>, grid, block, 0, s, logits, T, E, k, idx, w);
  else if (npl <= 8) launch_pdl(route_kernel<8>, grid, block, 0, s, logits, T, E, k, idx, w);
  else if (npl <= 16) launch_pdl(route_kernel<16>, grid, block, 0, s, logits, T, E, k, idx, w);
  else launch_pdl(route_kernel<32>, grid, block, 0, s, logits, T, E, k, idx, w);
  count_launches(1);
  return cudaGetLastError();
}

// ============================================================== dispatch
// (1) per-chunk expert histograms, (2) one-block scan that turns them into
// per-chunk write bases plus counts/offsets/tile prefix/touched list,
// (3) per-chunk stable placement, one warp walking its chunk in order.
// Out-of-range expert ids are skipped everywhere and flagged in the error
// word, so no later kernel ever indexes with them.

__global__ void __launch_bounds__(256) dispatch_count_kernel(const int32_t* __restrict__ idx,
                                                             long n, long chunk, int E,
                                                             int* blk_counts, int* err) {
  pdl_launch_dependents();
  pdl_wait();
  __shared__ int hist[kMaxE];
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const long base = static_cast<long>(blockIdx.x) * chunk;
  const long end = min(base + chunk, n);
  bool bad = false;
  for (long f = base + threadIdx.x; f < end; f += blockDim.x) {
    const int e = __ldg(idx + f);
    if (e >= 0 && e < E) atomicAdd(&hist[e], 1);
    else bad = true;
  }
  if (bad) atomicOr(err, ERR_BAD_INDEX);
  __syncthreads();
  // expert-major: the scan reads each expert's chunk counts contiguously
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    blk_counts[static_cast<long>(e) * gridDim.x + blockIdx.x] = hist[e];
}

// Per-chunk counts -> per-chunk write bases.  Counts are stored expert-major
// (blk_counts[e * nchunks + chunk]).  Warp w handles experts w, w+32, ...:
// its lanes read that expert's chunk counts 32 contiguous chunks at a time
// and a warp scan carries the running base.
// Then one block-wide scan over experts gives counts, offsets, the m-tile
// prefix and the touched list, and the bases are shifted by the offsets.
__global__ void __launch_bounds__(1024) dispatch_scan_kernel(int E, int nchunks, int* blk_counts,
                                                             int* counts, int* offsets,
                                                             int* tile_pref, int* touched) {
  pdl_launch_dependents();
  pdl_wait();
  __shared__ int s_warp[33];
  __shared__ int s_tot[kMaxE];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // nchunks <= 128: four counts per lane per expert; a batch of 8 experts'
  // counts is loaded before any of them is scanned and written back
  constexpr int kQ = 4, kBatch = 8;
  for (int e0 = warp; e0 < E; e0 += 32 * kBatch) {
    int v[kBatch][kQ];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int e = e0 + 32 * j;
#pragma unroll
      for (int q = 0; q < kQ; ++q) {
        const int b = 32 * q + lane;
        v[j][q] = (e < E && b < nchunks) ? blk_counts[static_cast<long>(e) * nchunks + b] : 0;
      }
    }
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int e = e0 + 32 * j;
      if (e >= E) break;
      int carry = 0;
#pragma unroll
      for (int q = 0; q < kQ; ++q) {
        const int b = 32 * q + lane;
        int x = v[j][q];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, x, off);
          if (lane >= off) x += y;
        }
        if (b < nchunks)   // exclusive within the expert
          blk_counts[static_cast<long>(e) * nchunks + b] = carry + x - v[j][q];
        carry += __shfl_sync(0xffffffffu, x, 31);
      }
      if (lane == 0) s_tot[e] = carry;
    }
  }
  __syncthreads();
  const int e = threadIdx.x;
  const int c = e < E ? s_tot[e] : 0;
  const int tiles = (c + kBM - 1) / kBM;
  const int tch = c > 0 ? 1 : 0;
  int tot_c, tot_t, tot_h;
  const int ex_c = block_exclusive_scan(c, s_warp, &tot_c);
  const int ex_t = block_exclusive_scan(tiles, s_warp, &tot_t);
  const int ex_h = block_exclusive_scan(tch, s_warp, &tot_h);
  if (e < E) {
    counts[e] = c;
    offsets[e] = ex_c;
    tile_pref[e] = ex_t;
    if (tch) touched[1 + ex_h] = e;
    s_tot[e] = ex_c;
  }
  if (e == 0) {
    offsets[E] = tot_c;
    tile_pref[E] = tot_t;
    touched[0] = tot_h;
  }
  __syncthreads();
  // shift the per-chunk bases by the expert offsets
  const long total = static_cast<long>(nchunks) * E;
  for (long i = threadIdx.x; i < total; i += 1024) blk_counts[i] += s_tot[i / nchunks];
}

__global__ void __launch_bounds__(32) dispatch_place_kernel(const int32_t* __restrict__ idx, long n,
                                                            long chunk, int E, const int* blk_base,
                                                            int* sorted_f, int* row_of) {
  pdl_launch_dependents();
  pdl_wait();
  __shared__ int cursor[kMaxE];
  const int lane = threadIdx.x;
  for (int e = lane; e < E; e += 32) cursor[e] = blk_base[static_cast<long>(e) * gridDim.x + blockIdx.x];
  __syncwarp();
  const long base = static_cast<long>(blockIdx.x) * chunk;
  const long end = min(base + chunk, n);
  const uint32_t lt = (1u << lane) - 1u;
  for (long f0 = base; f0 < end; f0 += 32) {
    const long f = f0 + lane;
    int e = (f < end) ? __ldg(idx + f) : -1;
    if (e >= E) e = -1;
    const uint32_t peers = __match_any_sync(0xffffffffu, e);
    int pos = -1;
    if (e >= 0) {
      pos = cursor[e] + __popc(peers & lt);
      sorted_f[pos] = static_cast<int>(f);
    }
    if (f < end) row_of[f] = pos;
    __syncwarp();
    if (e >= 0 && (peers & lt) == 0) cursor[e] += __popc(peers);
    __syncwarp();
  }
}

cudaError_t launch_dispatch(const int32_t* topk_idx, int T, int E, int k, const DispatchBufs& d,
                            cudaStream_t s) {
  const long n = static_cast<long>(T) * k;
  const long chunk = dispatch_chunk(n);
  const int nchunks = n ? ceil_div(n, chunk) : 0;
  if (nchunks) {
    launch_pdl(dispatch_count_kernel, nchunks, 256, 0, s, topk_idx, n, chunk, E, d.blk_counts, d.err);
  }
  launch_pdl(dispatch_scan_kernel, 1, 1024, 0, s, E, nchunks, d.blk_counts, d.counts, d.offsets,
                                          d.tile_pref, d.touched);
  if (nchunks) {
    launch_pdl(dispatch_place_kernel, nchunks, 32, 0, s, topk_idx, n, chunk, E, d.blk_counts,
                                                 d.sorted_f, d.row_of);
  }
  count_launches(nchunks ? 3 : 1);
  return cudaGetLastError();
}

// ============================================================== expert-sorted rows
// X_perm written from the token side.  A warp owns one (token t, column
// chunk of 32 B 16-byte vectors): it loads that piece of hidden[t] once and
// stores it to the rows the dispatch placed t's k slots at (row_of[t*k + j];
// -1 for a dropped slot), so hidden is read once rather than once per slot.
// The same warp zeroes the matching columns of the token's fp32 accumulator
// row out32[t, :], which the down GEMM's combine adds into.
template <int B>
__global__ void __launch_bounds__(128, B >= 8 ? 9 : 16)
    scatter_rows_bf16_kernel(const uint4* __restrict__ hidden, int H8, int T, int k, int nchunks,
                             const int* __restrict__ row_of, uint4* __restrict__ xperm,
                             float4* __restrict__ out32) {
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const long w = static_cast<long>(blockIdx.x) * 4 + (threadIdx.x >> 5);
  if (w >= static_cast<long>(T) * nchunks) return;   // warp-uniform
  const long t = w / nchunks;
  const int c0 = static_cast<int>(w - t * nchunks) * (32 * B);
  const int my_row = lane < k ? __ldg(row_of + t * k + lane) : -1;
  const uint4* src = hidden + t * H8;
  uint4 v[B];
#pragma unroll
  for (int i = 0; i < B; ++i) {
    const int c = c0 + 32 * i + lane;
    v[i] = c < H8 ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
  }
  for (int j = 0; j < k; ++j) {
    const int r = __shfl_sync(0xffffffffu, my_row, j);  // every lane reaches it
    if (r < 0) continue;
    uint4* dst = xperm + static_cast<long>(r) * H8;
#pragma unroll
    for (int i = 0; i < B; ++i) {
      const int c = c0 + 32 * i + lane;
      if (c < H8) __stcs(dst + c, v[i]);   // streaming: the rows are read back once
    }
  }
  // fp32 columns [8 c0, 8 (c0 + 32 B)) = float4 [2 c0, 2 (c0 + 32 B))
  float4* z = out32 + t * (2L * H8);
  const int zend = min(2 * (c0 + 32 * B), 2 * H8);
  for (int c = 2 * c0 + lane; c < zend; c += 32) z[c] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// Chunk width: the widest (8, 4, 2 or 1 vectors per lane) that still gives
// at least kScatterWarps warps, so small batches spread over many SMs; with
// at most 4 vectors a lane the kernel fits 16 blocks (64 warps) per SM; the
// 8-vector form gets 9 (capped at 12 it spilled).
// Measured at Qwen prefill size (T = 4096, H = 2048): 16384 warps (1 KB
// chunks) 30.1-30.3 us for the dispatch stage, 8192 warps 31.1 us, 4096
// warps 33.2-33.6 us; decode sizes the same either way.
constexpr long kScatterWarps = 16384;

cudaError_t launch_scatter_rows_bf16(const void* hidden, int H, int T, int k, const int* row_of,
                                     void* x_perm, float* out32, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int H8 = H / 8;
  int b = 8;
  while (b > 1 && static_cast<long>(T) * ceil_div(H8, 32 * b) < kScatterWarps) b >>= 1;
  const int nchunks = ceil_div(H8, 32 * b);
  const int grid = ceil_div(static_cast<long>(T) * nchunks, 4);
  const uint4* src = static_cast<const uint4*>(hidden);
  uint4* dst = static_cast<uint4*>(x_perm);
  float4* z = reinterpret_cast<float4*>(out32);
  switch (b) {
    case 8: launch_pdl(scatter_rows_bf16_kernel<8>, grid, 128, 0, s, src, H8, T, k, nchunks, row_of, dst, z); break;
    case 4: launch_pdl(scatter_rows_bf16_kernel<4>, grid, 128, 0, s, src, H8, T, k, nchunks, row_of, dst, z); break;
    case 2: launch_pdl(scatter_rows_bf16_kernel<2>, grid, 128, 0, s, src, H8, T, k, nchunks, row_of, dst, z); break;
    default: launch_pdl(scatter_rows_bf16_kernel<1>, grid, 128, 0, s, src, H8, T, k, nchunks, row_of, dst, z); break;
  }
  count_launches(1);
  return cudaGetLastError();
}

// ============================================================== FP8 helpers
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
  return v;
}

// Dynamic 1x128 activation quantisation written from the token side: a warp
// owns one token and 8 of its 128-wide blocks (a half-warp per block, 16
// lanes x 8 elements, four blocks per half-warp), quantises them once and
// stores codes and scales to the rows the dispatch placed the token's k
// slots at (row_of[t*k + j], -1 for a dropped slot).  Codes go to xq[r, :],
// scales to xs[r, b] with a row stride of scale_stride(H/128) blocks (a
// multiple of 4, so that one vector load fetches four blocks' scales).  The
// same warp zeroes the matching columns of the token's fp32 accumulator row.
__global__ void __launch_bounds__(128) scatter_fp8_kernel(const uint4* __restrict__ hidden, int H,
                                                          int T, int k, int nchunks,
                                                          const int* __restrict__ row_of,
                                                          bool ue8m0, uint2* __restrict__ xq,
                                                          void* __restrict__ xs,
                                                          float4* __restrict__ out32) {
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int half = lane >> 4, l16 = lane & 15;
  const long w = static_cast<long>(blockIdx.x) * 4 + (threadIdx.x >> 5);
  if (w >= static_cast<long>(T) * nchunks) return;   // warp-uniform
  const long t = w / nchunks;
  const int b0 = static_cast<int>(w - t * nchunks) * 8;
  const int nb = H / 128;
  const long sstride = scale_stride(nb);
  const int my_row = lane < k ? __ldg(row_of + t * k + lane) : -1;
  const uint4* src = hidden + t * (H / 8);
  uint4 raw[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int b = b0 + 2 * i + half;
    raw[i] = b < nb ? __ldg(src + b * 16 + l16) : make_uint4(0, 0, 0, 0);
  }
  uint2 code[4];
  uint32_t stored[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float x[8];
    const uint32_t wd[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      x[2 * j] = __uint_as_float(wd[j] << 16);
      x[2 * j + 1] = __uint_as_float(wd[j] & 0xFFFF0000u);
    }
    float amax = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(x[j]));
#pragma unroll
    for (int off = 8; off > 0; off >>= 1)  // stays inside the half-warp
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    const float sc = block_scale(amax, ue8m0, &stored[i]);
    const float inv = 1.0f / sc;
    code[i] = make_uint2(e4m3x2(x[0] * inv, x[1] * inv) | (e4m3x2(x[2] * inv, x[3] * inv) << 16),
                         e4m3x2(x[4] * inv, x[5] * inv) | (e4m3x2(x[6] * inv, x[7] * inv) << 16));
  }
  for (int j = 0; j < k; ++j) {
    const int r = __shfl_sync(0xffffffffu, my_row, j);  // every lane reaches it
    if (r < 0) continue;
    uint2* dst = xq + static_cast<long>(r) * (H / 8);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int b = b0 + 2 * i + half;
      if (b < nb) {
        dst[b * 16 + l16] = code[i];
        if (l16 == 0) {
          const long si = r * sstride + b;
          if (ue8m0) static_cast<uint8_t*>(xs)[si] = static_cast<uint8_t>(stored[i]);
          else static_cast<uint32_t*>(xs)[si] = stored[i];
        }
      }
    }
  }
  // fp32 columns of blocks [b0, b0 + 8): float4 [32 b0, 32 min(b0 + 8, nb))
  float4* z = out32 + t * (H / 4);
  const int zend = 32 * min(b0 + 8, nb);
  for (int c = 32 * b0 + lane; c < zend; c += 32) z[c] = make_float4(0.f, 0.f, 0.f, 0.f);
}

cudaError_t launch_scatter_fp8(const void* hidden, int H, int T, int k, const int* row_of,
                               bool ue8m0, uint8_t* xq, void* xs, float* out32, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int nchunks = ceil_div(H / 128, 8);
  launch_pdl(scatter_fp8_kernel, ceil_div(static_cast<long>(T) * nchunks, 4), 128, 0, s,
             static_cast<const uint4*>(hidden), H, T, k, nchunks, row_of, ue8m0,
             reinterpret_cast<uint2*>(xq), xs, reinterpret_cast<float4*>(out32));
  count_launches(1);
  return cudaGetLastError();
}

// Dynamic e4m3 quantisation of the routed rows with UE8M0 scales in 1 x BLK
// blocks (BLK = 128 for FP8 experts, 32 for FP4 experts), written from the
// token side: a warp owns one token and 8 of its 128-wide K blocks (a
// half-warp per block, 16 lanes x 8 elements, four blocks per half-warp),
// quantises them once and stores the codes and scale words to the rows the
// dispatch placed the token's k slots at (row_of[t*k + j], -1 for a dropped
// slot).  Codes go to xq[r, :], scale words (four sub-block bytes per
// 128-wide block, each byte the scale of its 32-wide sub-block) to
// xs[kb * rows + r].  The same warp zeroes the matching columns of the
// token's fp32 accumulator row.
template <int BLK>
__global__ void __launch_bounds__(128) scatter_quant_mx_kernel(const uint4* __restrict__ hidden,
                                                               int H, int T, int k, int nchunks,
                                                               const int* __restrict__ row_of,
                                                               int rows, uint2* __restrict__ xq,
                                                               uint32_t* __restrict__ xs,
                                                               float4* __restrict__ out32) {
  pdl_launch_dependents();
  pdl_wait();
  const int lane = threadIdx.x & 31;
  const int half = lane >> 4, l16 = lane & 15;
  const long w = static_cast<long>(blockIdx.x) * 4 + (threadIdx.x >> 5);
  if (w >= static_cast<long>(T) * nchunks) return;   // warp-uniform
  const long t = w / nchunks;
  const int b0 = static_cast<int>(w - t * nchunks) * 8;
  const int nb = H / 128;
  const int my_row = lane < k ? __ldg(row_of + t * k + lane) : -1;
  const uint4* src = hidden + t * (H / 8);
  uint4 raw[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int b = b0 + 2 * i + half;
    raw[i] = b < nb ? __ldg(src + b * 16 + l16) : make_uint4(0, 0, 0, 0);
  }
  uint2 code[4];
  uint32_t word[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float x[8];
    const uint32_t wd[4] = {raw[i].x, raw[i].y, raw[i].z, raw[i].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      x[2 * j] = __uint_as_float(wd[j] << 16);
      x[2 * j + 1] = __uint_as_float(wd[j] & 0xFFFF0000u);
    }
    float amax = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(x[j]));
    // lanes of one block: 16 (BLK = 128) or 4 (BLK = 32), inside the half-warp
#pragma unroll
    for (int off = BLK / 16; off > 0; off >>= 1)
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    uint32_t sb;
    const float sc = block_scale(amax, true, &sb);
    const float inv = 1.0f / sc;
    // scale word of the 128-wide block: byte j = sub-block j's exponent
    if (BLK == 128) {
      word[i] = sb * 0x01010101u;
    } else {
      const uint32_t s1 = __shfl_down_sync(0xffffffffu, sb, 4);
      const uint32_t s2 = __shfl_down_sync(0xffffffffu, sb, 8);
      const uint32_t s3 = __shfl_down_sync(0xffffffffu, sb, 12);
      word[i] = sb | (s1 << 8) | (s2 << 16) | (s3 << 24);
    }
    code[i] = make_uint2(e4m3x2(x[0] * inv, x[1] * inv) | (e4m3x2(x[2] * inv, x[3] * inv) << 16),
                         e4m3x2(x[4] * inv, x[5] * inv) | (e4m3x2(x[6] * inv, x[7] * inv) << 16));
  }
  for (int j = 0; j < k; ++j) {
    const int r = __shfl_sync(0xffffffffu, my_row, j);  // every lane reaches it
    if (r < 0) continue;
    uint2* dst = xq + static_cast<long>(r) * (H / 8);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int b = b0 + 2 * i + half;
      if (b < nb) {
        dst[b * 16 + l16] = code[i];
        if (l16 == 0) xs[static_cast<long>(b) * rows + r] = word[i];
      }
    }
  }
  // fp32 columns of blocks [b0, b0 + 8): float4 [32 b0, 32 min(b0 + 8, nb))
  float4* z = out32 + t * (H / 4);
  const int zend = 32 * min(b0 + 8, nb);
  for (int c = 32 * b0 + lane; c < zend; c += 32) z[c] = make_float4(0.f, 0.f, 0.f, 0.f);
}

cudaError_t launch_scatter_quant_mx(const void* hidden, int H, int T, int k, const int* row_of,
                                    int rows, int block, uint8_t* xq, uint32_t* xs, float* out32,
                                    cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int nchunks = ceil_div(H / 128, 8);
  const int grid = ceil_div(static_cast<long>(T) * nchunks, 4);
  auto kern = block == 32 ? scatter_quant_mx_kernel<32> : scatter_quant_mx_kernel<128>;
  launch_pdl(kern, grid, 128, 0, s, static_cast<const uint4*>(hidden), H, T, k, nchunks, row_of,
             rows, reinterpret_cast<uint2*>(xq), xs, reinterpret_cast<float4*>(out32));
  count_launches(1);
  return cudaGetLastError();
}

// ============================================================== finish
// out[8 i .. 8 i + 7] = bf16(src[8 i .. 8 i + 7]): per thread and step two
// 16-byte loads in flight and one 16-byte store.
__global__ void __launch_bounds__(256) to_bf16_kernel(const float4* __restrict__ src,
                                                      uint4* __restrict__ dst, long n8) {
  pdl_launch_dependents();
  pdl_wait();
  for (long i = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
       i += static_cast<long>(gridDim.x) * blockDim.x) {
    const float4 a = __ldg(src + 2 * i);
    const float4 b = __ldg(src + 2 * i + 1);
    dst[i] = make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w), pack_bf16x2(b.x, b.y),
                        pack_bf16x2(b.z, b.w));
  }
}

cudaError_t launch_to_bf16(const float* src, void* dst, long n, cudaStream_t s) {
  if (n % 8 != 0) return cudaErrorInvalidValue;  // n = T * H, H a multiple of 128
  const long n8 = n / 8;
  if (n8 == 0) return cudaSuccess;
  const long want = (n8 + 255) / 256;
  const int grid = static_cast<int>(want < 152L * 16 ? want : 152L * 16);
  launch_pdl(to_bf16_kernel, grid, 256, 0, s, reinterpret_cast<const float4*>(src),
             reinterpret_cast<uint4*>(dst), n8);
  count_launches(1);
  return cudaGetLastError();
}

// ============================================================== weight quantiser
// One 256-thread block per 128x128 block: amax, scale, codes.  Thread t
// covers row t/2, columns (t%2)*64 .. +63.
__global__ void __launch_bounds__(256) quantize_blocks_kernel(const uint4* __restrict__ w, int rows,
                                                              int cols, bool ue8m0,
                                                              uint2* __restrict__ q,
                                                              void* __restrict__ scale) {
  pdl_launch_dependents();
  pdl_wait();
  __shared__ float s_max[8];
  const int nbc = cols / 128, nbr = rows / 128;
  const long blk = blockIdx.x;  // over nmat * nbr * nbc
  const long mat = blk / (static_cast<long>(nbr) * nbc);
  const int rb = static_cast<int>((blk / nbc) % nbr), cb = static_cast<int>(blk % nbc);
  const int row = rb * 128 + (threadIdx.x >> 1);
  const int col0 = cb * 128 + (threadIdx.x & 1) * 64;
  const long base = (mat * rows + row) * static_cast<long>(cols) + col0;  // element index
  uint4 v[8];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    v[i] = __ldg(w + base / 8 + i);
    const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&v[i]);
#pragma unroll
    for (int j = 0; j < 4; ++j)
      amax = fmaxf(amax, fmaxf(fabsf(__low2float(p[j])), fabsf(__high2float(p[j]))));
  }
  amax = warp_max(amax);
  if ((threadIdx.x & 31) == 0) s_max[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = s_max[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) amax = fmaxf(amax, s_max[i]);
  uint32_t stored;
  const float sc = block_scale(amax, ue8m0, &stored);
  const float inv = 1.0f / sc;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&v[i]);
    uint32_t c[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) c[j] = e4m3x2(__low2float(p[j]) * inv, __high2float(p[j]) * inv);
    q[base / 8 + i] = make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
  }
  if (threadIdx.x == 0) {
    if (ue8m0) static_cast<uint8_t*>(scale)[blk] = static_cast<uint8_t>(stored);
    else static_cast<uint32_t*>(scale)[blk] = stored;
  }
}

cudaError_t launch_quantize_blocks(const void* w, int nmat, int rows, int cols, bool ue8m0,
                                   uint8_t* q, void* scale, cudaStream_t s) {
  const long nblk = static_cast<long>(nmat) * (rows / 128) * (cols / 128);
  if (nblk == 0) return cudaSuccess;
  launch_pdl(quantize_blocks_kernel, static_cast<unsigned>(nblk), 256, 0, s, 
      static_cast<const uint4*>(w), rows, cols, ue8m0, reinterpret_cast<uint2*>(q), scale);
  count_launches(1);
  return cudaGetLastError();
}

// ============================================================== self-test
// Waits on an mbarrier that nothing completes; the bounded wait must give up
// after limit_us, set the error word and return.
__global__ void selftest_wait_kernel(int* err, uint64_t limit_ns) {
  pdl_launch_dependents();
  pdl_wait();
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort;
  if (threadIdx.x != 0) return;
  abort = 0;
  mbar_init(smem_u32(&bar), 1);
  fence_mbar_init();
  mbar_wait_bounded(smem_u32(&bar), 0, &abort, err, ERR_TIMEOUT_SELFTEST, limit_ns);
}

cudaError_t launch_selftest_wait(int* err, int limit_us, cudaStream_t s) {
  launch_pdl(selftest_wait_kernel, 1, 32, 0, s, err, static_cast<uint64_t>(limit_us) * 1000ull);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace moe
