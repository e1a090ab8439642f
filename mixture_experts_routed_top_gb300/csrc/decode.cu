// Small-token decode path: with few routed rows per expert the forward is a
// stream over the touched experts' weights, so it runs on CUDA cores as
// GEMVs that read every touched weight row exactly once (the page's
// "Decode-stage switching" idea: a separate strategy for low token counts).
// Up to kFusedDecodeRows routed rows the path is two kernels (fused at the
// end of this file); above that it is the four below.
//
//   dispatch_small   one CTA: counts, scan, touched list, stable placement
//   decode_gate_up   item = (touched expert, 4 features); warp = feature f:
//                    gate and up rows of W_gate_up[e] streamed once, dotted
//                    with the expert's token rows, h = act(g) * u (bf16)
//   decode_down      item = (touched expert, 4 output columns); warp = one
//                    row of W_down[e]; Y[r, c] = topk_w * (h[r] . W_down[e,c])
//   decode_combine   out[t] = sum_j Y[row_of[t*k+j]] in fp32 -> bf16
// Work items are spread over a persistent grid (grid-stride), so every SM
// streams weights whatever the number of touched experts.
#include "decode_common.cuh"

namespace moe {

// ------------------------------------------------------------ dispatch
__global__ void __launch_bounds__(1024) dispatch_small_kernel(
    const int32_t* __restrict__ idx, int n, int E, int* counts, int* offsets, int* tile_pref,
    int* touched, int* sorted_f, int* row_of, int* err) {
  pdl_launch_dependents();
  pdl_wait();
  __shared__ int s_cnt[kMaxE];
  __shared__ int s_cur[kMaxE];
  __shared__ int s_warp[33];
  const int tid = threadIdx.x;
  if (tid < E) s_cnt[tid] = 0;
  __syncthreads();
  bool bad = false;
  for (int f = tid; f < n; f += 1024) {
    const int e = __ldg(idx + f);
    if (e >= 0 && e < E) atomicAdd(&s_cnt[e], 1);
    else bad = true;
  }
  if (bad) atomicOr(err, ERR_BAD_INDEX);
  __syncthreads();
  const int c = tid < E ? s_cnt[tid] : 0;
  const int tiles = (c + kBM - 1) / kBM;
  const int tch = c > 0 ? 1 : 0;
  int tot_c, tot_t, tot_h;
  const int ex_c = block_exclusive_scan(c, s_warp, &tot_c);
  const int ex_t = block_exclusive_scan(tiles, s_warp, &tot_t);
  const int ex_h = block_exclusive_scan(tch, s_warp, &tot_h);
  if (tid < E) {
    counts[tid] = c;
    offsets[tid] = ex_c;
    tile_pref[tid] = ex_t;
    if (tch) touched[1 + ex_h] = tid;
    s_cur[tid] = ex_c;
  }
  if (tid == 0) {
    offsets[E] = tot_c;
    tile_pref[E] = tot_t;
    touched[0] = tot_h;
  }
  __syncthreads();
  if (tid < 32) {
    const int lane = tid;
    const uint32_t lt = (1u << lane) - 1u;
    for (int f0 = 0; f0 < n; f0 += 32) {
      const int f = f0 + lane;
      int e = (f < n) ? __ldg(idx + f) : -1;
      if (e >= E) e = -1;
      const uint32_t peers = __match_any_sync(0xffffffffu, e);
      int pos = -1;
      if (e >= 0) {
        pos = s_cur[e] + __popc(peers & lt);
        sorted_f[pos] = f;
      }
      if (f < n) row_of[f] = pos;
      __syncwarp();
      if (e >= 0 && (peers & lt) == 0) s_cur[e] += __popc(peers);
      __syncwarp();
    }
  }
}

// ------------------------------------------------------------ helpers
__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

constexpr int kStreamBatch = 8;  // 16-byte weight vectors per lane loaded before any math

// ag[t] += w_gate . x_t and au[t] += w_up . x_t over 16-byte vectors
// lane, lane+32, ... < n8 of two weight rows; each lane first issues up to
// kStreamBatch loads per row (the tail of a short row included, guarded),
// then does the arithmetic.
template <int MT>
__device__ __forceinline__ void stream_dot2(const uint4* __restrict__ wg,
                                            const uint4* __restrict__ wu,
                                            const uint4* const (&xr)[MT], int n8, int lane,
                                            float (&ag)[MT], float (&au)[MT]) {
  for (int c0 = lane; c0 < n8; c0 += 32 * kStreamBatch) {
    uint4 g[kStreamBatch], u[kStreamBatch];
#pragma unroll
    for (int i = 0; i < kStreamBatch; ++i) {
      const int c = c0 + 32 * i;
      g[i] = c < n8 ? ld_stream(wg + c) : make_uint4(0, 0, 0, 0);
      u[i] = c < n8 ? ld_stream(wu + c) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int i = 0; i < kStreamBatch; ++i) {
      const int c = c0 + 32 * i;
      if (c >= n8) break;
      float gf[8], uf[8];
      bf16x8_to_f32(g[i], gf);
      bf16x8_to_f32(u[i], uf);
#pragma unroll
      for (int t = 0; t < MT; ++t) {
        float xf[8];
        bf16x8_to_f32(__ldg(xr[t] + c), xf);
        ag[t] = dot8(gf, xf, ag[t]);
        au[t] = dot8(uf, xf, au[t]);
      }
    }
  }
}

// acc[t] += w . x_t over one weight row, batched the same way.
template <int MT>
__device__ __forceinline__ void stream_dot1(const uint4* __restrict__ w,
                                            const uint4* const (&xr)[MT], int n8, int lane,
                                            float (&acc)[MT]) {
  for (int c0 = lane; c0 < n8; c0 += 32 * kStreamBatch) {
    uint4 v[kStreamBatch];
#pragma unroll
    for (int i = 0; i < kStreamBatch; ++i) {
      const int c = c0 + 32 * i;
      v[i] = c < n8 ? ld_stream(w + c) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int i = 0; i < kStreamBatch; ++i) {
      const int c = c0 + 32 * i;
      if (c >= n8) break;
      float wf[8];
      bf16x8_to_f32(v[i], wf);
#pragma unroll
      for (int t = 0; t < MT; ++t) {
        float xf[8];
        bf16x8_to_f32(__ldg(xr[t] + c), xf);
        acc[t] = dot8(wf, xf, acc[t]);
      }
    }
  }
}

// ------------------------------------------------------------ gate/up
template <int MT>
__global__ void __launch_bounds__(128) decode_gate_up_kernel(
    const __nv_bfloat16* __restrict__ hidden, int H, int I, int k,
    const __nv_bfloat16* __restrict__ wgu, const int* __restrict__ offsets,
    const int* __restrict__ touched, const int* __restrict__ sorted_f,
    __nv_bfloat16* __restrict__ h_out, int act) {
  pdl_launch_dependents();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int per_e = I / 4;
  const long n_items = static_cast<long>(__ldg(touched)) * per_e;
  const int H8 = H / 8;
  for (long item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int e = __ldg(touched + 1 + static_cast<int>(item / per_e));
    const int f = static_cast<int>(item % per_e) * 4 + warp;
    const int r0 = __ldg(offsets + e);
    const int m = __ldg(offsets + e + 1) - r0;
    const uint4* wg = reinterpret_cast<const uint4*>(wgu + (static_cast<long>(e) * 2 * I + f) * H);
    const uint4* wu = reinterpret_cast<const uint4*>(wgu + (static_cast<long>(e) * 2 * I + I + f) * H);
    for (int t0 = 0; t0 < m; t0 += MT) {
      const uint4* xr[MT];
#pragma unroll
      for (int t = 0; t < MT; ++t) {
        const int tt = min(t0 + t, m - 1);
        xr[t] = reinterpret_cast<const uint4*>(hidden) +
                static_cast<long>(__ldg(sorted_f + r0 + tt) / k) * H8;
      }
      float ag[MT], au[MT];
#pragma unroll
      for (int t = 0; t < MT; ++t) ag[t] = au[t] = 0.f;
      stream_dot2<MT>(wg, wu, xr, H8, lane, ag, au);
#pragma unroll
      for (int t = 0; t < MT; ++t) {
        const float g = warp_sum(ag[t]);
        const float u = warp_sum(au[t]);
        if (lane == 0 && t0 + t < m)
          h_out[static_cast<long>(r0 + t0 + t) * I + f] = __float2bfloat16_rn(gate_act(g, act) * u);
      }
    }
  }
}

// ------------------------------------------------------------ down
template <int MT>
__global__ void __launch_bounds__(128) decode_down_kernel(
    const __nv_bfloat16* __restrict__ h, int H, int I, const __nv_bfloat16* __restrict__ wd,
    const int* __restrict__ offsets, const int* __restrict__ touched,
    const int* __restrict__ sorted_f, const float* __restrict__ topk_w, float* __restrict__ Y) {
  pdl_launch_dependents();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int per_e = H / 4;
  const long n_items = static_cast<long>(__ldg(touched)) * per_e;
  const int I8 = I / 8;
  for (long item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int e = __ldg(touched + 1 + static_cast<int>(item / per_e));
    const int c = static_cast<int>(item % per_e) * 4 + warp;
    const int r0 = __ldg(offsets + e);
    const int m = __ldg(offsets + e + 1) - r0;
    const uint4* wr = reinterpret_cast<const uint4*>(wd + (static_cast<long>(e) * H + c) * I);
    for (int t0 = 0; t0 < m; t0 += MT) {
      const uint4* hr[MT];
#pragma unroll
      for (int t = 0; t < MT; ++t)
        hr[t] = reinterpret_cast<const uint4*>(h) + static_cast<long>(r0 + min(t0 + t, m - 1)) * I8;
      float acc[MT];
#pragma unroll
      for (int t = 0; t < MT; ++t) acc[t] = 0.f;
      stream_dot1<MT>(wr, hr, I8, lane, acc);
#pragma unroll
      for (int t = 0; t < MT; ++t) {
        const float y = warp_sum(acc[t]);
        if (lane == 0 && t0 + t < m) {
          const int r = r0 + t0 + t;
          Y[static_cast<long>(r) * H + c] = y * __ldg(topk_w + __ldg(sorted_f + r));
        }
      }
    }
  }
}

// ------------------------------------------------------------ combine
__global__ void __launch_bounds__(256) decode_combine_kernel(const float4* __restrict__ Y,
                                                             const int* __restrict__ row_of,
                                                             int T, int H, int k,
                                                             uint2* __restrict__ out) {
  pdl_launch_dependents();
  pdl_wait();
  const int H4 = H / 4;
  const long total = static_cast<long>(T) * H4;
  for (long i = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<long>(gridDim.x) * blockDim.x) {
    const long t = i / H4;
    const int c4 = static_cast<int>(i - t * H4);
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < k; ++j) {
      const int r = __ldg(row_of + t * k + j);
      if (r < 0) continue;
      const float4 y = __ldg(Y + static_cast<long>(r) * H4 + c4);
      s.x += y.x;
      s.y += y.y;
      s.z += y.z;
      s.w += y.w;
    }
    out[i] = make_uint2(pack_bf16x2(s.x, s.y), pack_bf16x2(s.z, s.w));
  }
}

// ------------------------------------------------------------ fused (tiny T*k)
// For T*k <= kFusedDecodeRows every CTA rebuilds the routing table itself in
// shared memory (stable order by expert, touched list), so no dispatch
// kernel runs; the down GEMV also sums the k contributions of each token in
// place, so no combine kernel runs either.
template <int MT>
__global__ void __launch_bounds__(128) decode_fused_gate_up_kernel(
    const __nv_bfloat16* __restrict__ hidden, int H, int I, int k, int E, int n,
    const __nv_bfloat16* __restrict__ wgu, const int32_t* __restrict__ topk_idx,
    __nv_bfloat16* __restrict__ h_out, int* err, int act) {
  pdl_launch_dependents();
  pdl_wait();
  __shared__ SmallTable tab;
  build_small_table(topk_idx, n, E, tab, err);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int per_e = I / 4;
  const int n_items = tab.nt * per_e;
  const int H8 = H / 8;
  for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int j = item / per_e;
    const int e = tab.te[j];
    const int f = (item - j * per_e) * 4 + warp;
    const int r0 = tab.tb[j];
    const int m = tab.tb[j + 1] - r0;
    const uint4* wg = reinterpret_cast<const uint4*>(wgu + (static_cast<long>(e) * 2 * I + f) * H);
    const uint4* wu = reinterpret_cast<const uint4*>(wgu + (static_cast<long>(e) * 2 * I + I + f) * H);
    for (int t0 = 0; t0 < m; t0 += MT) {
      const uint4* xr[MT];
#pragma unroll
      for (int t = 0; t < MT; ++t)
        xr[t] = reinterpret_cast<const uint4*>(hidden) +
                static_cast<long>(tab.sf[r0 + min(t0 + t, m - 1)] / k) * H8;
      float ag[MT], au[MT];
#pragma unroll
      for (int t = 0; t < MT; ++t) ag[t] = au[t] = 0.f;
      stream_dot2<MT>(wg, wu, xr, H8, lane, ag, au);
#pragma unroll
      for (int t = 0; t < MT; ++t) {
        const float gs = warp_sum(ag[t]);
        const float us = warp_sum(au[t]);
        if (lane == 0 && t0 + t < m)
          h_out[static_cast<long>(r0 + t0 + t) * I + f] = __float2bfloat16_rn(gate_act(gs, act) * us);
      }
    }
  }
}

// One output column per block: its four warps split the touched experts,
// each streaming W_down[e, c, :] once and adding w * y per token into its
// shared-memory row; the block then sums the four rows and writes the bf16
// outputs of the column.
template <int MT>
__global__ void __launch_bounds__(128) decode_fused_down_kernel(
    const __nv_bfloat16* __restrict__ h, int T, int H, int I, int k, int E, int n,
    const __nv_bfloat16* __restrict__ wd, const int32_t* __restrict__ topk_idx,
    const float* __restrict__ topk_w, __nv_bfloat16* __restrict__ out, int* err) {
  pdl_launch_dependents();
  pdl_wait();
  __shared__ SmallTable tab;
  __shared__ float s_acc[4][kFusedDecodeRows];
  build_small_table(topk_idx, n, E, tab, err);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int I8 = I / 8;
  for (int c = blockIdx.x; c < H; c += gridDim.x) {
    for (int t = lane; t < T; t += 32) s_acc[warp][t] = 0.f;
    __syncwarp();
    for (int j = warp; j < tab.nt; j += 4) {
      const int e = tab.te[j];
      const int r0 = tab.tb[j];
      const int m = tab.tb[j + 1] - r0;
      const uint4* wr = reinterpret_cast<const uint4*>(wd + (static_cast<long>(e) * H + c) * I);
      for (int t0 = 0; t0 < m; t0 += MT) {
        const uint4* hr[MT];
#pragma unroll
        for (int t = 0; t < MT; ++t)
          hr[t] = reinterpret_cast<const uint4*>(h) + static_cast<long>(r0 + min(t0 + t, m - 1)) * I8;
        float acc[MT];
#pragma unroll
        for (int t = 0; t < MT; ++t) acc[t] = 0.f;
        stream_dot1<MT>(wr, hr, I8, lane, acc);
#pragma unroll
        for (int t = 0; t < MT; ++t) {
          const float y = warp_sum(acc[t]);
          if (lane == 0 && t0 + t < m) {
            const int f = tab.sf[r0 + t0 + t];
            s_acc[warp][f / k] += y * __ldg(topk_w + f);
          }
        }
      }
    }
    __syncthreads();
    for (int t = threadIdx.x; t < T; t += 128)
      out[static_cast<long>(t) * H + c] =
          __float2bfloat16_rn(s_acc[0][t] + s_acc[1][t] + s_acc[2][t] + s_acc[3][t]);
    __syncthreads();
  }
}

// ------------------------------------------------------------ launchers
cudaError_t launch_dispatch_small(const int32_t* topk_idx, int T, int E, int k,
                                  const DispatchBufs& d, cudaStream_t s) {
  const int n = T * k;
  launch_pdl(dispatch_small_kernel, 1, 1024, 0, s, topk_idx, n, E, d.counts, d.offsets, d.tile_pref,
                                           d.touched, d.sorted_f, d.row_of, d.err);
  count_launches(1);
  return cudaGetLastError();
}

static int mt_for(int T) { return T >= 8 ? 8 : T >= 4 ? 4 : T >= 2 ? 2 : 1; }

static int decode_grid(const DecodeArgs& a, long items_per_expert) {
  const long n_exp_max = a.E < static_cast<long>(a.T) * a.k ? a.E : static_cast<long>(a.T) * a.k;
  const long items = n_exp_max * items_per_expert;
  const long slots = static_cast<long>(a.num_sms) * 16;
  return static_cast<int>(items < slots ? items : slots);
}

cudaError_t launch_decode_gate_up(const DecodeArgs& a, cudaStream_t s) {
  const int grid = decode_grid(a, a.I / 4);
  auto* hb = static_cast<__nv_bfloat16*>(a.h);
  auto* hid = static_cast<const __nv_bfloat16*>(a.hidden);
  auto* w = static_cast<const __nv_bfloat16*>(a.w_gate_up);
  switch (mt_for(a.T)) {
    case 8: launch_pdl(decode_gate_up_kernel<8>, grid, 128, 0, s, hid, a.H, a.I, a.k, w, a.offsets, a.touched, a.sorted_f, hb, a.act); break;
    case 4: launch_pdl(decode_gate_up_kernel<4>, grid, 128, 0, s, hid, a.H, a.I, a.k, w, a.offsets, a.touched, a.sorted_f, hb, a.act); break;
    case 2: launch_pdl(decode_gate_up_kernel<2>, grid, 128, 0, s, hid, a.H, a.I, a.k, w, a.offsets, a.touched, a.sorted_f, hb, a.act); break;
    default: launch_pdl(decode_gate_up_kernel<1>, grid, 128, 0, s, hid, a.H, a.I, a.k, w, a.offsets, a.touched, a.sorted_f, hb, a.act); break;
  }
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_decode_down(const DecodeArgs& a, cudaStream_t s) {
  const int grid = decode_grid(a, a.H / 4);
  auto* hb = static_cast<const __nv_bfloat16*>(a.h);
  auto* w = static_cast<const __nv_bfloat16*>(a.w_down);
  switch (mt_for(a.T)) {
    case 8: launch_pdl(decode_down_kernel<8>, grid, 128, 0, s, hb, a.H, a.I, w, a.offsets, a.touched, a.sorted_f, a.topk_w, a.Y); break;
    case 4: launch_pdl(decode_down_kernel<4>, grid, 128, 0, s, hb, a.H, a.I, w, a.offsets, a.touched, a.sorted_f, a.topk_w, a.Y); break;
    case 2: launch_pdl(decode_down_kernel<2>, grid, 128, 0, s, hb, a.H, a.I, w, a.offsets, a.touched, a.sorted_f, a.topk_w, a.Y); break;
    default: launch_pdl(decode_down_kernel<1>, grid, 128, 0, s, hb, a.H, a.I, w, a.offsets, a.touched, a.sorted_f, a.topk_w, a.Y); break;
  }
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_decode_fused_gate_up(const DecodeArgs& a, const int32_t* topk_idx, int* err,
                                       cudaStream_t s) {
  const int n = a.T * a.k;
  const int grid = decode_grid(a, a.I / 4);
  auto* hb = static_cast<__nv_bfloat16*>(a.h);
  auto* hid = static_cast<const __nv_bfloat16*>(a.hidden);
  auto* w = static_cast<const __nv_bfloat16*>(a.w_gate_up);
  switch (mt_for(a.T)) {
    case 8: launch_pdl(decode_fused_gate_up_kernel<8>, grid, 128, 0, s, hid, a.H, a.I, a.k, a.E, n, w, topk_idx, hb, err, a.act); break;
    case 4: launch_pdl(decode_fused_gate_up_kernel<4>, grid, 128, 0, s, hid, a.H, a.I, a.k, a.E, n, w, topk_idx, hb, err, a.act); break;
    case 2: launch_pdl(decode_fused_gate_up_kernel<2>, grid, 128, 0, s, hid, a.H, a.I, a.k, a.E, n, w, topk_idx, hb, err, a.act); break;
    default: launch_pdl(decode_fused_gate_up_kernel<1>, grid, 128, 0, s, hid, a.H, a.I, a.k, a.E, n, w, topk_idx, hb, err, a.act); break;
  }
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_decode_fused_down(const DecodeArgs& a, const int32_t* topk_idx, int* err,
                                     cudaStream_t s) {
  const int n = a.T * a.k;
  const long want = a.H;
  const long slots = static_cast<long>(a.num_sms) * 16;
  const int grid = static_cast<int>(want < slots ? want : slots);
  auto* hb = static_cast<const __nv_bfloat16*>(a.h);
  auto* w = static_cast<const __nv_bfloat16*>(a.w_down);
  auto* o = static_cast<__nv_bfloat16*>(a.out);
  switch (mt_for(a.T)) {
    case 8: launch_pdl(decode_fused_down_kernel<8>, grid, 128, 0, s, hb, a.T, a.H, a.I, a.k, a.E, n, w, topk_idx, a.topk_w, o, err); break;
    case 4: launch_pdl(decode_fused_down_kernel<4>, grid, 128, 0, s, hb, a.T, a.H, a.I, a.k, a.E, n, w, topk_idx, a.topk_w, o, err); break;
    case 2: launch_pdl(decode_fused_down_kernel<2>, grid, 128, 0, s, hb, a.T, a.H, a.I, a.k, a.E, n, w, topk_idx, a.topk_w, o, err); break;
    default: launch_pdl(decode_fused_down_kernel<1>, grid, 128, 0, s, hb, a.T, a.H, a.I, a.k, a.E, n, w, topk_idx, a.topk_w, o, err); break;
  }
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_decode_combine(const DecodeArgs& a, cudaStream_t s) {
  const long total = static_cast<long>(a.T) * (a.H / 4);
  const long want = (total + 255) / 256;
  const long slots = static_cast<long>(a.num_sms) * 16;
  const int grid = static_cast<int>(want < slots ? want : slots);
  launch_pdl(decode_combine_kernel, grid, 256, 0, s, reinterpret_cast<const float4*>(a.Y), a.row_of, a.T,
                                             a.H, a.k, static_cast<uint2*>(a.out));
  count_launches(1);
  return cudaGetLastError();
}

bool decode_fused_fits(const DecodeArgs& a) {
  return static_cast<long>(a.T) * a.k <= kFusedDecodeRows;
}

}  // namespace moe
