// Single-launch small-token decode path (bf16 weights, T*k <= 64 routed
// rows): the gate/up GEMV and the down GEMV with the combine in one kernel,
// so that the down projection's weight stream overlaps the gate/up stream
// instead of following it (the page's "Decode-stage switching" idea: a
// separate strategy for low token counts, where the forward is a stream over
// the touched experts' weights).
//
// Every CTA rebuilds the routing table in shared memory (stable order by
// expert, touched list), as the two-kernel fused path does.  Then:
//   phase A  one gate/up feature per warp item: the gate and up rows of
//            W_gate_up[e] streamed once against the expert's token rows,
//            h = act(g) * u stored in bf16; then the CTA publishes its h
//            (fence, then one increment of a device-wide counter)
//   phase B  a CTA item is a group of output columns c; its (expert, c)
//            rows of W_down are spread over the eight warps.  On its first
//            item every warp issues the loads of the first 8 x 16 bytes per
//            lane of its first row, then one thread of the CTA waits for
//            every CTA's h (bounded spin on the counter); the warps finish
//            the dot products with the expert's h rows, and the CTA sums the
//            k contributions of each token in ascending expert order and
//            writes the bf16 outputs of its columns.
// The grid is at most what the GPU holds at once (cooperative launch), so a
// CTA that waits never keeps another from running.  The last CTA to finish
// resets the counters for the next launch.  The wait gives up after a
// bounded time, flags the error word and skips its work.
#include <atomic>

#include "decode_common.cuh"

namespace moe {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kPre = 8;                       // 16-byte W_down vectors per lane loaded before the wait
constexpr int kItemRows = kFusedDecodeRows;   // (expert, column) rows per phase-B item, at most

__device__ __forceinline__ int ld_acquire_gpu(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// One thread waits (bounded) until *ctr >= target; a barrier after it
// hands the acquired view of memory to the rest of the CTA.
__device__ __forceinline__ bool cta_wait_count(const int* ctr, int target, int* err) {
  if (ld_acquire_gpu(ctr) >= target) return true;
  const uint64_t t0 = globaltimer_ns();
  while (ld_acquire_gpu(ctr) < target) {
    __nanosleep(256);
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      atomicOr(err, ERR_TIMEOUT_EPILOGUE);
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ void bf16x8(const uint4& v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

template <int MT>
__global__ void __launch_bounds__(kThreads) decode_single_kernel(
    const __nv_bfloat16* __restrict__ hidden, int T, int H, int I, int k, int E, int n,
    const __nv_bfloat16* __restrict__ wgu, const __nv_bfloat16* __restrict__ wd,
    const int32_t* __restrict__ topk_idx, const float* __restrict__ topk_w,
    __nv_bfloat16* h, __nv_bfloat16* __restrict__ out, int* head, int act) {
  pdl_launch_dependents();
  pdl_wait();
  __shared__ SmallTable tab;
  __shared__ float s_y[kItemRows][kFusedDecodeRows];
  int* err = head;
  int* arrive = head + kSyncArriveWord;
  int* done = head + kSyncDoneWord;
  build_small_table(topk_idx, n, E, tab, err);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H8 = H / 8, I8 = I / 8;
  const int nt = tab.nt;

  // ---------------------------------------------------------------- phase A
  const long nA = static_cast<long>(nt) * I;
  for (long item = static_cast<long>(blockIdx.x) * kWarps + warp; item < nA;
       item += static_cast<long>(gridDim.x) * kWarps) {
    const int j = static_cast<int>(item / I);
    const int f = static_cast<int>(item - static_cast<long>(j) * I);
    const int e = tab.te[j];
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
      for (int c0 = lane; c0 < H8; c0 += 32 * kPre) {
        uint4 g[kPre], u[kPre];
#pragma unroll
        for (int i = 0; i < kPre; ++i) {
          const int c = c0 + 32 * i;
          g[i] = c < H8 ? ld_stream(wg + c) : make_uint4(0, 0, 0, 0);
          u[i] = c < H8 ? ld_stream(wu + c) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int i = 0; i < kPre; ++i) {
          const int c = c0 + 32 * i;
          if (c >= H8) break;
          float gf[8], uf[8];
          bf16x8(g[i], gf);
          bf16x8(u[i], uf);
#pragma unroll
          for (int t = 0; t < MT; ++t) {
            float xf[8];
            bf16x8(__ldg(xr[t] + c), xf);
            ag[t] = dot8(gf, xf, ag[t]);
            au[t] = dot8(uf, xf, au[t]);
          }
        }
      }
#pragma unroll
      for (int t = 0; t < MT; ++t) {
        const float gs = warp_sum(ag[t]);
        const float us = warp_sum(au[t]);
        if (lane == 0 && t0 + t < m)
          h[static_cast<long>(r0 + t0 + t) * I + f] = __float2bfloat16_rn(gate_act(gs, act) * us);
      }
    }
  }
  // publish this CTA's h before it counts itself in
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) atomicAdd(arrive, 1);

  // ---------------------------------------------------------------- phase B
  const int cpi = nt >= kWarps ? 1 : kWarps / max(nt, 1);   // columns per item
  const int rows_item = cpi * nt;                    // <= max(8, nt) <= kItemRows
  const int n_items = (H + cpi - 1) / cpi;
  __shared__ int s_h_ok;
  bool waited = false;
  for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int c0 = item * cpi;
    for (int i = threadIdx.x; i < rows_item * kFusedDecodeRows; i += kThreads)
      s_y[i / kFusedDecodeRows][i % kFusedDecodeRows] = 0.f;
    // the first row of each warp: its first weights are loaded before h is
    // known to be ready
    const int q0 = warp;
    const bool has0 = q0 < rows_item && c0 + q0 / max(nt, 1) < H;
    uint4 pre[kPre];
    if (has0) {
      const int e = tab.te[q0 - (q0 / nt) * nt];
      const uint4* wr =
          reinterpret_cast<const uint4*>(wd + (static_cast<long>(e) * H + c0 + q0 / nt) * I);
#pragma unroll
      for (int i = 0; i < kPre; ++i) {
        const int idx = lane + 32 * i;
        pre[i] = idx < I8 ? ld_stream(wr + idx) : make_uint4(0, 0, 0, 0);
      }
    }
    if (!waited) {
      // one thread per CTA waits for every CTA's h (bounded), the others at
      // the barrier
      if (threadIdx.x == 0) s_h_ok = cta_wait_count(arrive, gridDim.x, err) ? 1 : 0;
      waited = true;
    }
    __syncthreads();
    if (!s_h_ok) break;
    for (int q = warp; q < rows_item; q += kWarps) {
      const int cc = q / nt, j = q - cc * nt;
      const int c = c0 + cc;
      if (c >= H) continue;
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
        // first batch: the preloaded weights (loaded again for later token chunks and rows)
#pragma unroll
        for (int i = 0; i < kPre; ++i) {
          const int idx = lane + 32 * i;
          if (idx >= I8) break;
          const uint4 wv = (q == q0 && t0 == 0) ? pre[i] : __ldg(wr + idx);
          float wf[8];
          bf16x8(wv, wf);
#pragma unroll
          for (int t = 0; t < MT; ++t) {
            float hf[8];
            bf16x8(__ldcg(hr[t] + idx), hf);
            acc[t] = dot8(wf, hf, acc[t]);
          }
        }
        // the rest of the row
        for (int b0 = lane + 32 * kPre; b0 < I8; b0 += 32 * kPre) {
          uint4 v[kPre];
#pragma unroll
          for (int i = 0; i < kPre; ++i) {
            const int idx = b0 + 32 * i;
            v[i] = idx < I8 ? ld_stream(wr + idx) : make_uint4(0, 0, 0, 0);
          }
#pragma unroll
          for (int i = 0; i < kPre; ++i) {
            const int idx = b0 + 32 * i;
            if (idx >= I8) break;
            float wf[8];
            bf16x8(v[i], wf);
#pragma unroll
            for (int t = 0; t < MT; ++t) {
              float hf[8];
              bf16x8(__ldcg(hr[t] + idx), hf);
              acc[t] = dot8(wf, hf, acc[t]);
            }
          }
        }
#pragma unroll
        for (int t = 0; t < MT; ++t) {
          const float y = warp_sum(acc[t]);
          if (lane == 0 && t0 + t < m) {
            const int f = tab.sf[r0 + t0 + t];
            s_y[q][f / k] = y * __ldg(topk_w + f);
          }
        }
      }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < cpi * T; i += kThreads) {
      const int cc = i / T, t = i - cc * T;
      const int c = c0 + cc;
      if (c >= H) continue;
      float s = 0.f;
      for (int j = 0; j < nt; ++j) s += s_y[cc * nt + j][t];
      out[static_cast<long>(t) * H + c] = __float2bfloat16_rn(s);
    }
    __syncthreads();
  }

  // the last CTA out resets the counters for the next launch on this workspace
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(done, 1) == static_cast<int>(gridDim.x) - 1) {
      atomicExch(arrive, 0);
      atomicExch(done, 0);
    }
  }
}

// CTAs of one instantiation the GPU holds at once, per device (0 = unknown).
template <int MT>
int resident_blocks(int dev, int num_sms) {
  static std::atomic<int> cache[64] = {};
  if (dev >= 0 && dev < 64) {
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c) return c;
  }
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_single_kernel<MT>, kThreads, 0) !=
      cudaSuccess)
    return 0;
  const int total = per_sm * num_sms;
  if (dev >= 0 && dev < 64) cache[dev].store(total, std::memory_order_relaxed);
  return total;
}

template <int MT>
cudaError_t launch_single(const DecodeArgs& a, const int32_t* topk_idx, int* head, cudaStream_t s) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int cap = resident_blocks<MT>(dev, a.num_sms);
  if (cap <= 0) return cudaErrorCooperativeLaunchTooLarge;
  const int n = a.T * a.k;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cap);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, decode_single_kernel<MT>, static_cast<const __nv_bfloat16*>(a.hidden),
                         a.T, a.H, a.I, a.k, a.E, n, static_cast<const __nv_bfloat16*>(a.w_gate_up),
                         static_cast<const __nv_bfloat16*>(a.w_down), topk_idx, a.topk_w,
                         static_cast<__nv_bfloat16*>(a.h), static_cast<__nv_bfloat16*>(a.out), head,
                         a.act);
  if (e == cudaSuccess) count_launches(1);
  return e;
}

}  // namespace

cudaError_t launch_decode_single(const DecodeArgs& a, const int32_t* topk_idx, int* head,
                                 cudaStream_t s) {
  const int T = a.T;
  if (T >= 8) return launch_single<8>(a, topk_idx, head, s);
  if (T >= 4) return launch_single<4>(a, topk_idx, head, s);
  if (T >= 2) return launch_single<2>(a, topk_idx, head, s);
  return launch_single<1>(a, topk_idx, head, s);
}

}  // namespace moe
