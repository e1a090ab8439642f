// Helpers shared by the small-token decode kernels (bf16 and FP4 weights):
// streaming loads, warp reductions and the per-CTA routing table of the
// fused kernels.
#pragma once

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {

// Weights are read once: cache-streaming loads, which the compiler can
// batch ahead of the arithmetic that consumes them.
__device__ __forceinline__ uint4 ld_stream(const uint4* p) { return __ldcs(p); }

__device__ __forceinline__ float dot8(const float (&a)[8], const float (&b)[8], float acc) {
#pragma unroll
  for (int i = 0; i < 8; ++i) acc = fmaf(a[i], b[i], acc);
  return acc;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// For T*k <= kFusedDecodeRows every CTA of a fused decode kernel rebuilds
// the routing table itself in shared memory: rows in stable order by expert
// and the touched experts, ascending.
struct SmallTable {
  int sf[kFusedDecodeRows];       // row r -> flat entry f (stable, by expert)
  int te[kFusedDecodeRows];       // touched experts, ascending
  int tb[kFusedDecodeRows + 1];   // first row of each touched expert (+ end)
  int nt;                         // number of touched experts
  int idx[kFusedDecodeRows];
};

// All threads of the block call this; blockDim.x >= n.
static __device__ void build_small_table(const int32_t* __restrict__ topk_idx, int n, int E,
                                         SmallTable& t, int* err) {
  const int tid = threadIdx.x;
  if (tid < n) t.idx[tid] = __ldg(topk_idx + tid);
  __syncthreads();
  if (tid < n) {
    const int e = t.idx[tid];
    if (e >= 0 && e < E) {
      int rank = 0;
      for (int f2 = 0; f2 < n; ++f2) {
        const int e2 = t.idx[f2];
        rank += (e2 >= 0 && e2 < E) && (e2 < e || (e2 == e && f2 < tid));
      }
      t.sf[rank] = tid;
    } else if (blockIdx.x == 0) {
      atomicOr(err, ERR_BAD_INDEX);
    }
  }
  __syncthreads();
  if (tid == 0) {
    int nv = 0;
    for (int f = 0; f < n; ++f) nv += t.idx[f] >= 0 && t.idx[f] < E;
    int nt = 0, prev = -1;
    for (int r = 0; r < nv; ++r) {
      const int e = t.idx[t.sf[r]];
      if (e != prev) {
        t.te[nt] = e;
        t.tb[nt] = r;
        ++nt;
        prev = e;
      }
    }
    t.tb[nt] = nv;
    t.nt = nt;
  }
  __syncthreads();
}

}  // namespace moe
