// FP4 (e2m1) experts on the small-token path.  The page's "FP8 and FP4
// quantized experts" section names FP4-packed expert weights (two codes per
// int8) with UE8M0 weight scales, and dynamic per-row activation scales.
// This file runs that format for routed batches of at most kFusedDecodeRows
// rows, where the forward is a stream over the touched experts' packed
// weights, on CUDA cores.
//
// Formats:
//   weights      e2m1 codes, two per byte, the even element in the low
//                nibble, one UE8M0 byte (scale 2^(b-127)) per 1x32 block
//                along the contraction axis: W_gate_up [E, 2I, H/2] with
//                scales [E, 2I, H/32], W_down [E, H, I/2] with [E, H, I/32].
//                A 16-byte vector of codes is exactly one scale block.
//   activations  the hidden rows and h are quantised to e4m3 in 1x32 UE8M0
//                blocks (scale = smallest power of two >= amax/448); the
//                kernels keep the dequantised values, exact in fp32, in eight
//                "planes" per row (float4 group g of block c at g * C/32 + c),
//                so that the lanes of a warp, one block each, load 512
//                contiguous bytes per group.
//
//   fp4_quant_x      hidden [T, H] bf16 -> quantised values, fp32 [T, H]
//   fp4_gate_up      item = (touched expert, 32 features), 8 features per
//                    warp: gate and up rows streamed once against the
//                    expert's token rows (in chunks of 8, 4, 2, 1 rows, so
//                    no row is computed twice); h = act(g) * u of the 32 features
//                    is one 1x32 block per row, quantised in the CTA ->
//                    fp32 [n, I] in expert-sorted row order
//   fp4_down         2 output columns per warp: their W_down rows streamed
//                    once per touched expert, w * y summed per token in
//                    shared memory (ascending expert order), bf16 out
//   fp4_quantize     offline: bf16 weights -> packed codes + UE8M0 bytes
#include <cuda_fp16.h>

#include <type_traits>

#include "decode_common.cuh"

namespace moe {

namespace {

constexpr int kFp4Block = 32;  // elements per scale; one 16-byte code vector
constexpr int kFp4Batch = 4;   // code vectors per row a lane loads before the math

__device__ __forceinline__ float ue8m0_value(uint32_t b) {
  return b == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(b << 23);
}

// bf16 bit patterns of the e2m1 magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6
// (codes 0..7) split into high and low bytes; byte c of a table (first word
// = bytes 0..3, second = bytes 4..7) belongs to code c.
constexpr uint32_t kMagHi0 = 0x3F3F3F00u, kMagHi1 = 0x40404040u;
constexpr uint32_t kMagLo0 = 0xC0800000u, kMagLo1 = 0xC0804000u;

// Eight e2m1 codes (nibble i of v = element i) -> their exact fp32 values.
// The magnitude's two bytes come from byte-permute table lookups indexed by
// the low three bits of each nibble; the sign is nibble bit 3.
__device__ __forceinline__ void e2m1x8_to_f32(uint32_t v, float (&f)[8]) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint32_t sel = (v >> (16 * h)) & 0x7777u;  // selectors of elements 4h..4h+3
    const uint32_t hi = __byte_perm(kMagHi0, kMagHi1, sel);
    const uint32_t lo = __byte_perm(kMagLo0, kMagLo1, sel);
    const uint32_t p01 = __byte_perm(lo, hi, 0x5140);  // bf16 of elements 4h, 4h+1
    const uint32_t p23 = __byte_perm(lo, hi, 0x7362);  // elements 4h+2, 4h+3
    const uint32_t bits[4] = {p01 << 16, p01 & 0xFFFF0000u, p23 << 16, p23 & 0xFFFF0000u};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = 4 * h + i;
      f[e] = __uint_as_float(bits[i] | ((v << (28 - 4 * e)) & 0x80000000u));
    }
  }
}

// acc_a[t] += row_a . x_t and acc_b[t] += row_b . x_t for two packed e2m1
// rows of nblk 32-element blocks (codes wa/wb, UE8M0 bytes sa/sb) and fp32
// rows x_t stored in planes: float4 group g (elements 4g..4g+3) of block c
// at x_t[g * nblk + c].  Lane handles blocks lane, lane+32, ..., so the 32
// lanes' loads of one group are 512 contiguous bytes; per block the code
// products are summed first and then scaled once.
template <int MT>
__device__ __forceinline__ void fp4_dot2(const uint4* __restrict__ wa, const uint8_t* __restrict__ sa,
                                         const uint4* __restrict__ wb, const uint8_t* __restrict__ sb,
                                         const float4* const (&xr)[MT], int nblk, int lane,
                                         float (&acc_a)[MT], float (&acc_b)[MT]) {
  for (int c0 = lane; c0 < nblk; c0 += 32 * kFp4Batch) {
    uint4 va[kFp4Batch], vb[kFp4Batch];
    uint32_t ea[kFp4Batch], eb[kFp4Batch];
#pragma unroll
    for (int i = 0; i < kFp4Batch; ++i) {
      const int c = c0 + 32 * i;
      const bool in = c < nblk;
      va[i] = in ? ld_stream(wa + c) : make_uint4(0, 0, 0, 0);
      vb[i] = in ? ld_stream(wb + c) : make_uint4(0, 0, 0, 0);
      ea[i] = in ? __ldg(sa + c) : 0u;
      eb[i] = in ? __ldg(sb + c) : 0u;
    }
#pragma unroll
    for (int i = 0; i < kFp4Batch; ++i) {
      const int c = c0 + 32 * i;
      if (c >= nblk) break;
      float pa[MT], pb[MT];
#pragma unroll
      for (int t = 0; t < MT; ++t) pa[t] = pb[t] = 0.f;
      const uint32_t wa4[4] = {va[i].x, va[i].y, va[i].z, va[i].w};
      const uint32_t wb4[4] = {vb[i].x, vb[i].y, vb[i].z, vb[i].w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {  // elements 8q .. 8q+7 of the block
        float fa[8], fb[8];
        e2m1x8_to_f32(wa4[q], fa);
        e2m1x8_to_f32(wb4[q], fb);
#pragma unroll
        for (int t = 0; t < MT; ++t) {
          const float4 x0 = __ldg(xr[t] + (2 * q) * nblk + c);
          const float4 x1 = __ldg(xr[t] + (2 * q + 1) * nblk + c);
          const float xf[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
          pa[t] = dot8(fa, xf, pa[t]);
          pb[t] = dot8(fb, xf, pb[t]);
        }
      }
      const float scale_a = ue8m0_value(ea[i]), scale_b = ue8m0_value(eb[i]);
#pragma unroll
      for (int t = 0; t < MT; ++t) {
        acc_a[t] = fmaf(pa[t], scale_a, acc_a[t]);
        acc_b[t] = fmaf(pb[t], scale_b, acc_b[t]);
      }
    }
  }
}

__device__ __forceinline__ float warp_absmax(float v) {
  v = fabsf(v);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
  return v;
}

__device__ __forceinline__ float2 e4m3x2_to_f32(uint16_t codes) {
  const __half2_raw r = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(codes), __NV_E4M3);
  return __half22float2(__half2(r));
}

// e2m1 code of y (fp32): the nearest of 0, 0.5, 1, 1.5, 2, 3, 4, 6 with ties
// to the even code, saturating at 6; bit 3 is y's sign bit.  Each threshold
// is a midpoint, counted with >= where the upper neighbour has the even code.
__device__ __forceinline__ uint32_t e2m1_code(float y) {
  const float a = fabsf(y);
  const uint32_t m = (a > 0.25f) + (a >= 0.75f) + (a > 1.25f) + (a >= 1.75f) + (a > 2.5f) +
                     (a >= 3.5f) + (a > 5.0f);
  return m | ((__float_as_uint(y) >> 28) & 8u);
}

// ------------------------------------------------------------ activations
// One thread per 1x32 block of hidden: e4m3 codes with a UE8M0 scale, kept
// as their values (code value * scale, exact in fp32), in the plane layout
// the GEMVs read: row t, block c, group g at xdq[t * H/4 + g * rblk + c].
__global__ void __launch_bounds__(256) fp4_quant_x_kernel(const uint4* __restrict__ hidden, long nblk,
                                                          int rblk, float4* __restrict__ xdq) {
  pdl_launch_dependents();
  pdl_wait();
  for (long b = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x; b < nblk;
       b += static_cast<long>(gridDim.x) * blockDim.x) {
    float x[kFp4Block];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 v = __ldg(hidden + b * 4 + i);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        x[8 * i + 2 * j] = __uint_as_float(w[j] << 16);
        x[8 * i + 2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
      }
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < kFp4Block; ++i) amax = fmaxf(amax, fabsf(x[i]));
    uint32_t stored;
    const float sc = block_scale(amax, true, &stored);
    const float inv = 1.0f / sc;
#pragma unroll
    for (int i = 0; i < kFp4Block / 2; ++i) {
      const float2 d = e4m3x2_to_f32(e4m3x2(x[2 * i] * inv, x[2 * i + 1] * inv));
      x[2 * i] = d.x * sc;
      x[2 * i + 1] = d.y * sc;
    }
    const long t = b / rblk, c = b - t * rblk;
    float4* row = xdq + t * (rblk * 8);
#pragma unroll
    for (int i = 0; i < kFp4Block / 4; ++i)
      row[i * rblk + c] = make_float4(x[4 * i], x[4 * i + 1], x[4 * i + 2], x[4 * i + 3]);
  }
}

// ------------------------------------------------------------ gate/up
template <int MT>
__global__ void __launch_bounds__(128) fp4_gate_up_kernel(
    const float* __restrict__ xdq, int H, int I, int k, int E, int n,
    const uint8_t* __restrict__ wgu, const uint8_t* __restrict__ sgu,
    const int32_t* __restrict__ topk_idx, float* __restrict__ hq, int* err, int act) {
  pdl_launch_dependents();
  pdl_wait();
  __shared__ SmallTable tab;
  __shared__ float s_h[kFusedDecodeRows][kFp4Block];
  build_small_table(topk_idx, n, E, tab, err);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nfb = I / kFp4Block;        // h blocks per row
  const int nblk = H / kFp4Block;       // scale blocks per weight row
  const long row_bytes = H / 2;
  const int n_items = tab.nt * nfb;
  for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int j = item / nfb;
    const int fb = item - j * nfb;
    const int e = tab.te[j];
    const int r0 = tab.tb[j];
    const int m = tab.tb[j + 1] - r0;
    // the expert's rows in chunks of 8, 4, 2, 1 (no duplicated rows)
    auto chunk = [&](auto mt_tag, int t0) {
      constexpr int C = decltype(mt_tag)::value;
      const float4* xr[C];
#pragma unroll
      for (int t = 0; t < C; ++t)
        xr[t] = reinterpret_cast<const float4*>(xdq) +
                static_cast<long>(tab.sf[r0 + t0 + t] / k) * (H / 4);
      for (int q = 0; q < 8; ++q) {
        const int fl = warp * 8 + q;                              // feature in the block
        const long ga = static_cast<long>(e) * 2 * I + fb * kFp4Block + fl;  // gate row
        const long ua = ga + I;                                   // up row
        float ag[C], au[C];
#pragma unroll
        for (int t = 0; t < C; ++t) ag[t] = au[t] = 0.f;
        fp4_dot2<C>(reinterpret_cast<const uint4*>(wgu + ga * row_bytes), sgu + ga * nblk,
                    reinterpret_cast<const uint4*>(wgu + ua * row_bytes), sgu + ua * nblk, xr,
                    nblk, lane, ag, au);
#pragma unroll
        for (int t = 0; t < C; ++t) {
          const float g = warp_sum(ag[t]);
          const float u = warp_sum(au[t]);
          if (lane == 0) s_h[t0 + t][fl] = gate_act(g, act) * u;
        }
      }
    };
    for (int t0 = 0; t0 < m;) {
      const int rem = m - t0;
      if (MT >= 8 && rem >= 8) { chunk(std::integral_constant<int, 8>{}, t0); t0 += 8; }
      else if (MT >= 4 && rem >= 4) { chunk(std::integral_constant<int, 4>{}, t0); t0 += 4; }
      else if (MT >= 2 && rem >= 2) { chunk(std::integral_constant<int, 2>{}, t0); t0 += 2; }
      else { chunk(std::integral_constant<int, 1>{}, t0); t0 += 1; }
    }
    __syncthreads();
    // row t's block: lane = feature; stored in the plane layout of the down GEMV
    for (int t = warp; t < m; t += 4) {
      const float v = s_h[t][lane];
      uint32_t stored;
      const float sc = block_scale(warp_absmax(v), true, &stored);
      const float d = e4m3x2_to_f32(e4m3x2(v * (1.0f / sc), 0.f)).x;
      hq[static_cast<long>(r0 + t) * I + ((lane >> 2) * nfb + fb) * 4 + (lane & 3)] = d * sc;
    }
    __syncthreads();
  }
}

// ------------------------------------------------------------ down + combine
template <int MT>
__global__ void __launch_bounds__(128) fp4_down_kernel(
    const float* __restrict__ hq, int T, int H, int I, int k, int E, int n,
    const uint8_t* __restrict__ wd, const uint8_t* __restrict__ sd,
    const int32_t* __restrict__ topk_idx, const float* __restrict__ topk_w,
    __nv_bfloat16* __restrict__ out, int* err) {
  pdl_launch_dependents();
  pdl_wait();
  __shared__ SmallTable tab;
  __shared__ float s_acc[4][2][kFusedDecodeRows];
  build_small_table(topk_idx, n, E, tab, err);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nblk = I / kFp4Block;
  const long row_bytes = I / 2;
  const int npairs = H / 2;
  float(&acc)[2][kFusedDecodeRows] = s_acc[warp];
  for (int p = blockIdx.x * 4 + warp; p < npairs; p += gridDim.x * 4) {
    const int c = 2 * p;
    for (int t = lane; t < T; t += 32) acc[0][t] = acc[1][t] = 0.f;
    __syncwarp();
    for (int j = 0; j < tab.nt; ++j) {
      const int e = tab.te[j];
      const int r0 = tab.tb[j];
      const int m = tab.tb[j + 1] - r0;
      const long ra = static_cast<long>(e) * H + c;  // W_down rows of columns c, c+1
      auto chunk = [&](auto mt_tag, int t0) {
        constexpr int C = decltype(mt_tag)::value;
        const float4* hr[C];
#pragma unroll
        for (int t = 0; t < C; ++t)
          hr[t] = reinterpret_cast<const float4*>(hq) + static_cast<long>(r0 + t0 + t) * (I / 4);
        float ya[C], yb[C];
#pragma unroll
        for (int t = 0; t < C; ++t) ya[t] = yb[t] = 0.f;
        fp4_dot2<C>(reinterpret_cast<const uint4*>(wd + ra * row_bytes), sd + ra * nblk,
                    reinterpret_cast<const uint4*>(wd + (ra + 1) * row_bytes), sd + (ra + 1) * nblk,
                    hr, nblk, lane, ya, yb);
#pragma unroll
        for (int t = 0; t < C; ++t) {
          const float a = warp_sum(ya[t]);
          const float b = warp_sum(yb[t]);
          if (lane == 0) {
            const int f = tab.sf[r0 + t0 + t];
            const float w = __ldg(topk_w + f);
            acc[0][f / k] += a * w;
            acc[1][f / k] += b * w;
          }
        }
      };
      // the expert's rows in chunks of 8, 4, 2, 1 (no duplicated rows)
      for (int t0 = 0; t0 < m;) {
        const int rem = m - t0;
        if (MT >= 8 && rem >= 8) { chunk(std::integral_constant<int, 8>{}, t0); t0 += 8; }
        else if (MT >= 4 && rem >= 4) { chunk(std::integral_constant<int, 4>{}, t0); t0 += 4; }
        else if (MT >= 2 && rem >= 2) { chunk(std::integral_constant<int, 2>{}, t0); t0 += 2; }
        else { chunk(std::integral_constant<int, 1>{}, t0); t0 += 1; }
      }
    }
    __syncwarp();
    for (int t = lane; t < T; t += 32)
      reinterpret_cast<uint32_t*>(out)[(static_cast<long>(t) * H + c) / 2] =
          pack_bf16x2(acc[0][t], acc[1][t]);
    __syncwarp();
  }
}

// ------------------------------------------------------------ weights
// One thread per 1x32 block: UE8M0 scale = smallest power of two >= amax/6
// (amax = 0 -> 1), codes e2m1(x * (1/scale)) packed into one 16-byte vector.
__global__ void __launch_bounds__(256) fp4_quantize_kernel(const uint4* __restrict__ w, long nblk,
                                                           uint4* __restrict__ q,
                                                           uint8_t* __restrict__ scale) {
  pdl_launch_dependents();
  pdl_wait();
  for (long b = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x; b < nblk;
       b += static_cast<long>(gridDim.x) * blockDim.x) {
    float x[kFp4Block];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 v = __ldg(w + b * 4 + i);
      const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        x[8 * i + 2 * j] = __uint_as_float(u[j] << 16);
        x[8 * i + 2 * j + 1] = __uint_as_float(u[j] & 0xFFFF0000u);
      }
    }
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < kFp4Block; ++i) amax = fmaxf(amax, fabsf(x[i]));
    uint32_t stored = 127u;
    float sc = 1.0f;
    if (amax != 0.f) sc = ue8m0_ceil(amax / 6.0f, &stored);
    const float inv = 1.0f / sc;
    uint32_t words[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint32_t wd = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) wd |= e2m1_code(x[8 * i + j] * inv) << (4 * j);
      words[i] = wd;
    }
    q[b] = make_uint4(words[0], words[1], words[2], words[3]);
    scale[b] = static_cast<uint8_t>(stored);
  }
}

// Largest token chunk the kernels instantiate: chunks of 8 rows spilled
// registers, so experts with more rows take several chunks of 4.
int mt_for_fp4(int T) { return T >= 4 ? 4 : T >= 2 ? 2 : 1; }

int grid_for(long items, int num_sms) {
  const long slots = static_cast<long>(num_sms) * 16;
  const long g = items < slots ? items : slots;
  return static_cast<int>(g > 0 ? g : 1);
}

}  // namespace

cudaError_t launch_fp4_quant_x(const Fp4DecodeArgs& a, cudaStream_t s) {
  const long nxb = static_cast<long>(a.T) * (a.H / kFp4Block);
  launch_pdl(fp4_quant_x_kernel, grid_for((nxb + 255) / 256, a.num_sms), 256, 0, s,
             static_cast<const uint4*>(a.hidden), nxb, a.H / kFp4Block,
             reinterpret_cast<float4*>(a.xdq));
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_fp4_gate_up(const Fp4DecodeArgs& a, cudaStream_t s) {
  const int n = a.T * a.k;
  const int g = grid_for(static_cast<long>(n < a.E ? n : a.E) * (a.I / kFp4Block), a.num_sms);
  const auto* w = static_cast<const uint8_t*>(a.w_gate_up);
  const auto* sc = static_cast<const uint8_t*>(a.scale_gate_up);
  switch (mt_for_fp4(a.T)) {
    case 4: launch_pdl(fp4_gate_up_kernel<4>, g, 128, 0, s, a.xdq, a.H, a.I, a.k, a.E, n, w, sc, a.topk_idx, a.hq, a.err, a.act); break;
    case 2: launch_pdl(fp4_gate_up_kernel<2>, g, 128, 0, s, a.xdq, a.H, a.I, a.k, a.E, n, w, sc, a.topk_idx, a.hq, a.err, a.act); break;
    default: launch_pdl(fp4_gate_up_kernel<1>, g, 128, 0, s, a.xdq, a.H, a.I, a.k, a.E, n, w, sc, a.topk_idx, a.hq, a.err, a.act); break;
  }
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_fp4_down(const Fp4DecodeArgs& a, cudaStream_t s) {
  const int n = a.T * a.k;
  const int g = grid_for((a.H / 2 + 3) / 4, a.num_sms);
  const auto* w = static_cast<const uint8_t*>(a.w_down);
  const auto* sc = static_cast<const uint8_t*>(a.scale_down);
  auto* o = static_cast<__nv_bfloat16*>(a.out);
  switch (mt_for_fp4(a.T)) {
    case 4: launch_pdl(fp4_down_kernel<4>, g, 128, 0, s, a.hq, a.T, a.H, a.I, a.k, a.E, n, w, sc, a.topk_idx, a.topk_w, o, a.err); break;
    case 2: launch_pdl(fp4_down_kernel<2>, g, 128, 0, s, a.hq, a.T, a.H, a.I, a.k, a.E, n, w, sc, a.topk_idx, a.topk_w, o, a.err); break;
    default: launch_pdl(fp4_down_kernel<1>, g, 128, 0, s, a.hq, a.T, a.H, a.I, a.k, a.E, n, w, sc, a.topk_idx, a.topk_w, o, a.err); break;
  }
  count_launches(1);
  return cudaGetLastError();
}

cudaError_t launch_quantize_fp4(const void* w, long rows, int cols, uint8_t* q, uint8_t* scale,
                                int num_sms, cudaStream_t s) {
  const long nblk = rows * (cols / kFp4Block);
  if (nblk == 0) return cudaSuccess;
  launch_pdl(fp4_quantize_kernel, grid_for((nblk + 255) / 256, num_sms * 8), 256, 0, s,
             static_cast<const uint4*>(w), nblk, reinterpret_cast<uint4*>(q), scale);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace moe
