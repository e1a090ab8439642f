// FP8 (e4m3) block-scaled grouped GEMMs of the routed experts forward.
//
// Weights carry one scale per 128x128 block, activations one per 1x128 block
// along the contraction axis (float32, or UE8M0 powers of two).  A K-block
// here is 128 e4m3 values = one 128-byte swizzled row = exactly one scale
// block, so
//     acc[r, c] = sum_kb s_a[r, kb] * s_w[c/128, kb] * (sum_{k in kb} qa[r,k] qw[c,k])
// The tensor core computes each K-block's inner sum into a fresh TMEM buffer
// (tcgen05.mma kind::f8f6f4, M=128, N=256, K=32 per instruction); four
// epilogue warpgroups read it back and fold it into fp32 register
// accumulators with the block's scale product.  Two 256-column TMEM buffers
// let the MMA of K-block kb+1 run while K-block kb is being promoted.
//
// The promotion is what bounds this kernel: every K-block each epilogue
// thread reads 64 partial sums in four rounds of two 8-column TMEM loads
// (64 register accumulators and the 96-register ceiling of 18 warps leave
// room for no more) and folds them in with one fused multiply-add each.  Per
// K-block a thread loads its three scales for the next K-block (the row's
// activation scale, and the two weight-block scales at one address across
// the warp); one thread waits for the partial buffer and the others block
// on a named barrier rather than polling it.
//
// Roles (persistent, one CTA per SM, 576 threads):
//   warp 0       TMA producer, 4-stage ring of A 128x128 B + B 256x128 B
//   warp 1       TMEM allocator + MMA issuer
//   warps 2-17   epilogue, four warpgroups (warps 2-5, 6-9, 10-13, 14-17);
//                thread = tile row (TMEM lane), warpgroup = a quarter of the
//                columns, so the per-K-block promotion is spread over 16 warps
//     gate/up:   warpgroup g owns gate columns 32g..32g+31 and the matching up
//                columns; at tile end h = act(g)*u (silu, exact GELU or
//                relu) is re-quantised per row
//                over the tile's 128 columns (one 1x128 block of I; the four
//                warpgroups exchange their row maxima through shared memory)
//     down:      warpgroup g owns output columns 64g..64g+63 (inside weight
//                block row g/2); at tile end y * routing weight is added into
//                the fp32 accumulator of the token (vector reductions)
// All mbarrier waits are bounded as in the bf16 kernel.  The epilogue's
// named barriers (one per K-block, one per gate/up tile for the row maxima)
// cannot be left waiting: the epilogue warps leave their loops only on the
// decision one thread publishes for the K-block, which all of them read.
#include <cuda_fp8.h>

#include <atomic>

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 128;  // e4m3 per 128-byte row = one scale block
constexpr int kStages = 4;
constexpr int kEpiWarps = 16;
constexpr int kEpiGroups = kEpiWarps / 4;
constexpr int kGroupCols = 256 / kEpiGroups;  // partial-sum columns per warpgroup
constexpr int kThreads = 64 + kEpiWarps * 32;
constexpr int kTmemCols = 512;
constexpr int kBufCols = 256;

enum { EPI_SWIGLU_Q = 0, EPI_COMBINE = 1 };

struct L8 {
  static constexpr int A_BYTES = BM * BK;
  static constexpr int B_BYTES = BN * BK;
  static constexpr int STAGE_TX = A_BYTES + B_BYTES;
  static constexpr int OFF_B = kStages * A_BYTES;
  static constexpr int OFF_BAR = OFF_B + kStages * B_BYTES;
  static constexpr int NBARS = 2 * kStages + 2 + 2 + 1 + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBARS * 8;
  static constexpr int OFF_AMAX = OFF_MISC + 16;  // float [2 tiles][kEpiGroups][128]
  static constexpr int OFF_OFF = OFF_AMAX + 2 * kEpiGroups * 128 * 4;
  static constexpr int OFF_PREF = OFF_OFF + (kMaxE + 1) * 4;
  static constexpr int BYTES = OFF_PREF + (kMaxE + 1) * 4;
  static constexpr int SMEM = BYTES + 1024;
};

struct Fp8Dev {
  const int* offsets;
  const int* tile_pref;
  int E, K, I, H, k, n_rows;
  int* err;
  const void* a_scale;  // [n_rows, scale_stride(K/128)], fp32 or UE8M0 byte
  const void* w_scale;  // [E, Nw/128, K/128], fp32 or UE8M0 byte
  int ue8m0;
  uint8_t* hq;          // gate/up: h codes [n_rows, I]
  void* hs;             // gate/up: h scales [n_rows, scale_stride(I/128)]
  float* out32;         // down: [T, H]
  const int* sorted_f;
  const float* topk_w;
  int act;              // moe_activation of the gate/up epilogue
  int group;            // m-tiles per tile group (0: all of the expert's)
  int phases;           // n-tile slices run one after the other (>= 1)
  int l2_hints;         // down: bit 0 accumulator evict_last
};

// Tile -> (expert e, m-tile m, n-tile n).  The n-tiles are cut into
// `phases` equal slices run one after the other (the down GEMM's combine
// then touches a [T, H / phases] slice of the fp32 accumulator at a time);
// inside a slice and an expert the m-tiles run in groups of `group` (0:
// all), a group's tiles for every n-tile of the slice, m fastest.
__device__ __forceinline__ void decode_tile8(int tile, int NT, int E, const int* s_pref,
                                             int group, int phases, int& e, int& m, int& n) {
  const int ntp = NT / phases;
  const int per_phase = s_pref[E] * ntp;
  const int ph = tile / per_phase;
  tile -= ph * per_phase;
  const int v = tile / ntp;
  int lo = 0, hi = E;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_pref[mid] <= v) lo = mid;
    else hi = mid - 1;
  }
  e = lo;
  const int mt = s_pref[e + 1] - s_pref[e];
  const int local = tile - s_pref[e] * ntp;
  const int G = (group > 0 && group < mt) ? group : mt;
  const int g = local / (G * ntp);
  const int gg = min(G, mt - g * G);
  const int r = local - g * G * ntp;
  n = ph * ntp + r / gg;
  m = g * G + (r - (r / gg) * gg);
}

__device__ __forceinline__ float load_scale(const void* base, long i, int ue8m0) {
  if (ue8m0) {
    const uint32_t b = __ldg(static_cast<const uint8_t*>(base) + i);
    return b == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(b << 23);
  }
  return __ldg(static_cast<const float*>(base) + i);
}

__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return lo | (hi << 16);
}

template <int EPI, int UE>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_fp8_kernel(const __grid_constant__ CUtensorMap tm_a,
                            const __grid_constant__ CUtensorMap tm_b, const Fp8Dev p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + L8::OFF_B;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L8::OFF_BAR);
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* pfull = bars + 2 * kStages;
  uint64_t* pempty = pfull + 2;
  uint64_t* fin = pempty + 2;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + L8::OFF_MISC);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + L8::OFF_MISC + 4);
  volatile int* s_pok = reinterpret_cast<volatile int*>(smem + L8::OFF_MISC + 8);  // [2]
  float* s_amax = reinterpret_cast<float*>(smem + L8::OFF_AMAX);
  int* s_off = reinterpret_cast<int*>(smem + L8::OFF_OFF);
  int* s_pref = reinterpret_cast<int*>(smem + L8::OFF_PREF);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = p.E;
  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&pfull[b]), 1);
      mbar_init(smem_u32(&pempty[b]), kEpiWarps);
    }
    mbar_init(smem_u32(fin), 1);
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_a);
    tma_prefetch_desc(&tm_b);
  }
  if (warp == 1) tmem_alloc(smem_u32(s_tmem), kTmemCols);
  // everything above touched only this CTA's shared memory, TMEM and the
  // kernel parameters; the previous kernel's outputs are read from here on
  pdl_wait();
  for (int i = threadIdx.x; i <= E; i += kThreads) {
    s_off[i] = p.offsets[i];
    s_pref[i] = p.tile_pref[i];
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;

  const int NT = (EPI == EPI_SWIGLU_Q) ? p.I / 128 : p.H / BN;
  const int total = s_pref[E] * NT;
  const int KB = p.K / BK;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------- producer
      int stage = 0;
      uint32_t ph = 0, issued = 0, last_par = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        int e, m, n;
        decode_tile8(tile, NT, E, s_pref, p.group, p.phases, e, m, n);
        const int arow = s_off[e] + m * BM;
        // gate/up: feature n*128 in the [2E, I, H] view; down: the first of
        // the tile's 256 rows of W_down[e]
        const int brow = (EPI == EPI_SWIGLU_Q) ? n * 128 : e * p.H + n * BN;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait_bounded<true>(smem_u32(&empty[stage]), ph ^ 1u, s_abort, p.err,
                                 ERR_TIMEOUT_PRODUCER)) {
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(&full[stage]);
          mbar_arrive_expect_tx(fb, L8::STAGE_TX);
          const uint32_t a_dst = smem_u32(sA + stage * L8::A_BYTES);
          const uint32_t b_dst = smem_u32(sB + stage * L8::B_BYTES);
          tma_load_2d(&tm_a, fb, a_dst, kb * BK, arow);
          if (EPI == EPI_SWIGLU_Q)  // 128 gate rows, then their up rows: one 3-D box
            tma_load_3d(&tm_b, fb, b_dst, kb * BK, brow, 2 * e);
          else                      // 256 rows of W_down[e]: one box
            tma_load_2d(&tm_b, fb, b_dst, kb * BK, brow);
          issued |= 1u << stage;
          last_par = (last_par & ~(1u << stage)) | (ph << stage);
          if (++stage == kStages) {
            stage = 0;
            ph ^= 1u;
          }
        }
      }
      for (int s = 0; s < kStages; ++s) {
        if ((issued >> s) & 1u) {
          volatile int no_abort = 0;
          mbar_wait_bounded<true>(smem_u32(&full[s]), (last_par >> s) & 1u, &no_abort, p.err,
                            ERR_TIMEOUT_PRODUCER, 20000000ull);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------- MMA issuer
      const uint32_t idesc = idesc_e4m3_f32(BM, BN);
      int stage = 0;
      uint32_t ph = 0;
      uint32_t g = 0;  // K-blocks issued so far (selects the partial buffer)
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        for (int kb = 0; kb < KB; ++kb, ++g) {
          const int b = g & 1;
          const uint32_t bph = (g >> 1) & 1;
          if (!mbar_wait_bounded<true>(smem_u32(&pempty[b]), bph ^ 1u, s_abort, p.err, ERR_TIMEOUT_MMA) ||
              !mbar_wait_bounded<true>(smem_u32(&full[stage]), ph, s_abort, p.err, ERR_TIMEOUT_MMA)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d = tmem + b * kBufCols;
          const uint64_t ad = sdesc_k_sw128(smem_u32(sA + stage * L8::A_BYTES));
          const uint64_t bd = sdesc_k_sw128(smem_u32(sB + stage * L8::B_BYTES));
#pragma unroll
          for (int kk = 0; kk < BK / 32; ++kk)
            umma_f8(d, ad + 2 * kk, bd + 2 * kk, idesc, kk != 0 ? 1u : 0u);
          umma_commit(smem_u32(&empty[stage]));
          umma_commit(smem_u32(&pfull[b]));
          if (++stage == kStages) {
            stage = 0;
            ph ^= 1u;
          }
        }
      }
      if (g > 0) {
        umma_commit(smem_u32(fin));
        volatile int no_abort = 0;
        mbar_wait_bounded<true>(smem_u32(fin), 0, &no_abort, p.err, ERR_TIMEOUT_MMA);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int wg = (warp - 2) >> 2;  // warpgroup 0..kEpiGroups-1
    const int q = warp & 3;          // TMEM lane quarter
    const int r = q * 32 + lane;
    const int KBn = p.K / 128;
    uint32_t g = 0;
    uint32_t amax_phase = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
      int e, m, n;
      decode_tile8(tile, NT, E, s_pref, p.group, p.phases, e, m, n);
      const int m_e = s_off[e + 1] - s_off[e];
      const bool valid = m * BM + r < m_e;
      const long R = static_cast<long>(s_off[e]) + m * BM + r;
      // weight block rows feeding this warpgroup's columns
      long wrow0, wrow1;
      int col0, col1;  // partial-sum columns of acc0 / acc1
      if (EPI == EPI_SWIGLU_Q) {
        wrow0 = static_cast<long>(e) * (2 * p.I / 128) + n;              // gate block row
        wrow1 = static_cast<long>(e) * (2 * p.I / 128) + p.I / 128 + n;  // up block row
        col0 = 32 * wg;
        col1 = 128 + 32 * wg;
      } else {
        wrow0 = static_cast<long>(e) * (p.H / 128) + 2 * n + (kGroupCols * wg) / 128;
        wrow1 = wrow0;
        col0 = kGroupCols * wg;
        col1 = col0 + 32;
      }
      float acc0[32], acc1[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) acc0[i] = acc1[i] = 0.f;
      // Scales of K-block kb + 1 are loaded while K-block kb is promoted:
      // the row's activation scale and the weight-block scales (one address
      // across the warp, a broadcast load).
      const long a_base = R * scale_stride(KBn);
      const long w0_base = wrow0 * KBn, w1_base = wrow1 * KBn;
      float sa = valid ? load_scale(p.a_scale, a_base, UE) : 0.f;
      float sw0 = load_scale(p.w_scale, w0_base, UE);
      float sw1 = (EPI == EPI_SWIGLU_Q) ? load_scale(p.w_scale, w1_base, UE) : sw0;
      for (int kb = 0; kb < KB; ++kb) {
        const float s0 = sa * sw0;
        const float s1 = (EPI == EPI_SWIGLU_Q) ? sa * sw1 : s0;
        if (kb + 1 < KB) {
          sa = valid ? load_scale(p.a_scale, a_base + kb + 1, UE) : 0.f;
          sw0 = load_scale(p.w_scale, w0_base + kb + 1, UE);
          if (EPI == EPI_SWIGLU_Q) sw1 = load_scale(p.w_scale, w1_base + kb + 1, UE);
        }
        const int b = g & 1;
        // One thread waits for the partial sums and publishes the outcome in
        // this K-block's slot; the other epilogue warps block on a named
        // barrier instead of polling the mbarrier, and all of them take the
        // same decision (the slot is rewritten only after every warp has
        // passed the next barrier, so no reader sees a later value).
        if (warp == 2 && lane == 0)
          s_pok[b] = mbar_wait_bounded(smem_u32(&pfull[b]), (g >> 1) & 1, s_abort, p.err,
                                       ERR_TIMEOUT_EPILOGUE) ? 1 : 0;
        named_bar_sync(1, kEpiWarps * 32);
        if (!s_pok[b]) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t tb = tmem + b * kBufCols + (static_cast<uint32_t>(q * 32) << 16);
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          uint32_t v0[8], v1[8];
          tmem_ld_32x32b_x8(tb + col0 + 8 * h, v0);
          tmem_ld_32x32b_x8(tb + col1 + 8 * h, v1);
          tmem_ld_wait_x8x2(v0, v1);
          if (h == 3) {  // buffer fully read: the MMA may reuse it
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&pempty[b]));
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            acc0[8 * h + i] = fmaf(__uint_as_float(v0[i]), s0, acc0[8 * h + i]);
            acc1[8 * h + i] = fmaf(__uint_as_float(v1[i]), s1, acc1[8 * h + i]);
          }
        }
        ++g;
      }
      if (!ok) break;

      if (EPI == EPI_SWIGLU_Q) {
        // h = silu(g) * u over this warpgroup's 32 columns; the 1x128 block is
        // the tile's 128 columns, shared by the four warpgroups.
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          acc0[i] = gate_act(acc0[i], p.act) * acc1[i];
          amax = fmaxf(amax, fabsf(acc0[i]));
        }
        float* am = s_amax + (amax_phase ? kEpiGroups * 128 : 0);   // double-buffered by tile
        am[wg * 128 + r] = amax;
        // every epilogue warp reaches this barrier: their only exits are the
        // K-block decisions above, which all of them take together
        named_bar_sync(1, kEpiWarps * 32);
        amax = am[r];
#pragma unroll
        for (int j = 1; j < kEpiGroups; ++j) amax = fmaxf(amax, am[j * 128 + r]);
        amax_phase ^= 1u;
        // scale as in the weight quantiser: amax/448 or its power-of-two ceiling
        float sc = 1.0f;
        uint32_t stored = UE ? 127u : __float_as_uint(1.0f);
        if (amax != 0.f) {
          const float qv = amax / 448.0f;
          if (!UE) {
            sc = qv;
            stored = __float_as_uint(qv);
          } else {
            const uint32_t bits = __float_as_uint(qv);
            int bexp = static_cast<int>((bits >> 23) & 0xFFu) + ((bits & 0x7FFFFFu) ? 1 : 0);
            bexp = bexp > 254 ? 254 : bexp;
            stored = static_cast<uint32_t>(bexp);
            sc = bexp == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(stored << 23);
          }
        }
        const float inv = 1.0f / sc;
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(p.hq + R * p.I + n * 128 + 32 * wg);
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            uint32_t w4[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) {
              const int i = 16 * j + 4 * t;
              w4[t] = e4m3x4(acc0[i] * inv, acc0[i + 1] * inv, acc0[i + 2] * inv, acc0[i + 3] * inv);
            }
            dst[j] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
          }
          if (wg == 0) {
            const long si = R * scale_stride(p.I / 128) + n;
            if (UE) static_cast<uint8_t*>(p.hs)[si] = static_cast<uint8_t>(stored);
            else static_cast<uint32_t*>(p.hs)[si] = stored;
          }
        }
      } else {
        if (valid) {
          const int f = __ldg(p.sorted_f + R);
          const int tok = f / p.k;
          const float wgt = __ldg(p.topk_w + f);
          float* orow = p.out32 + static_cast<long>(tok) * p.H + n * BN + col0;
          if (p.l2_hints & 1) {
            const uint64_t pol = l2_policy_evict_last();
#pragma unroll
            for (int j = 0; j < 8; ++j)
              red_add_v4_hint(orow + 4 * j, wgt * acc0[4 * j], wgt * acc0[4 * j + 1],
                              wgt * acc0[4 * j + 2], wgt * acc0[4 * j + 3], pol);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              red_add_v4_hint(orow + 32 + 4 * j, wgt * acc1[4 * j], wgt * acc1[4 * j + 1],
                              wgt * acc1[4 * j + 2], wgt * acc1[4 * j + 3], pol);
          } else {
#pragma unroll
            for (int j = 0; j < 8; ++j)
              red_add_v4(orow + 4 * j, wgt * acc0[4 * j], wgt * acc0[4 * j + 1],
                         wgt * acc0[4 * j + 2], wgt * acc0[4 * j + 3]);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              red_add_v4(orow + 32 + 4 * j, wgt * acc1[4 * j], wgt * acc1[4 * j + 1],
                         wgt * acc1[4 * j + 2], wgt * acc1[4 * j + 3]);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

template <int EPI>
cudaError_t launch_fp8_impl(const GroupedGemmFp8Args& a, cudaStream_t s) {
  auto kern = a.ue8m0 ? grouped_gemm_fp8_kernel<EPI, 1> : grouped_gemm_fp8_kernel<EPI, 0>;
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  // one flag per device; any host thread may launch, so the flags are atomic
  // (setting the attribute twice is harmless, reading a torn flag is not)
  static std::atomic<bool> attr_set[2][64] = {};
  std::atomic<bool>* flag = &attr_set[a.ue8m0 ? 1 : 0][dev < 64 ? dev : 0];
  if (dev >= 64 || !flag->load(std::memory_order_acquire)) {
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L8::SMEM);
    if (err != cudaSuccess) return err;
    if (dev < 64) flag->store(true, std::memory_order_release);
  }
  Fp8Dev p;
  p.offsets = a.offsets;
  p.tile_pref = a.tile_pref;
  p.E = a.E;
  p.K = a.K;
  p.I = a.I;
  p.H = a.H;
  p.k = a.k;
  p.n_rows = a.n_rows;
  p.err = a.err;
  p.a_scale = a.a_scale;
  p.w_scale = a.w_scale;
  p.ue8m0 = a.ue8m0 ? 1 : 0;
  p.hq = static_cast<uint8_t*>(a.hq);
  p.hs = a.hs;
  p.out32 = a.out32;
  p.sorted_f = a.sorted_f;
  p.topk_w = a.topk_w;
  p.act = a.act;
  p.group = a.tile_group;
  p.phases = a.phases > 0 ? a.phases : 1;
  p.l2_hints = a.l2_hints;
  launch_pdl(kern, a.num_sms, kThreads, L8::SMEM, s, *a.tm_a, *a.tm_b, p);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm1_fp8(const GroupedGemmFp8Args& a, cudaStream_t s) {
  return launch_fp8_impl<EPI_SWIGLU_Q>(a, s);
}

cudaError_t launch_gemm2_fp8(const GroupedGemmFp8Args& a, cudaStream_t s) {
  return launch_fp8_impl<EPI_COMBINE>(a, s);
}

}  // namespace moe
