// Grouped tensor-core GEMMs (bf16), swap-AB orientation, for experts with
// few routed rows (decode-sized batches; prefill runs on the token-row
// kernel in gemm_rows.cu or on CTA pairs in gemm_pair.cu).
//
// The expert's weight rows are the MMA's M side and its tokens the N side,
// D[f, t] = W[f, :] . X[t, :].  A tile is (expert e, feature block fb,
// token tile j): two 128-row weight boxes (256 weight rows) against up to 128
// of the expert's tokens.  An expert's M_e rows are split into
// ceil(M_e / 128) token tiles of near-equal size and N is that size rounded
// up to 16, so a handful of rows costs a 16-wide MMA instead of a 128-row
// tile.  Per 64-wide K block a CTA loads 32 KB of weights and at most 16 KB
// of tokens; with few tokens the kernel is a weight stream.
//
// Gate/up GEMM: box 0 = 128 gate rows, box 1 = the same 128 features' up
//   rows; accumulators D0 (gate) and D1 (up) share TMEM lanes, so lane f
//   holds gate and up of feature f: h[t, f] = act(D0[f,t]) * D1[f,t] (act:
//   silu, exact GELU or relu, uniform over the launch).
// Down GEMM: boxes = 256 (or 128) consecutive rows of W_down[e]; the
//   epilogue adds topk_w * D[f, t] into the fp32 accumulator row of the
//   token (fp32 reductions, coalesced across the warp's 32 features).
//
// One persistent CTA per SM, six warps: warp 0 TMA producer (4-stage ring of
// 48 KB),
// warp 1 TMEM allocator + MMA issuer (tcgen05.mma kind::f16, M=128,
// N=16..128, K=16; two accumulator buffers of 256 columns: D0 at +0, D1 at
// +128), warps 2-5 epilogue (tcgen05.ld 32x32b, thread = feature).  Tiles
// run in (expert, feature block, token tile) order.  Every mbarrier wait is
// bounded.
#include <atomic>

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int BK = 64;               // bf16 elements per 128-byte swizzled row
constexpr int kStages = 4;
constexpr int kThreads = 192;
constexpr int kTmemCols = 512;
constexpr int kBufCols = 256;        // accumulator buffer: D0 at +0, D1 at +128
constexpr int kD1 = 128;
constexpr int kMaxN = 128;
constexpr int A_BOX = 128 * BK * 2;  // 128 weight rows
constexpr int B_BOX = 64 * BK * 2;   // 64 token rows
constexpr int A_BYTES = 2 * A_BOX;
constexpr int B_BYTES = 2 * B_BOX;

constexpr int OFF_B = kStages * A_BYTES;
constexpr int OFF_BAR = OFF_B + kStages * B_BYTES;
constexpr int NBARS = 2 * kStages + 4 + 1;
constexpr int OFF_MISC = OFF_BAR + NBARS * 8;
constexpr int OFF_OFF = OFF_MISC + 16;
constexpr int OFF_PREF = OFF_OFF + (kMaxE + 1) * 4;
constexpr int SMEM_BYTES = OFF_PREF + (kMaxE + 1) * 4 + 1024;

enum { EPI_SWIGLU = 0, EPI_COMBINE = 1 };

struct GemmDev {
  const int* offsets;
  const int* tile_pref;  // prefix of ceil(M_e / 128)
  int E, K, I, H, k;
  int* err;
  __nv_bfloat16* h_out;
  float* out32;
  const int* sorted_f;
  const float* topk_w;
  int act;               // moe_activation of the gate/up epilogue
  int phases;            // feature-block slices run one after the other (>= 1)
  int l2_hints;          // down: bit 0 accumulator evict_last, bit 1 weights evict_first
};

struct Tile {
  int e, fb, t0, size;
};

// Tile -> (expert, feature block, token tile).  With phases > 1 the feature
// blocks are cut into `phases` equal slices that run one after the other
// (every expert's tiles of slice 0, then of slice 1, ...), so the down GEMM's
// combine only touches a T x H/phases slice of the fp32 accumulator at a
// time; inside a slice the order is expert, feature block, token tile.
__device__ __forceinline__ Tile decode_tile(int tile, int NFT, int E, const int* s_off,
                                            const int* s_pref, int phases) {
  const int nfp = NFT / phases;
  const int per_phase = s_pref[E] * nfp;
  const int ph = tile / per_phase;
  tile -= ph * per_phase;
  NFT = nfp;
  const int v = tile / NFT;
  int lo = 0, hi = E;
  while (lo < hi) {  // largest e with s_pref[e] <= v
    const int mid = (lo + hi + 1) >> 1;
    if (s_pref[mid] <= v) lo = mid;
    else hi = mid - 1;
  }
  Tile t;
  t.e = lo;
  const int ntt = s_pref[lo + 1] - s_pref[lo];
  const int local = tile - s_pref[lo] * NFT;
  t.fb = ph * nfp + local / ntt;
  const int j = local - (local / ntt) * ntt;
  const int M = s_off[lo + 1] - s_off[lo];
  const int b = static_cast<int>(static_cast<long>(j) * M / ntt);      // sizes differ by <= 1
  const int en = static_cast<int>(static_cast<long>(j + 1) * M / ntt);
  t.t0 = s_off[lo] + b;
  t.size = en - b;
  return t;
}

template <int EPI, int NA>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_swap_kernel(const __grid_constant__ CUtensorMap tm_w,
                           const __grid_constant__ CUtensorMap tm_x, const GemmDev p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + OFF_B;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* tfull = bars + 2 * kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* fin = tempty + 2;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);
  int* s_off = reinterpret_cast<int*>(smem + OFF_OFF);
  int* s_pref = reinterpret_cast<int*>(smem + OFF_PREF);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = p.E;
  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&tfull[a]), 1);
      mbar_init(smem_u32(&tempty[a]), 4);
    }
    mbar_init(smem_u32(fin), 1);
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_w);
    tma_prefetch_desc(&tm_x);
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

  const int NFT = (EPI == EPI_SWIGLU) ? p.I / 128 : p.H / (128 * NA);
  const int total = s_pref[E] * NFT;
  const int KB = p.K / BK;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------- producer
      int stage = 0;
      uint32_t ph = 0, issued = 0, last_par = 0;
      bool ok = true;
      const uint64_t pol_first = l2_policy_evict_first();
      // gate/up: feature fb*128 in the [2E, I, H] view of the weights (one
      // 3-D box: 128 gate rows, then their up rows); down: the first of the
      // tile's 128*NA rows of W_down[e] (one box of 128*NA rows)
      auto weight_row = [&](const Tile& t) {
        return EPI == EPI_SWIGLU ? t.fb * 128 : t.e * p.H + t.fb * 128 * NA;
      };
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        const Tile t = decode_tile(tile, NFT, E, s_off, s_pref, p.phases);
        const int nbox = (t.size + 63) >> 6;
        const uint32_t tx = NA * A_BOX + nbox * B_BOX;
        const int wrow = weight_row(t);
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait_bounded<true>(smem_u32(&empty[stage]), ph ^ 1u, s_abort, p.err,
                                 ERR_TIMEOUT_PRODUCER)) {
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(&full[stage]);
          mbar_arrive_expect_tx(fb, tx);
          const uint32_t a_dst = smem_u32(sA + stage * A_BYTES);
          const uint32_t b_dst = smem_u32(sB + stage * B_BYTES);
          if (EPI == EPI_SWIGLU) tma_load_3d(&tm_w, fb, a_dst, kb * BK, wrow, 2 * t.e);
          else if (p.l2_hints & 2) tma_load_2d_hint(&tm_w, fb, a_dst, kb * BK, wrow, pol_first);
          else tma_load_2d(&tm_w, fb, a_dst, kb * BK, wrow);
          for (int b = 0; b < nbox; ++b)
            tma_load_2d(&tm_x, fb, b_dst + b * B_BOX, kb * BK, t.t0 + 64 * b);
          issued |= 1u << stage;
          last_par = (last_par & ~(1u << stage)) | (ph << stage);
          if (++stage == kStages) {
            stage = 0;
            ph ^= 1u;
          }
        }
      }
      for (int s = 0; s < kStages; ++s) {  // drain: every issued load has landed
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
      int stage = 0;
      uint32_t ph = 0;
      int it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x, ++it) {
        const Tile t = decode_tile(tile, NFT, E, s_off, s_pref, p.phases);
        const int N = (t.size + 15) & ~15;  // <= kMaxN
        const uint32_t idesc = idesc_bf16_f32(128, N);
        const int acc = it & 1;
        if (!mbar_wait_bounded<true>(smem_u32(&tempty[acc]), ((it >> 1) & 1) ^ 1u, s_abort, p.err,
                               ERR_TIMEOUT_MMA))
          break;
        tc_fence_after();
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait_bounded<true>(smem_u32(&full[stage]), ph, s_abort, p.err, ERR_TIMEOUT_MMA)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = sdesc_k_sw128(smem_u32(sA + stage * A_BYTES));
          const uint64_t bd = sdesc_k_sw128(smem_u32(sB + stage * B_BYTES));
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
#pragma unroll
            for (int a = 0; a < NA; ++a)
              umma_f16(tmem + acc * kBufCols + a * kD1, ad + (a * A_BOX >> 4) + 2 * kk,
                       bd + 2 * kk, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          umma_commit(smem_u32(&empty[stage]));
          if (++stage == kStages) {
            stage = 0;
            ph ^= 1u;
          }
        }
        if (ok) umma_commit(smem_u32(&tfull[acc]));
      }
      if (it > 0) {
        umma_commit(smem_u32(fin));
        volatile int no_abort = 0;
        mbar_wait_bounded<true>(smem_u32(fin), 0, &no_abort, p.err, ERR_TIMEOUT_MMA);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;            // TMEM lane quarter this warp may access
    const int f = q * 32 + lane;       // feature row within the 128-row box
    const uint32_t tl = tmem + (static_cast<uint32_t>(q * 32) << 16);
    const uint64_t pol_last = l2_policy_evict_last();
    int it = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++it) {
      const Tile t = decode_tile(tile, NFT, E, s_off, s_pref, p.phases);
      const int acc = it & 1;
      int ok = 1;
      if (lane == 0)
        ok = mbar_wait_bounded<true>(smem_u32(&tfull[acc]), (it >> 1) & 1, s_abort, p.err,
                               ERR_TIMEOUT_EPILOGUE);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const int nch = (t.size + 31) >> 5;
      const uint32_t tb = tl + acc * kBufCols;
      for (int c = 0; c < nch; ++c) {
        uint32_t d0[32], d1[32];
        tmem_ld_32x32b_x32(tb + 32 * c, d0);
        if (NA == 2) tmem_ld_32x32b_x32(tb + kD1 + 32 * c, d1);
        tmem_ld_wait();
        if (c == nch - 1) {  // all columns read: this buffer is free again
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&tempty[acc]));
        }
        const int cnt = min(32, t.size - 32 * c);
        if (EPI == EPI_SWIGLU) {
          __nv_bfloat16* dst = p.h_out + static_cast<long>(t.t0 + 32 * c) * p.I + t.fb * 128 + f;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            if (i < cnt) {
              const float g = __uint_as_float(d0[i]), u = __uint_as_float(d1[i]);
              dst[static_cast<long>(i) * p.I] = __float2bfloat16_rn(gate_act(g, p.act) * u);
            }
          }
        } else {
          int tok_l = 0;
          float w_l = 0.f;
          if (lane < cnt) {
            const int fl = __ldg(p.sorted_f + t.t0 + 32 * c + lane);
            tok_l = fl / p.k;
            w_l = __ldg(p.topk_w + fl);
          }
          const int col = t.fb * 128 * NA + f;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const int tok = __shfl_sync(0xffffffffu, tok_l, i);
            const float w = __shfl_sync(0xffffffffu, w_l, i);
            if (i < cnt) {
              float* orow = p.out32 + static_cast<long>(tok) * p.H + col;
              if (p.l2_hints & 1) {
                red_add_f32_hint(orow, w * __uint_as_float(d0[i]), pol_last);
                if (NA == 2) red_add_f32_hint(orow + 128, w * __uint_as_float(d1[i]), pol_last);
              } else {
                red_add_f32(orow, w * __uint_as_float(d0[i]));
                if (NA == 2) red_add_f32(orow + 128, w * __uint_as_float(d1[i]));
              }
            }
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

template <int EPI, int NA>
cudaError_t launch_impl(const GroupedGemmArgs& a, cudaStream_t s) {
  auto kern = grouped_gemm_swap_kernel<EPI, NA>;
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  // one flag per device; any host thread may launch, so the flags are atomic
  // (setting the attribute twice is harmless, reading a torn flag is not)
  static std::atomic<bool> attr_set[64] = {};
  if (dev < 64 && !attr_set[dev].load(std::memory_order_acquire)) {
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (err != cudaSuccess) return err;
    attr_set[dev].store(true, std::memory_order_release);
  }
  GemmDev p;
  p.offsets = a.offsets;
  p.tile_pref = a.tile_pref;
  p.E = a.E;
  p.K = a.K;
  p.I = a.I;
  p.H = a.H;
  p.k = a.k;
  p.err = a.err;
  p.h_out = static_cast<__nv_bfloat16*>(a.h_out);
  p.out32 = a.out32;
  p.sorted_f = a.sorted_f;
  p.topk_w = a.topk_w;
  p.act = a.act;
  p.phases = a.phases > 0 ? a.phases : 1;
  p.l2_hints = a.l2_hints;
  launch_pdl(kern, a.num_sms, kThreads, SMEM_BYTES, s, *a.tm_a, *a.tm_b, p);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace

// tm_a: weights (gate/up: the [2E, I, H] view with boxes {64, 128, 2};
// down: boxes of 128 * NA rows), tm_b: activations (box 64 rows),
// tile_pref: prefix of ceil(M_e / 128).
cudaError_t launch_gemm1_bf16_swap(const GroupedGemmArgs& a, cudaStream_t s) {
  return launch_impl<EPI_SWIGLU, 2>(a, s);
}

cudaError_t launch_gemm2_bf16_swap(const GroupedGemmArgs& a, cudaStream_t s) {
  if (a.H % 256 == 0) return launch_impl<EPI_COMBINE, 2>(a, s);
  return launch_impl<EPI_COMBINE, 1>(a, s);
}

}  // namespace moe
