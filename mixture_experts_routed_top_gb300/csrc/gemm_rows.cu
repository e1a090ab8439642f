// Grouped tensor-core GEMMs (bf16), token-row orientation, for experts with
// many routed rows (prefill).  The swap-AB kernel in gemm_swap.cu covers
// experts with few rows.
//
// Rows of the activation matrix are expert-contiguous (the dispatch step);
// expert e owns rows [offsets[e], offsets[e+1]).  The work is cut into tiles
// of 128 rows x BN output columns; tile t maps to (expert, m-tile, n-tile)
// through the per-expert prefix of m-tile counts, m varying fastest so that
// CTAs running at the same time share one weight tile through L2.
//
// One persistent CTA per SM, six warps:
//   warp 0     TMA producer: A (activations) and B (weights) K-blocks of 64
//              elements into a 4-stage shared-memory ring, 128-byte swizzle
//   warp 1     TMEM allocator and MMA issuer: tcgen05.mma kind::f16,
//              M=128, N=BN, K=16 per instruction, fp32 accumulators in TMEM,
//              two accumulator buffers of 256 columns
//   warps 2-5  epilogue: tcgen05.ld of the accumulator, thread = tile row
//     gate/up GEMM:  B tile = 128 gate rows then the matching 128 up rows of
//                    W_gate_up[e], so accumulator column j is gate and j+128
//                    is up; h = act(gate) * up stored as bf16 (act: silu,
//                    exact GELU or relu, uniform over the launch)
//     down GEMM:     y scaled by the row's routing weight and added (fp32
//                    vector reductions) into out32[token] - the combine
// Every mbarrier wait is bounded; on expiry the kernel flags the error word,
// lets the other roles drain, frees its TMEM and returns.
#include <atomic>

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int BM = 128;

constexpr int kThreads = 192;
constexpr int kTmemCols = 512;
constexpr int kAccCols = 256;

enum { EPI_SWIGLU = 0, EPI_COMBINE = 1 };

static_assert(kRowsBK == 64 || kRowsBK == 32, "K-block must be 64 or 32 bf16");

// BK = bf16 elements per K-block: 64 (128-byte rows, 128-byte swizzle,
// 4 stages of 48 KB) or 32 (64-byte rows, 64-byte swizzle, 9 stages of
// 24 KB: the same shared memory holds more K-blocks in flight).
template <int BN, int BK>
struct Layout {
  static constexpr int kStages = BK == 64 ? 4 : (BN == 256 ? 9 : 12);
  static constexpr int kBoxBytes = 128 * BK * 2;  // one 128-row TMA box
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE_TX = A_BYTES + B_BYTES;
  static constexpr int OFF_B = kStages * A_BYTES;
  static constexpr int OFF_BAR = OFF_B + kStages * B_BYTES;
  static constexpr int NBARS = 2 * kStages + 2 + 2 + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBARS * 8;      // tmem base, abort flag
  static constexpr int OFF_OFF = OFF_MISC + 16;
  static constexpr int OFF_PREF = OFF_OFF + (kMaxE + 1) * 4;
  static constexpr int BYTES = OFF_PREF + (kMaxE + 1) * 4;
  static constexpr int SMEM = BYTES + 1024;                 // alignment slack
};

struct GemmDev {
  const int* offsets;
  const int* tile_pref;
  int E, K, I, H, k;
  int* err;
  __nv_bfloat16* h_out;
  float* out32;
  const int* sorted_f;
  const float* topk_w;
  int act;             // moe_activation of the gate/up epilogue
  int group;           // m-tiles per tile group (0: all of the expert's)
};

// Tile -> (expert e, m-tile m, n-tile n).  Inside an expert the m-tiles run
// in groups of `group`: a group's tiles for every n-tile, m fastest, then
// the next group.  So CTAs running together share a weight tile through L2
// (m fastest), and an expert with many m-tiles re-reads only one group's
// activation tiles per n-tile instead of all of them.
__device__ __forceinline__ void decode_tile(int tile, int NT, int E, const int* s_pref,
                                            int group, int& e, int& m, int& n) {
  const int v = tile / NT;
  int lo = 0, hi = E;
  while (lo < hi) {  // largest e with s_pref[e] <= v
    const int mid = (lo + hi + 1) >> 1;
    if (s_pref[mid] <= v) lo = mid;
    else hi = mid - 1;
  }
  e = lo;
  const int mt = s_pref[e + 1] - s_pref[e];
  const int local = tile - s_pref[e] * NT;
  const int G = (group > 0 && group < mt) ? group : mt;
  const int g = local / (G * NT);
  const int gg = min(G, mt - g * G);      // m-tiles in this group
  const int r = local - g * G * NT;
  n = r / gg;
  m = g * G + (r - n * gg);
}

template <int EPI, int BN, int BK>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_rows_kernel(const __grid_constant__ CUtensorMap tm_a,
                             const __grid_constant__ CUtensorMap tm_b, const GemmDev p) {
  using L = Layout<BN, BK>;
  constexpr int kStages = L::kStages;
  constexpr int kBoxBytes = L::kBoxBytes;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + L::OFF_B;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* tfull = bars + 2 * kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* fin = tempty + 2;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 4);
  int* s_off = reinterpret_cast<int*>(smem + L::OFF_OFF);
  int* s_pref = reinterpret_cast<int*>(smem + L::OFF_PREF);

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

  const int NT = (EPI == EPI_SWIGLU) ? p.I / 128 : p.H / BN;
  const int total = s_pref[E] * NT;
  const int KB = p.K / BK;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------- producer
      int stage = 0;
      uint32_t ph = 0;
      uint32_t issued = 0, last_par = 0;  // per-stage bit sets for the final drain
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        int e, m, n;
        decode_tile(tile, NT, E, s_pref, p.group, e, m, n);
        const int arow = s_off[e] + m * BM;
        // gate/up: feature n*128 in the [2E, I, H] view of the weights; down:
        // the first W_down row of the n-tile
        const int brow = (EPI == EPI_SWIGLU) ? n * 128 : e * p.H + n * BN;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait_bounded<true>(smem_u32(&empty[stage]), ph ^ 1u, s_abort, p.err,
                                 ERR_TIMEOUT_PRODUCER)) {
            ok = false;
            break;
          }
          const uint32_t fb = smem_u32(&full[stage]);
          mbar_arrive_expect_tx(fb, L::STAGE_TX);
          const uint32_t a_dst = smem_u32(sA + stage * L::A_BYTES);
          const uint32_t b_dst = smem_u32(sB + stage * L::B_BYTES);
          tma_load_2d(&tm_a, fb, a_dst, kb * BK, arow);
          if (EPI == EPI_SWIGLU) {  // 128 gate rows, then their up rows: one 3-D box
            tma_load_3d(&tm_b, fb, b_dst, kb * BK, brow, 2 * e);
          } else {
#pragma unroll
            for (int h = 0; h < BN / 128; ++h)
              tma_load_2d(&tm_b, fb, b_dst + h * kBoxBytes, kb * BK, brow + h * 128);
          }
          issued |= 1u << stage;
          last_par = (last_par & ~(1u << stage)) | (ph << stage);
          if (++stage == kStages) {
            stage = 0;
            ph ^= 1u;
          }
        }
      }
      // Drain: every issued load has landed before the CTA may exit.
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
      const uint32_t idesc = idesc_bf16_f32(BM, BN);
      int stage = 0;
      uint32_t ph = 0;
      int it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x, ++it) {
        const int acc = it & 1;
        const uint32_t aph = (it >> 1) & 1;
        if (!mbar_wait_bounded<true>(smem_u32(&tempty[acc]), aph ^ 1u, s_abort, p.err, ERR_TIMEOUT_MMA))
          break;
        tc_fence_after();
        const uint32_t d = tmem + acc * kAccCols;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait_bounded<true>(smem_u32(&full[stage]), ph, s_abort, p.err, ERR_TIMEOUT_MMA)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(sA + stage * L::A_BYTES);
          const uint32_t sb = smem_u32(sB + stage * L::B_BYTES);
          const uint64_t ad = BK == 64 ? sdesc_k_sw128(sa) : sdesc_k_sw64(sa);
          const uint64_t bd = BK == 64 ? sdesc_k_sw128(sb) : sdesc_k_sw64(sb);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            umma_f16(d, ad + 2 * kk, bd + 2 * kk, idesc, (kb | kk) != 0 ? 1u : 0u);
          umma_commit(smem_u32(&empty[stage]));
          if (++stage == kStages) {
            stage = 0;
            ph ^= 1u;
          }
        }
        if (ok) umma_commit(smem_u32(&tfull[acc]));
      }
      // Every MMA issued by this thread has completed before TMEM is freed.
      if (it > 0) {
        umma_commit(smem_u32(fin));
        volatile int no_abort = 0;
        mbar_wait_bounded<true>(smem_u32(fin), 0, &no_abort, p.err, ERR_TIMEOUT_MMA);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int r = q * 32 + lane;
    int it = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++it) {
      int e, m, n;
      decode_tile(tile, NT, E, s_pref, p.group, e, m, n);
      const int acc = it & 1;
      const uint32_t aph = (it >> 1) & 1;
      int ok = 1;
      if (lane == 0)
        ok = mbar_wait_bounded<true>(smem_u32(&tfull[acc]), aph, s_abort, p.err, ERR_TIMEOUT_EPILOGUE);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const int m_e = s_off[e + 1] - s_off[e];
      const bool valid = m * BM + r < m_e;
      const long R = static_cast<long>(s_off[e]) + m * BM + r;
      const uint32_t tb = tmem + acc * kAccCols + (static_cast<uint32_t>(q * 32) << 16);
      if (EPI == EPI_SWIGLU) {
        __nv_bfloat16* hrow = p.h_out + R * p.I + n * 128;
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t g[32], u[32];
          tmem_ld_32x32b_x32(tb + c * 32, g);
          tmem_ld_32x32b_x32(tb + 128 + c * 32, u);
          tmem_ld_wait();
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float g0 = __uint_as_float(g[2 * i]), g1 = __uint_as_float(g[2 * i + 1]);
            const float u0 = __uint_as_float(u[2 * i]), u1 = __uint_as_float(u[2 * i + 1]);
            pk[i] = pack_bf16x2(gate_act(g0, p.act) * u0, gate_act(g1, p.act) * u1);
          }
          if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(hrow + c * 32);
#pragma unroll
            for (int j = 0; j < 4; ++j)
              dst[j] = make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
          }
        }
      } else {
        int tok = 0;
        float wgt = 0.f;
        if (valid) {
          const int f = __ldg(p.sorted_f + R);
          tok = f / p.k;
          wgt = __ldg(p.topk_w + f);
        }
        float* orow = p.out32 + static_cast<long>(tok) * p.H + n * BN;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tb + c * 32, v);
          tmem_ld_wait();
          if (valid) {
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              red_add_v4(orow + c * 32 + 4 * j, wgt * __uint_as_float(v[4 * j]),
                         wgt * __uint_as_float(v[4 * j + 1]), wgt * __uint_as_float(v[4 * j + 2]),
                         wgt * __uint_as_float(v[4 * j + 3]));
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&tempty[acc]));
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

template <int EPI, int BN>
cudaError_t launch_impl(const GroupedGemmArgs& a, cudaStream_t s) {
  using L = Layout<BN, kRowsBK>;
  auto kern = grouped_gemm_rows_kernel<EPI, BN, kRowsBK>;
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  // one flag per device; any host thread may launch, so the flags are atomic
  // (setting the attribute twice is harmless, reading a torn flag is not)
  static std::atomic<bool> attr_set[64] = {};
  if (dev < 64 && !attr_set[dev].load(std::memory_order_acquire)) {
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM);
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
  p.group = a.tile_group;
  launch_pdl(kern, a.num_sms, kThreads, L::SMEM, s, *a.tm_a, *a.tm_b, p);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace

// tm_a: activations (box 128 rows), tm_b: weights (box 128 rows),
// tile_pref: prefix of ceil(M_e / 128).
cudaError_t launch_gemm1_bf16_rows(const GroupedGemmArgs& a, cudaStream_t s) {
  return launch_impl<EPI_SWIGLU, 256>(a, s);
}

cudaError_t launch_gemm2_bf16_rows(const GroupedGemmArgs& a, cudaStream_t s) {
  if (a.H % 256 == 0) return launch_impl<EPI_COMBINE, 256>(a, s);
  return launch_impl<EPI_COMBINE, 128>(a, s);
}

}  // namespace moe
