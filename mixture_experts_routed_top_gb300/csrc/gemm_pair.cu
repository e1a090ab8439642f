// Grouped tensor-core GEMMs (bf16) on CTA pairs, weight rows as the MMA's M
// side: tcgen05.mma.cta_group::2 with M = 256 weight rows (128 in each CTA
// of a cluster of two) against N <= 256 of one expert's tokens (N/2 token
// rows in each CTA).
//
// Against the one-CTA kernels (gemm_rows.cu, gemm_swap.cu) a pair reads per
// MMA only its own half of each operand from its own shared memory, so the
// operand bytes per multiply-add fall from 3/128 (token rows, M = 128,
// N = 256) or 4/128 (swap-AB, two M = 128 MMAs of N = 128) to 2/128; and
// with tokens on the N side an expert's rows are cut into ceil(M_e / 256)
// near-equal tiles padded to 16 rows, not to 128.
//
// Tile (pair) = (expert e, feature block fb, token tile j).  An expert's M_e
// rows form ceil(M_e / 256) near-equal token tiles; rank 0 holds the first
// N/2 tokens of a tile, rank 1 the rest, and accumulator column c is token c.
// Inside an expert the token tiles run in groups of `group`: every feature
// block of one group (token tile fastest), then the next group.
//
// Gate/up GEMM: fb covers 128 features of I; CTA r loads, as one box of
//   the weights viewed as [2E, I, H], the gate rows of features f0..f0+63
//   and their up rows (f0 = 128 fb + 64 r).  So TMEM lane quarter p (p = 0, 1) holds gate and
//   quarter p+2 up of the same 32 features; the two epilogue warps of such a
//   pair swap half of their columns through shared memory (the gate warp
//   computes h for the first 16 tokens of each 32-column step, the up warp
//   for the other 16) and store h = act(g) * u.
// Down GEMM: fb covers 256 rows of W_down[e] (H % 256 == 0), 128 per CTA;
//   thread = output feature (TMEM lane).  Each 32-token step of a warp goes
//   through a shared-memory transpose to token rows, and the
//   routing-weighted outputs are added into the fp32 accumulator row of each
//   token with 4-wide vector reductions (a lane: 4 consecutive features of
//   one token).  With one scalar reduction and two shuffles per token and
//   lane, the epilogue held the MMA back (its thread waited for a free
//   accumulator 34-43 % of the time) and the pair lost to the one-CTA
//   swap-AB kernel; with the transpose it wins from about 8 routed rows per
//   expert.
//
// Stages cover 128 of K as two 64-wide swizzled slices: one TMA box per
// operand and stage (the weights' [2E, I, K] view and the tokens' [n, K]
// view with the K slice as the outermost coordinate), which halves the TMA
// operations and barrier hand-offs per byte against 64-wide stages.
//
// Roles in each CTA (192 threads): warp 0 TMA producer (3-stage ring of
// 32 KB weights + 32 KB tokens), warp 1 TMEM (512 columns, allocated
// by the pair together) and, on rank 0, the MMA issuer (two 256-column
// accumulator buffers), warps 2-5 epilogue.  Both CTAs' loads complete on
// rank 0's stage barrier; rank 0's commits arrive on the stage-free and
// accumulator-full barriers of both CTAs; both CTAs' epilogues arrive on
// rank 0's accumulator-free barrier.  Every mbarrier wait is bounded.
#include <atomic>

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int BK = 64;                   // bf16 elements per 128-byte swizzled row
constexpr int KA = 2;                    // swizzle atoms (64-wide K slices) per stage
constexpr int kStages = 3;
constexpr int kThreads = 192;
constexpr int kTmemCols = 512;
constexpr int kBufCols = 256;            // one accumulator buffer: N <= 256 columns
constexpr int ATOM = 128 * BK * 2;       // 128 rows x one 64-wide K slice: 16 KB
constexpr int A_BYTES = KA * ATOM;       // this CTA's 128 weight rows, 128 of K
constexpr int B_BYTES = KA * ATOM;       // 128 token rows, 128 of K
constexpr int kXStride = 17;             // floats per exchange row: 16 values + 1 (no bank conflicts)
constexpr int kXBuf = 32 * kXStride;     // floats: one direction, one warp pair, one parity
constexpr int kTempty = 8;               // epilogue warps of both CTAs

constexpr int OFF_B = kStages * A_BYTES;
constexpr int OFF_X = OFF_B + kStages * B_BYTES;
constexpr int OFF_OK = OFF_X + 8 * kXBuf * 4;          // int [2 warp pairs][2 parities][2 warps]
constexpr int OFF_BAR = OFF_OK + 64;
constexpr int NBARS = 2 * kStages + 2 + 2 + 1;
constexpr int OFF_MISC = OFF_BAR + NBARS * 8;          // TMEM base, abort flag
constexpr int OFF_OFF = OFF_MISC + 16;
constexpr int OFF_PREF = OFF_OFF + (kMaxE + 1) * 4;
constexpr int OFF_HEAVY = OFF_PREF + (kMaxE + 1) * 4;
constexpr int SMEM_BYTES = OFF_HEAVY + (kMaxE + 1) * 4 + 1024;
constexpr int kHeavyTiles = 2;           // experts with more token tiles than this are "heavy"
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");

enum { EPI_SWIGLU = 0, EPI_COMBINE = 1 };

struct PairDev {
  const int* offsets;
  int E, K, I, H, k;
  int* err;
  __nv_bfloat16* h_out;
  float* out32;
  const int* sorted_f;
  const float* topk_w;
  int act;
  int group;             // token tiles per tile group (0: all of the expert's)
  int l2_hints;          // down: bit 0 accumulator evict_last
  int phases;            // down: feature-block slices run one after the other (>= 1)
  int interleave;        // heavy experts' tiles spread over the light ones' (one phase)
};

struct Tile {
  int e, fb, t0, size;
};

// Tile -> (expert, feature block, token tile); s_pref = prefix of the
// experts' token-tile counts ceil(M_e / 256).  With phases > 1 the feature
// blocks are cut into `phases` equal slices run one after the other (every
// expert's tiles of slice 0, then of slice 1, ...), so the down GEMM's
// combine touches a [T, H / phases] slice of the fp32 accumulator at a time.
//
// With s_heavy (gate/up, one phase) the order interleaves two classes of
// experts: those with more than kHeavyTiles token tiles (s_heavy = their
// prefix, the others counting 0) and the rest.  The heavy experts' tiles
// are spread evenly over the sequence (position k is heavy when
// floor((k+1) TA / total) > floor(k TA / total)), so their compute-bound
// tiles run beside the light experts' weight-streaming ones instead of in
// one block; inside each class the order is as above.
__device__ __forceinline__ Tile decode_tile(int tile, int NFB, int E, const int* s_off,
                                            const int* s_pref, int group, int phases = 1,
                                            const int* s_heavy = nullptr) {
  bool heavy = false;
  if (s_heavy != nullptr) {
    const long TA = static_cast<long>(s_heavy[E]) * NFB;
    const long total = static_cast<long>(s_pref[E]) * NFB;
    const long a0 = static_cast<long>(tile) * TA / total;
    const long a1 = static_cast<long>(tile + 1) * TA / total;
    heavy = a1 > a0;
    tile = heavy ? static_cast<int>(a0) : static_cast<int>(tile - a0);
  }
  // prefix of the token-tile counts of the class decoded
  auto pref = [&](int e) {
    return s_heavy == nullptr ? s_pref[e] : (heavy ? s_heavy[e] : s_pref[e] - s_heavy[e]);
  };
  const int nfp = NFB / phases;
  const int per_phase = pref(E) * nfp;
  const int ph = tile / per_phase;
  tile -= ph * per_phase;
  NFB = nfp;
  const int v = tile / NFB;
  int lo = 0, hi = E;
  while (lo < hi) {  // largest e with pref(e) <= v
    const int mid = (lo + hi + 1) >> 1;
    if (pref(mid) <= v) lo = mid;
    else hi = mid - 1;
  }
  Tile t;
  t.e = lo;
  const int base = pref(lo);
  const int mt = pref(lo + 1) - base;
  const int local = tile - base * NFB;
  const int G = (group > 0 && group < mt) ? group : mt;
  const int g = local / (G * NFB);
  const int gg = min(G, mt - g * G);
  const int r = local - g * G * NFB;
  t.fb = r / gg;
  const int j = g * G + (r - t.fb * gg);
  t.fb += ph * nfp;
  const int M = s_off[lo + 1] - s_off[lo];
  const int b = static_cast<int>(static_cast<long>(j) * M / mt);  // sizes differ by <= 1
  const int en = static_cast<int>(static_cast<long>(j + 1) * M / mt);
  t.t0 = s_off[lo] + b;
  t.size = en - b;
  return t;
}

template <int EPI>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tm_w,
                             const __grid_constant__ CUtensorMap tm_x, const PairDev p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + OFF_B;
  float* sX = reinterpret_cast<float*>(smem + OFF_X);
  volatile int* s_ok = reinterpret_cast<volatile int*>(smem + OFF_OK);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint64_t* full = bars;                 // rank 0: both CTAs' loads of a stage landed
  uint64_t* empty = bars + kStages;      // both: the stage's MMAs are done
  uint64_t* tfull = bars + 2 * kStages;  // both: accumulator buffer complete
  uint64_t* tempty = tfull + 2;          // rank 0: both CTAs drained the buffer
  uint64_t* fin = tempty + 2;            // rank 0: every MMA done
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);
  int* s_off = reinterpret_cast<int*>(smem + OFF_OFF);
  int* s_pref = reinterpret_cast<int*>(smem + OFF_PREF);
  int* s_heavy = reinterpret_cast<int*>(smem + OFF_HEAVY);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank() & 1u;
  const int E = p.E;
  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&tfull[a]), 1);
      mbar_init(smem_u32(&tempty[a]), kTempty);
    }
    mbar_init(smem_u32(fin), 1);
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_w);
    tma_prefetch_desc(&tm_x);
  }
  // both CTAs are running and their barriers initialised before the pair
  // allocates TMEM together or signals the other's barriers
  cluster_sync_all();
  if (warp == 1) tmem_alloc_pair(smem_u32(s_tmem), kTmemCols);
  // everything above touched only the pair's shared memory, TMEM and the
  // kernel parameters; the previous kernel's outputs are read from here on
  pdl_wait();
  for (int i = threadIdx.x; i <= E; i += kThreads) s_off[i] = p.offsets[i];
  __syncthreads();
  if (warp == 0) {  // s_pref: prefix of ceil(M_e / 256), one warp scan per 32 experts
    int carry = 0, carry_h = 0;
    for (int base = 0; base < E; base += 32) {
      const int e = base + lane;
      int x = e < E ? (s_off[e + 1] - s_off[e] + 255) >> 8 : 0;
      int xh = x > kHeavyTiles ? x : 0;   // the heavy experts' share
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, d);
        const int yh = __shfl_up_sync(0xffffffffu, xh, d);
        if (lane >= d) {
          x += y;
          xh += yh;
        }
      }
      if (e < E) {
        s_pref[e + 1] = carry + x;
        s_heavy[e + 1] = carry_h + xh;
      }
      carry += __shfl_sync(0xffffffffu, x, 31);
      carry_h += __shfl_sync(0xffffffffu, xh, 31);
    }
    if (lane == 0) s_pref[0] = s_heavy[0] = 0;
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();   // the pair's TMEM is allocated in both CTAs
  tc_fence_after();
  const uint32_t tmem = *s_tmem;

  const int NFB = (EPI == EPI_SWIGLU) ? p.I / 128 : p.H / 256;
  // interleaved class order: one phase only, and only when both classes exist
  const int* ilv = (p.interleave && p.phases == 1 && s_heavy[E] > 0 && s_heavy[E] < s_pref[E])
                       ? s_heavy : nullptr;
  const int total = s_pref[E] * NFB;
  const int KB = p.K / (KA * BK);          // stages per tile (128 of K each)
  const int cid = blockIdx.x >> 1, ncl = gridDim.x >> 1;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------- producer
      int stage = 0;
      uint32_t ph = 0, issued = 0, last_par = 0;
      bool ok = true;
      for (int tile = cid; ok && tile < total; tile += ncl) {
        const Tile t = decode_tile(tile, NFB, E, s_off, s_pref, p.group, p.phases, ilv);
        const int half = ((t.size + 15) & ~15) >> 1;
        const uint32_t tx = 2u * static_cast<uint32_t>(A_BYTES + B_BYTES);
        // gate/up: feature f0 of expert e in the [2E, I, H] view; down: the
        // first of this CTA's 128 rows of W_down[e]
        int arow[1];
        if (EPI == EPI_SWIGLU) arow[0] = t.fb * 128 + 64 * static_cast<int>(rank);
        else arow[0] = t.e * p.H + t.fb * 256 + 128 * static_cast<int>(rank);
        const int brow = t.t0 + static_cast<int>(rank) * half;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait_bounded<true, true>(smem_u32(&empty[stage]), ph ^ 1u, s_abort, p.err,
                                             ERR_TIMEOUT_PRODUCER)) {
            ok = false;
            break;
          }
          const uint32_t fb_local = smem_u32(&full[stage]);
          if (rank == 0) mbar_arrive_expect_tx(fb_local, tx);
          const uint32_t fb_lead = mapa_shared(fb_local, 0);
          const uint32_t a_dst = smem_u32(sA + stage * A_BYTES);
          const uint32_t b_dst = smem_u32(sB + stage * B_BYTES);
          // one box per operand covers both 64-wide K slices of the stage
          // (the last coordinate counts 64-wide slices along K)
          if (EPI == EPI_SWIGLU)  // gate rows f0..f0+63, then their up rows, per K slice
            tma_load_4d_pair(&tm_w, fb_lead, a_dst, 0, arow[0], 2 * t.e, KA * kb);
          else
            tma_load_3d_pair(&tm_w, fb_lead, a_dst, 0, arow[0], KA * kb);
          tma_load_3d_pair(&tm_x, fb_lead, b_dst, 0, brow, KA * kb);
          issued |= 1u << stage;
          last_par = (last_par & ~(1u << stage)) | (ph << stage);
          if (++stage == kStages) {
            stage = 0;
            ph ^= 1u;
          }
        }
      }
      // drain: rank 0 waits until every issued stage's loads (both CTAs')
      // landed; rank 1 until its last loads of each stage were consumed
      for (int s = 0; s < kStages; ++s) {
        if ((issued >> s) & 1u) {
          volatile int no_abort = 0;
          const uint32_t par = (last_par >> s) & 1u;
          if (rank == 0)
            mbar_wait_bounded<true, true>(smem_u32(&full[s]), par, &no_abort, p.err,
                                          ERR_TIMEOUT_PRODUCER, 20000000ull);
          else
            mbar_wait_bounded<true, true>(smem_u32(&empty[s]), par, &no_abort, p.err,
                                          ERR_TIMEOUT_PRODUCER, 20000000ull);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ---------------------------------------------------------- MMA issuer
      int stage = 0;
      uint32_t ph = 0;
      int it = 0;
      bool ok = true;
      for (int tile = cid; ok && tile < total; tile += ncl, ++it) {
        const Tile t = decode_tile(tile, NFB, E, s_off, s_pref, p.group, p.phases, ilv);
        const int N = (t.size + 15) & ~15;  // <= 256
        const uint32_t idesc = idesc_bf16_f32(256, N);
        const int acc = it & 1;
        if (!mbar_wait_bounded<true, true>(smem_u32(&tempty[acc]), ((it >> 1) & 1) ^ 1u, s_abort,
                                           p.err, ERR_TIMEOUT_MMA))
          break;
        tc_fence_after();
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait_bounded<true, true>(smem_u32(&full[stage]), ph, s_abort, p.err,
                                             ERR_TIMEOUT_MMA)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = sdesc_k_sw128(smem_u32(sA + stage * A_BYTES));
          const uint64_t bd = sdesc_k_sw128(smem_u32(sB + stage * B_BYTES));
#pragma unroll
          for (int kk = 0; kk < KA * BK / 16; ++kk) {
            const uint32_t off = ((kk >> 2) * ATOM >> 4) + 2 * (kk & 3);  // K slice, then 16 of K
            umma_f16_pair(tmem + acc * kBufCols, ad + off, bd + off, idesc,
                          (kb | kk) != 0 ? 1u : 0u);
          }
          umma_commit_pair_both(smem_u32(&empty[stage]));
          if (++stage == kStages) {
            stage = 0;
            ph ^= 1u;
          }
        }
        if (ok) umma_commit_pair_both(smem_u32(&tfull[acc]));
      }
      if (it > 0) {
        umma_commit_pair_local(smem_u32(fin));
        volatile int no_abort = 0;
        mbar_wait_bounded<true, true>(smem_u32(fin), 0, &no_abort, p.err, ERR_TIMEOUT_MMA);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;            // TMEM lane quarter this warp may access
    const uint64_t pol_last = l2_policy_evict_last();
    const uint32_t tl = tmem + (static_cast<uint32_t>(q * 32) << 16);
    const int wp = q & 1;              // warp pair (gate/up): quarters wp and wp+2
    const bool upw = q >= 2;
    const bool odd = lane & 1;
    int it = 0, xs = 0;
    for (int tile = cid; tile < total; tile += ncl, ++it) {
      const Tile t = decode_tile(tile, NFB, E, s_off, s_pref, p.group, p.phases, ilv);
      const int acc = it & 1;
      int ok = 1;
      if (lane == 0)
        ok = mbar_wait_bounded<true, true>(smem_u32(&tfull[acc]), (it >> 1) & 1, s_abort, p.err,
                                           ERR_TIMEOUT_EPILOGUE);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (EPI == EPI_SWIGLU) {
        // the two warps of a pair leave together or not at all: each
        // publishes its wait's outcome and both read the pair's
        volatile int* okp = s_ok + (wp * 2 + (it & 1)) * 2;
        if (lane == 0) okp[upw ? 1 : 0] = ok;
        named_bar_sync(1 + wp, 64);
        ok = okp[0] & okp[1];
      }
      if (!ok) break;
      tc_fence_after();
      const uint32_t tb = tl + acc * kBufCols;
      const int N = (t.size + 15) & ~15;
      const int nst = (N + 31) >> 5;
      auto release = [&]() {  // every column of this buffer read: hand it back
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (rank == 0) mbar_arrive(smem_u32(&tempty[acc]));
          else mbar_arrive_remote(mapa_shared(smem_u32(&tempty[acc]), 0));
        }
      };
      if (EPI == EPI_SWIGLU) {
        const int fcol = t.fb * 128 + 64 * static_cast<int>(rank) + 32 * wp + (lane & ~1);
        for (int s = 0; s < nst; ++s, ++xs) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tb + 32 * s, v);
          tmem_ld_wait();
          if (s == nst - 1) release();
          // gate warp: keeps columns 0..15 of the step, sends 16..31; up
          // warp: sends 0..15, keeps 16..31
          float* snd = sX + ((wp * 2 + (upw ? 1 : 0)) * 2 + (xs & 1)) * kXBuf + lane * kXStride;
          const float* rcv =
              sX + ((wp * 2 + (upw ? 0 : 1)) * 2 + (xs & 1)) * kXBuf + lane * kXStride;
#pragma unroll
          for (int j = 0; j < 16; ++j) snd[j] = __uint_as_float(upw ? v[j] : v[16 + j]);
          named_bar_sync(1 + wp, 64);
          float hv[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float mine = __uint_as_float(upw ? v[16 + j] : v[j]);
            const float g = upw ? rcv[j] : mine, u = upw ? mine : rcv[j];
            hv[j] = gate_act(g, p.act) * u;
          }
          // lane pairs: the even lane stores features (f, f+1) of token
          // c0 + j, the odd lane those of token c0 + j + 1
          const int c0 = 32 * s + (upw ? 16 : 0);
#pragma unroll
          for (int j = 0; j < 16; j += 2) {
            const float r = __shfl_xor_sync(0xffffffffu, odd ? hv[j] : hv[j + 1], 1);
            const int c = c0 + j + (odd ? 1 : 0);
            if (c < t.size)
              *reinterpret_cast<uint32_t*>(p.h_out + static_cast<long>(t.t0 + c) * p.I + fcol) =
                  odd ? pack_bf16x2(r, hv[j + 1]) : pack_bf16x2(hv[j], r);
          }
        }
      } else {
        // Combine: per 32-token step the warp's 32 features x 32 tokens go
        // through a shared-memory transpose (token rows of 32 floats), so a
        // lane adds 4 consecutive features of one token with one vector
        // reduction: 8 of them per step instead of 32 scalar ones.
        float* stg = sX + q * 32 * 32;
        const int col = t.fb * 256 + 128 * static_cast<int>(rank) + 32 * q + 4 * (lane & 7);
        for (int s = 0; s < nst; ++s) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tb + 32 * s, v);
          tmem_ld_wait();
          if (s == nst - 1) release();
          const int cnt = min(32, t.size - 32 * s);
          int tok_l = 0;
          float w_l = 0.f;
          if (lane < cnt) {
            const int fl = __ldg(p.sorted_f + t.t0 + 32 * s + lane);
            tok_l = fl / p.k;
            w_l = __ldg(p.topk_w + fl);
          }
          __syncwarp();  // the previous step's reads of the staging tile are done
#pragma unroll
          for (int i = 0; i < 32; ++i) stg[i * 32 + lane] = __uint_as_float(v[i]);
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int ti = 4 * j + (lane >> 3);  // token of this lane within the step
            const int tok = __shfl_sync(0xffffffffu, tok_l, ti);
            const float w = __shfl_sync(0xffffffffu, w_l, ti);
            if (ti < cnt) {
              const float4 y = *reinterpret_cast<const float4*>(stg + ti * 32 + 4 * (lane & 7));
              float* o = p.out32 + static_cast<long>(tok) * p.H + col;
              if (p.l2_hints & 1) red_add_v4_hint(o, w * y.x, w * y.y, w * y.z, w * y.w, pol_last);
              else red_add_v4(o, w * y.x, w * y.y, w * y.z, w * y.w);
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  // neither CTA leaves while the other may still touch its shared memory
  cluster_sync_all();
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem, kTmemCols);
}

template <int EPI>
cudaError_t launch_impl(const GroupedGemmArgs& a, long tiles_max, cudaStream_t s) {
  auto kern = grouped_gemm_pair_kernel<EPI>;
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev >= 64) return cudaErrorInvalidDevice;
  // per device: the shared-memory attribute, then how many clusters of two
  // fit at once (any host thread may launch, so both are atomic)
  static std::atomic<int> max_clusters[64] = {};
  int nc = max_clusters[dev].load(std::memory_order_acquire);
  if (nc == 0) {
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    err = cudaOccupancyMaxActiveClusters(&nc, kern, &cfg);
    if (err != cudaSuccess) return err;
    if (nc < 1) return cudaErrorLaunchOutOfResources;
    max_clusters[dev].store(nc, std::memory_order_release);
  }
  const int ncl = static_cast<int>(std::min<long>(nc, std::max<long>(tiles_max, 1)));
  PairDev p;
  p.offsets = a.offsets;
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
  p.l2_hints = a.l2_hints;
  p.phases = (EPI == EPI_COMBINE && a.phases > 0) ? a.phases : 1;
  // gate/up: the heavy experts' tiles interleaved with the light ones'
  // (measured 1.7 % faster at DeepSeek-V3 size); down: slower that way
  // (2.06 against 1.96 ms with one phase), and its phases keep it off anyway
  p.interleave = EPI == EPI_SWIGLU ? 1 : 0;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * ncl);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  err = cudaLaunchKernelEx(&cfg, kern, *a.tm_a, *a.tm_b, p);
  count_launches(1);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

}  // namespace

// tm_a: weights (gate/up: the [2E, I, H] view, boxes of 64 gate + 64 up
// rows; down: 128-row boxes), tm_b: activations (128-row boxes), each box
// two 64-wide K slices (maps made by the library's 128-wide-K map builder).
cudaError_t launch_gemm1_bf16_pair(const GroupedGemmArgs& a, long n_rows, cudaStream_t s) {
  return launch_impl<EPI_SWIGLU>(a, (n_rows / 256 + a.E) * (a.I / 128), s);
}

cudaError_t launch_gemm2_bf16_pair(const GroupedGemmArgs& a, long n_rows, cudaStream_t s) {
  return launch_impl<EPI_COMBINE>(a, (n_rows / 256 + a.E) * (a.H / 256), s);
}

}  // namespace moe
