// Block-scaled grouped GEMMs of the routed experts forward, on the tensor
// core's own block scaling (tcgen05.mma kind::mxf8f6f4 with UE8M0 scale
// factors): FP8 experts with UE8M0 scales, and FP4 (e2m1) experts.  The page
// ("FP8 and FP4 quantized experts" section) ties UE8M0 power-of-two scales
// to Blackwell and names FP4 weights packed in int8 with UE8M0 scales; this
// hardware path applies such scales inside the MMA, so no software
// promotion of partial sums is needed.
//
// Operands, token-row orientation (expert-contiguous rows as the MMA's M):
//   A  e4m3 activations [n_rows, K] (the gathered hidden rows, or h), with
//      one 32-bit scale word per row and 128-wide K block holding the four
//      UE8M0 bytes of its 32-wide sub-blocks: a_sf[K/128][n_rows]
//   B  weights [E * Nw, K]: e4m3 with one UE8M0 byte per 128x128 block
//      (FP8), or e2m1 packed two per byte with one UE8M0 byte per 1x32 block
//      along K (FP4); TMA expands e2m1 rows to the one-byte-per-element-slot
//      shared-memory form the MMA reads (16 codes in 8 bytes, then 8 bytes
//      of padding)
// A stage holds one 128-wide K block: A 128 x 128 B, B 256 x 128 B and the
// scale factors of its rows (A) and columns (B), written into shared memory
// by the producer warp in the tensor core's scale-factor tile form (32 rows
// of 16 bytes: byte 4c + j of row i belongs to operand row 32c + i, K
// sub-block j) and copied to TMEM by the MMA thread (tcgen05.cp) ahead of
// the four K = 32 MMAs, whose descriptors select sub-block j.
//
// Roles (persistent, one CTA per SM, 320 threads):
//   warp 0      producer: lane 0 issues the TMA loads of A and B, all lanes
//               gather the stage's scale factors into shared memory
//   warp 1      TMEM allocator (512 columns) and MMA issuer: one 256-column
//               fp32 accumulator (M=128, N=256) at column 0, scale-factor
//               slots of 16 columns per stage from column 256
//   warps 2-9   epilogue, two warps per TMEM lane quarter (thread = tile
//               row, warp half = half of the columns).  The accumulator is
//               read into registers at once and released, so the MMAs of
//               the next tile overlap the rest of the epilogue.
//     gate/up:  tile columns 0..127 are the gate rows of 128 features, 128..
//               255 the matching up rows; h = act(g) * u is quantised to e4m3
//               per row (1x128 blocks for FP8, the two warps of a row
//               exchanging their maxima through shared memory and a bounded
//               mbarrier; 1x32 blocks for FP4) and written with its scale
//               words for the down GEMM
//     down:     y scaled by the routing weight and added into the fp32
//               output row of the token (vector reductions)
// Every mbarrier wait is bounded; on expiry the kernel flags the error word,
// lets the other roles drain, frees its TMEM and returns.
#include <atomic>

#include "moe_device.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 128;                       // K elements per stage: 4 MMAs of K = 32
constexpr int kStages = 4;
constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + kEpiWarps * 32;
constexpr int kTmemCols = 512;
constexpr int kSfCol0 = 256;                  // first scale-factor slot
constexpr int kSfSlotCols = 16;               // A: +0..3, B: +8..15
constexpr int kSfAhead = 3;                   // K blocks the scale-factor loads run ahead

struct LM {
  static constexpr int A_BYTES = BM * BK;                 // 16 KB
  static constexpr int B_BYTES = BN * BK;                 // 32 KB in shared memory
  static constexpr int SF_BYTES = 512 + 1024;             // A tile, two B tiles
  static constexpr int OFF_B = kStages * A_BYTES;
  static constexpr int OFF_SF = OFF_B + kStages * B_BYTES;
  static constexpr int OFF_BAR = OFF_SF + kStages * SF_BYTES;
  static constexpr int NBARS = 2 * kStages + 4;
  static constexpr int OFF_MISC = OFF_BAR + NBARS * 8;    // tmem base, abort flag
  static constexpr int OFF_AMAX = OFF_MISC + 16;          // float [2 tiles][2 halves][128]
  static constexpr int OFF_OFF = OFF_AMAX + 2 * 2 * 128 * 4;
  static constexpr int OFF_PREF = OFF_OFF + (kMaxE + 1) * 4;
  static constexpr int BYTES = OFF_PREF + (kMaxE + 1) * 4;
  static constexpr int SMEM = BYTES + 1024;
};
static_assert(LM::SMEM <= 227 * 1024, "shared memory budget");

enum { EPI_SWIGLU_Q = 0, EPI_COMBINE = 1 };

struct MxDev {
  const int* offsets;
  const int* tile_pref;
  int E, K, I, H, k, n_rows;
  int* err;
  const uint32_t* a_sf;     // [K/128][n_rows] scale words of A
  const uint8_t* w_sf;      // FP8: [E, Nw/128, K/128]; FP4: [E * Nw, K/32]
  uint8_t* hq;              // gate/up: h codes [n_rows, I]
  uint32_t* hs;             // gate/up: h scale words [I/128][n_rows]
  float* out32;             // down: [T, H]
  const int* sorted_f;
  const float* topk_w;
  int act;
  int group;                // m-tiles per tile group (0: all of the expert's)
  int l2_hints;             // down: bit 0 accumulator evict_last, bit 1 weights evict_first
  int phases;               // n-tile slices run one after the other (>= 1)
};

// Tile -> (expert e, m-tile m, n-tile n).  The n-tiles are cut into
// `phases` equal slices run one after the other (the down GEMM's combine
// then touches a T x H/phases slice of the fp32 accumulator at a time).
// Inside a slice and an expert the m-tiles run in groups of `group` (0:
// all): a group's tiles for every n-tile of the slice, m fastest.
__device__ __forceinline__ void decode_tile_mx(int tile, int NT, int E, const int* s_pref,
                                               int group, int phases, int& e, int& m, int& n) {
  const int ntp = NT / phases;
  const int per_phase = s_pref[E] * ntp;
  const int ph = tile / per_phase;
  tile -= ph * per_phase;
  const int v = tile / ntp;
  int lo = 0, hi = E;
  while (lo < hi) {  // largest e with s_pref[e] <= v
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

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  return static_cast<uint32_t>(e4m3x2(a, b)) | (static_cast<uint32_t>(e4m3x2(c, d)) << 16);
}

// UE8M0 scale of a block for e4m3 codes: the smallest power of two >= amax/448
// (amax = 0 gives 1); returns the scale, *b its exponent byte.
__device__ __forceinline__ float ue8m0_block_scale(float amax, uint32_t* b) {
  return block_scale(amax, true, b);
}

// Quantise n consecutive values v[0..n) with scale s into packed e4m3 words.
template <int N>
__device__ __forceinline__ void quant_words(const float* v, float inv, uint32_t* w) {
#pragma unroll
  for (int i = 0; i < N / 4; ++i)
    w[i] = e4m3x4(v[4 * i] * inv, v[4 * i + 1] * inv, v[4 * i + 2] * inv, v[4 * i + 3] * inv);
}

template <int EPI, bool FP4W>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_mx_kernel(const __grid_constant__ CUtensorMap tm_a,
                           const __grid_constant__ CUtensorMap tm_b, const MxDev p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + LM::OFF_B;
  uint8_t* sSF = smem + LM::OFF_SF;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + LM::OFF_BAR);
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* tfull = bars + 2 * kStages;
  uint64_t* tempty = tfull + 1;
  uint64_t* fin = tempty + 1;
  uint64_t* amax_bar = fin + 1;     // FP8 h rows: both halves' maxima are in
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + LM::OFF_MISC);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + LM::OFF_MISC + 4);
  float* s_amax = reinterpret_cast<float*>(smem + LM::OFF_AMAX);
  int* s_off = reinterpret_cast<int*>(smem + LM::OFF_OFF);
  int* s_pref = reinterpret_cast<int*>(smem + LM::OFF_PREF);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = p.E;
  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&full[s]), 2);   // TMA bytes (with their arrive) + scale factors
      mbar_init(smem_u32(&empty[s]), 1);
    }
    mbar_init(smem_u32(tfull), 1);
    mbar_init(smem_u32(tempty), kEpiWarps);
    mbar_init(smem_u32(fin), 1);
    mbar_init(smem_u32(amax_bar), kEpiWarps * 32);
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
  const int Nw = (EPI == EPI_SWIGLU_Q) ? 2 * p.I : p.H;   // weight rows per expert

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // Two cursors walk this CTA's (tile, K block) sequence: `ld` issues the
    // TMA loads of the stage being filled and writes its scale factors into
    // shared memory; `pf` runs kSfAhead iterations ahead and loads the scale
    // factors of its iteration into one of kSfAhead register slots, so no
    // stage waits for a global-memory round trip of its scale factors.
    struct Cursor {
      int tile, kb, arow, brow0, brow1, e, n;
    };
    auto place = [&](Cursor& c) {
      if (c.tile >= total) return;
      int e, m, n;
      decode_tile_mx(c.tile, NT, E, s_pref, p.group, p.phases, e, m, n);
      c.arow = s_off[e] + m * BM;
      c.e = e;
      c.n = n;
      c.brow0 = (EPI == EPI_SWIGLU_Q) ? e * Nw + n * 128 : e * Nw + n * BN;
      c.brow1 = (EPI == EPI_SWIGLU_Q) ? c.brow0 + p.I : c.brow0 + 128;
    };
    auto advance = [&](Cursor& c) {
      if (++c.kb == KB) {
        c.kb = 0;
        c.tile += gridDim.x;
        place(c);
      }
    };
    // scale factors of one K block: A words of rows 32c + lane (c < 4), then
    // B words (FP4: rows 32c + lane of each 128-row box; FP8: the two boxes'
    // block exponents)
    auto load_sf = [&](const Cursor& c, uint32_t (&sa)[4], uint32_t (&sb)[8]) {
      if (c.tile >= total) return;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int R = c.arow + 32 * q + lane;
        sa[q] = R < p.n_rows ? __ldg(p.a_sf + static_cast<long>(c.kb) * p.n_rows + R) : 0x7F7F7F7Fu;
      }
      if (FP4W) {
        const int kw = p.K / 32;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const long row0 = (h == 0 ? c.brow0 : c.brow1) + lane;
#pragma unroll
          for (int q = 0; q < 4; ++q)
            sb[4 * h + q] =
                __ldg(reinterpret_cast<const uint32_t*>(p.w_sf + (row0 + 32 * q) * kw) + c.kb);
        }
      } else {
        sb[0] = __ldg(p.w_sf + (static_cast<long>(c.brow0) / 128) * KB + c.kb);
        sb[1] = __ldg(p.w_sf + (static_cast<long>(c.brow1) / 128) * KB + c.kb);
      }
    };
    auto store_sf = [&](uint32_t sf, const uint32_t (&sa)[4], const uint32_t (&sb)[8]) {
      st_shared_v4(sf + 16 * lane, sa[0], sa[1], sa[2], sa[3]);
      if (FP4W) {
        st_shared_v4(sf + 512 + 16 * lane, sb[0], sb[1], sb[2], sb[3]);
        st_shared_v4(sf + 1024 + 16 * lane, sb[4], sb[5], sb[6], sb[7]);
      } else {
        const uint32_t s0 = sb[0] * 0x01010101u, s1 = sb[1] * 0x01010101u;
        st_shared_v4(sf + 512 + 16 * lane, s0, s0, s0, s0);
        st_shared_v4(sf + 1024 + 16 * lane, s1, s1, s1, s1);
      }
    };
    uint32_t sa0[4], sa1[4], sa2[4], sb0[8], sb1[8], sb2[8];
    static_assert(kSfAhead == 3, "three scale-factor register slots");
    Cursor ld{static_cast<int>(blockIdx.x), 0, 0, 0, 0};
    place(ld);
    Cursor pf = ld;
    load_sf(pf, sa0, sb0);
    advance(pf);
    load_sf(pf, sa1, sb1);
    advance(pf);
    load_sf(pf, sa2, sb2);
    advance(pf);
    int slot = 0;
    int stage = 0;
    uint32_t ph = 0, issued = 0, last_par = 0;
    while (ld.tile < total) {
      int w_ok = 1;
      if (lane == 0)
        w_ok = mbar_wait_bounded<true>(smem_u32(&empty[stage]), ph ^ 1u, s_abort, p.err,
                                       ERR_TIMEOUT_PRODUCER);
      if (!__shfl_sync(0xffffffffu, w_ok, 0)) break;
      const uint32_t fb = smem_u32(&full[stage]);
      if (lane == 0) {
        // the e2m1 boxes deliver 8 bytes of codes per 16-byte chunk of
        // their shared-memory image; the transaction count is those bytes
        mbar_arrive_expect_tx(fb, LM::A_BYTES + (FP4W ? LM::B_BYTES / 2 : LM::B_BYTES));
        const uint32_t a_dst = smem_u32(sA + stage * LM::A_BYTES);
        const uint32_t b_dst = smem_u32(sB + stage * LM::B_BYTES);
        tma_load_2d(&tm_a, fb, a_dst, ld.kb * BK, ld.arow);
        if (EPI == EPI_SWIGLU_Q)  // 128 gate rows, then their up rows: one 3-D box
          tma_load_3d(&tm_b, fb, b_dst, ld.kb * BK, ld.n * 128, 2 * ld.e);
        else if (p.l2_hints & 2)  // 256 rows of W_down[e]: one box
          tma_load_2d_hint(&tm_b, fb, b_dst, ld.kb * BK, ld.brow0, l2_policy_evict_first());
        else
          tma_load_2d(&tm_b, fb, b_dst, ld.kb * BK, ld.brow0);
      }
      // this stage's scale factors (loaded kSfAhead iterations ago) into
      // shared memory, then the slot takes those of iteration + kSfAhead
      const uint32_t sf = smem_u32(sSF + stage * LM::SF_BYTES);
      if (slot == 0) {
        store_sf(sf, sa0, sb0);
        load_sf(pf, sa0, sb0);
      } else if (slot == 1) {
        store_sf(sf, sa1, sb1);
        load_sf(pf, sa1, sb1);
      } else {
        store_sf(sf, sa2, sb2);
        load_sf(pf, sa2, sb2);
      }
      slot = slot == kSfAhead - 1 ? 0 : slot + 1;
      advance(pf);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(fb);
      issued |= 1u << stage;
      last_par = (last_par & ~(1u << stage)) | (ph << stage);
      if (++stage == kStages) {
        stage = 0;
        ph ^= 1u;
      }
      advance(ld);
    }
    // Drain: every issued load has landed before the CTA may exit.
    if (lane == 0) {
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
      const uint32_t bf = FP4W ? kMxE2M1 : kMxE4M3;
      const uint32_t id0 = idesc_mx(BM, BN, kMxE4M3, bf, 0), id1 = idesc_mx(BM, BN, kMxE4M3, bf, 1);
      const uint32_t id2 = idesc_mx(BM, BN, kMxE4M3, bf, 2), id3 = idesc_mx(BM, BN, kMxE4M3, bf, 3);
      int stage = 0;
      uint32_t ph = 0;
      int it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x, ++it) {
        if (!mbar_wait_bounded<true>(smem_u32(tempty), (it & 1) ^ 1u, s_abort, p.err,
                                     ERR_TIMEOUT_MMA))
          break;
        tc_fence_after();
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait_bounded<true>(smem_u32(&full[stage]), ph, s_abort, p.err,
                                       ERR_TIMEOUT_MMA)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sfs = smem_u32(sSF + stage * LM::SF_BYTES);
          const uint32_t sft = tmem + kSfCol0 + stage * kSfSlotCols;
          tmem_cp_sf(sft, sdesc_sf(sfs));
          tmem_cp_sf(sft + 8, sdesc_sf(sfs + 512));
          tmem_cp_sf(sft + 12, sdesc_sf(sfs + 1024));
          const uint64_t ad = sdesc_k_sw128(smem_u32(sA + stage * LM::A_BYTES));
          const uint64_t bd = sdesc_k_sw128(smem_u32(sB + stage * LM::B_BYTES));
          const uint32_t acc = kb != 0 ? 1u : 0u;
          umma_mx(tmem, ad, bd, id0, sft, sft + 8, acc);
          umma_mx(tmem, ad + 2, bd + 2, id1, sft, sft + 8, 1u);
          umma_mx(tmem, ad + 4, bd + 4, id2, sft, sft + 8, 1u);
          umma_mx(tmem, ad + 6, bd + 6, id3, sft, sft + 8, 1u);
          umma_commit(smem_u32(&empty[stage]));
          if (++stage == kStages) {
            stage = 0;
            ph ^= 1u;
          }
        }
        if (ok) umma_commit(smem_u32(tfull));
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
    const int q = warp & 3;               // TMEM lane quarter this warp may access
    const int half = (warp - 2) >> 2;     // which half of the tile's columns
    const int r = q * 32 + lane;
    const uint32_t tl = tmem + (static_cast<uint32_t>(q * 32) << 16);
    int it = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++it) {
      int e, m, n;
      decode_tile_mx(tile, NT, E, s_pref, p.group, p.phases, e, m, n);
      int ok = 1;
      if (lane == 0)
        ok = mbar_wait_bounded<true>(smem_u32(tfull), it & 1, s_abort, p.err,
                                     ERR_TIMEOUT_EPILOGUE);
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      tc_fence_after();
      const int m_e = s_off[e + 1] - s_off[e];
      const bool valid = m * BM + r < m_e;
      const long R = static_cast<long>(s_off[e]) + m * BM + r;
      // the whole accumulator share of this thread into registers, then free it
      uint32_t v[128];
      const int c0 = (EPI == EPI_SWIGLU_Q) ? 64 * half : 128 * half;
      const int c1 = (EPI == EPI_SWIGLU_Q) ? 128 + 64 * half : 128 * half + 64;
      tmem_ld_32x32b_x32(tl + c0, *reinterpret_cast<uint32_t(*)[32]>(v));
      tmem_ld_32x32b_x32(tl + c0 + 32, *reinterpret_cast<uint32_t(*)[32]>(v + 32));
      tmem_ld_32x32b_x32(tl + c1, *reinterpret_cast<uint32_t(*)[32]>(v + 64));
      tmem_ld_32x32b_x32(tl + c1 + 32, *reinterpret_cast<uint32_t(*)[32]>(v + 96));
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(tempty));

      if (EPI == EPI_SWIGLU_Q) {
        // h of features 128n + 64 half + i, i < 64: gate in v[i], up in v[64 + i]
        float hv[64];
#pragma unroll
        for (int i = 0; i < 64; ++i)
          hv[i] = gate_act(__uint_as_float(v[i]), p.act) * __uint_as_float(v[64 + i]);
        uint32_t codes[16];
        if (FP4W) {
          // two 1x32 blocks per thread
          uint32_t b2[2];
#pragma unroll
          for (int b = 0; b < 2; ++b) {
            float amax = 0.f;
#pragma unroll
            for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(hv[32 * b + i]));
            const float sc = ue8m0_block_scale(amax, &b2[b]);
            quant_words<32>(hv + 32 * b, 1.0f / sc, codes + 8 * b);
          }
          if (valid) {
            uint8_t* hs8 = reinterpret_cast<uint8_t*>(p.hs + static_cast<long>(n) * p.n_rows + R);
            *reinterpret_cast<uint16_t*>(hs8 + 2 * half) = static_cast<uint16_t>(b2[0] | (b2[1] << 8));
          }
        } else {
          // one 1x128 block per row: the two halves exchange their maxima
          float amax = 0.f;
#pragma unroll
          for (int i = 0; i < 64; ++i) amax = fmaxf(amax, fabsf(hv[i]));
          float* am = s_amax + (it & 1) * 256;     // double-buffered by tile
          am[half * 128 + r] = amax;
          mbar_arrive(smem_u32(amax_bar));
          int a_ok = 1;
          if (lane == 0)
            a_ok = mbar_wait_bounded(smem_u32(amax_bar), it & 1, s_abort, p.err,
                                     ERR_TIMEOUT_EPILOGUE);
          if (!__shfl_sync(0xffffffffu, a_ok, 0)) break;
          amax = fmaxf(am[r], am[128 + r]);
          uint32_t b;
          const float sc = ue8m0_block_scale(amax, &b);
          quant_words<64>(hv, 1.0f / sc, codes);
          if (valid && half == 0) p.hs[static_cast<long>(n) * p.n_rows + R] = b * 0x01010101u;
        }
        if (valid) {
          uint4* dst = reinterpret_cast<uint4*>(p.hq + R * p.I + n * 128 + 64 * half);
#pragma unroll
          for (int j = 0; j < 4; ++j)
            dst[j] = make_uint4(codes[4 * j], codes[4 * j + 1], codes[4 * j + 2], codes[4 * j + 3]);
        }
      } else {
        if (valid) {
          const int f = __ldg(p.sorted_f + R);
          const int tok = f / p.k;
          const float wgt = __ldg(p.topk_w + f);
          float* orow = p.out32 + static_cast<long>(tok) * p.H + n * BN + 128 * half;
          if (p.l2_hints & 1) {
            const uint64_t pol = l2_policy_evict_last();
#pragma unroll
            for (int j = 0; j < 32; ++j)
              red_add_v4_hint(orow + 4 * j, wgt * __uint_as_float(v[4 * j]),
                              wgt * __uint_as_float(v[4 * j + 1]),
                              wgt * __uint_as_float(v[4 * j + 2]),
                              wgt * __uint_as_float(v[4 * j + 3]), pol);
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              red_add_v4(orow + 4 * j, wgt * __uint_as_float(v[4 * j]),
                         wgt * __uint_as_float(v[4 * j + 1]), wgt * __uint_as_float(v[4 * j + 2]),
                         wgt * __uint_as_float(v[4 * j + 3]));
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

template <int EPI, bool FP4W>
cudaError_t launch_mx_impl(const GroupedGemmMxArgs& a, cudaStream_t s) {
  auto kern = grouped_gemm_mx_kernel<EPI, FP4W>;
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  // one flag per device; any host thread may launch, so the flags are atomic
  static std::atomic<bool> attr_set[64] = {};
  if (dev < 64 && !attr_set[dev].load(std::memory_order_acquire)) {
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, LM::SMEM);
    if (err != cudaSuccess) return err;
    attr_set[dev].store(true, std::memory_order_release);
  }
  MxDev p;
  p.offsets = a.offsets;
  p.tile_pref = a.tile_pref;
  p.E = a.E;
  p.K = a.K;
  p.I = a.I;
  p.H = a.H;
  p.k = a.k;
  p.n_rows = a.n_rows;
  p.err = a.err;
  p.a_sf = a.a_sf;
  p.w_sf = a.w_sf;
  p.hq = a.hq;
  p.hs = a.hs;
  p.out32 = a.out32;
  p.sorted_f = a.sorted_f;
  p.topk_w = a.topk_w;
  p.act = a.act;
  p.group = a.tile_group;
  p.phases = a.phases > 0 ? a.phases : 1;
  p.l2_hints = a.l2_hints;
  launch_pdl(kern, a.num_sms, kThreads, LM::SMEM, s, *a.tm_a, *a.tm_b, p);
  count_launches(1);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm1_mx(const GroupedGemmMxArgs& a, bool fp4, cudaStream_t s) {
  return fp4 ? launch_mx_impl<EPI_SWIGLU_Q, true>(a, s) : launch_mx_impl<EPI_SWIGLU_Q, false>(a, s);
}

cudaError_t launch_gemm2_mx(const GroupedGemmMxArgs& a, bool fp4, cudaStream_t s) {
  return fp4 ? launch_mx_impl<EPI_COMBINE, true>(a, s) : launch_mx_impl<EPI_COMBINE, false>(a, s);
}

}  // namespace moe
