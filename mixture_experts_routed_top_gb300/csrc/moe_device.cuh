// Device-side building blocks for sm_103a: mbarriers with bounded waits,
// TMA tile loads, tcgen05 (UMMA) descriptors, MMA issue, commit and TMEM
// loads, all as inline PTX.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "moe_internal.h"

namespace moe {

// Upper bound for any single wait on an mbarrier inside a kernel (ns).
// Every legitimate wait in these kernels lasts microseconds.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- PDL
// pdl_launch_dependents: the next kernel on the stream may be scheduled now.
// pdl_wait: block until the previous kernel on the stream has completed and
// its memory operations are visible; every kernel calls it before touching
// global memory.  Both are no-ops for a launch without the PDL attribute.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// The same with acquire semantics at cluster scope, for barriers that the
// other CTA of a pair arrives on (remote arrives, multicast commits, TMA
// completions of its loads).
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// The same with a suspend-time hint: the thread may sleep (not poll) for
// up to kSuspendHintNs until the phase completes, leaving the issue slots of
// its SM sub-partition to the other roles.  Measured: faster for the bf16
// grouped GEMMs, slower for the FP8 one, whose epilogue must wake at once.
constexpr uint32_t kSuspendHintNs = 20000;

__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(kSuspendHintNs)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete, giving up after
// `limit_ns` or as soon as another warp of the CTA has raised `*abort`.
// On giving up it ORs `code` into the global error word and raises *abort.
// kSleep selects mbar_try_wait_sleep for the repeated tries, kCluster the
// cluster-scope acquire of mbar_try_wait_cluster.
template <bool kSleep = false, bool kCluster = false>
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  volatile int* abort, int* err, int code,
                                                  uint64_t limit_ns = kWaitLimitNs) {
  auto try_once = [&](bool sleep) {
    return kCluster ? mbar_try_wait_cluster(bar, parity)
                    : (sleep ? mbar_try_wait_sleep(bar, parity) : mbar_try_wait(bar, parity));
  };
  if (try_once(false)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (try_once(kSleep)) return true;
    if (*abort) return false;
    if (globaltimer_ns() - t0 > limit_ns) {
      atomicOr(err, code);
      *abort = 1;
      return false;
    }
  }
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 2-D tiled bulk tensor load global -> shared, completing `bar`'s transaction
// count.  x is the innermost (contiguous) coordinate in elements.
__device__ __forceinline__ void tma_load_2d(const CUtensorMap* map, uint32_t bar, uint32_t dst,
                                            int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
      : "memory");
}

// The same with an L2 policy for the loaded lines.
__device__ __forceinline__ void tma_load_2d_hint(const CUtensorMap* map, uint32_t bar,
                                                 uint32_t dst, int x, int y, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "l"(pol)
      : "memory");
}

// 3-D tiled bulk tensor load (coordinates x innermost, then y, z).  Used
// for the gate/up weights viewed as [2E, I, K]: one box of {x, rows, 2}
// brings the gate rows and then the matching up rows of one expert.
__device__ __forceinline__ void tma_load_3d(const CUtensorMap* map, uint32_t bar, uint32_t dst,
                                            int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Warp-wide: allocate `ncols` TMEM columns, address written to smem `dst`.
__device__ __forceinline__ void tmem_alloc(uint32_t dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// Shared-memory matrix descriptor for a K-major operand tile written by TMA
// with 128-byte swizzling: rows of 128 bytes, 8-row swizzle atoms 1024 bytes
// apart (stride byte offset), tile base 1024-byte aligned.
__device__ __forceinline__ uint64_t sdesc_k_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);   // start address / 16
  d |= static_cast<uint64_t>(1) << 16;                   // leading byte offset (unused here)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;           // stride byte offset / 16
  d |= static_cast<uint64_t>(1) << 46;                   // descriptor version (sm_100 family)
  d |= static_cast<uint64_t>(2) << 61;                   // swizzle mode: 128 B
  return d;
}

// Same for a K-major tile written by TMA with 64-byte swizzling: rows of
// 64 bytes, 8-row swizzle atoms 512 bytes apart, tile base 512-byte aligned.
__device__ __forceinline__ uint64_t sdesc_k_sw64(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);   // start address / 16
  d |= static_cast<uint64_t>(1) << 16;                   // leading byte offset (unused here)
  d |= static_cast<uint64_t>(512 >> 4) << 32;            // stride byte offset / 16
  d |= static_cast<uint64_t>(1) << 46;                   // descriptor version (sm_100 family)
  d |= static_cast<uint64_t>(4) << 61;                   // swizzle mode: 64 B
  return d;
}

// Instruction descriptor, kind::f16 with bf16 A/B, fp32 D, both K-major.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4)                                   // D format f32
         | (1u << 7)                                 // A format bf16
         | (1u << 10)                                // B format bf16
         | (static_cast<uint32_t>(N >> 3) << 17)     // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);    // M / 16
}

// Instruction descriptor, kind::f8f6f4 with e4m3 A/B, fp32 D, both K-major.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N) {
  return (1u << 4)                                   // D format f32
         | (0u << 7)                                 // A format e4m3
         | (0u << 10)                                // B format e4m3
         | (static_cast<uint32_t>(N >> 3) << 17)
         | (static_cast<uint32_t>(M >> 4) << 24);
}

// Instruction descriptor of a block-scaled kind::mxf8f6f4 MMA: fp32 D,
// K-major A and B in the formats a_fmt / b_fmt (kMxE4M3, kMxE2M1), UE8M0
// scale factors, and sf_id = which byte of each operand's 32-bit scale word
// (that is, which 32-wide K sub-block of a 128-wide K block) this
// instruction applies.
constexpr uint32_t kMxE4M3 = 0, kMxE2M1 = 5;
__host__ __device__ constexpr uint32_t idesc_mx(int M, int N, uint32_t a_fmt, uint32_t b_fmt,
                                                uint32_t sf_id) {
  return (sf_id << 4)                                // B scale-factor byte
         | (a_fmt << 7)                              // A format
         | (b_fmt << 10)                             // B format
         | (static_cast<uint32_t>(N >> 3) << 17)     // N / 8
         | (1u << 23)                                // scale factors are UE8M0
         | (static_cast<uint32_t>(M >> 4) << 24)     // M / 16
         | (sf_id << 29);                            // A scale-factor byte
}

// Shared-memory descriptor of a 32-row x 16-byte tile without swizzling
// (8-row core matrices of 128 bytes, stored one after the other): the
// source of a scale-factor copy into TMEM.
__device__ __forceinline__ uint64_t sdesc_sf(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);   // start address / 16
  d |= static_cast<uint64_t>(128 >> 4) << 16;            // leading byte offset
  d |= static_cast<uint64_t>(128 >> 4) << 32;            // stride byte offset: next 8 rows
  d |= static_cast<uint64_t>(1) << 46;                   // descriptor version (sm_100 family)
  return d;                                              // swizzle mode 0: none
}

// Warp-independent (one thread): copy a 32-row x 16-byte scale-factor tile
// from shared memory into TMEM columns taddr..taddr+3, lanes 0..31, and the
// same data into each of the other three lane quarters.
__device__ __forceinline__ void tmem_cp_sf(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
               : "memory");
}

// Block-scaled D[tmem] (+)= (A * sfA) (B * sfB)^T, single CTA, K = 32 per
// instruction, scale factors read from TMEM (one byte per row of A and per
// column of B, selected by the descriptor's sf_id).
__device__ __forceinline__ void umma_mx(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                        uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X "
      "[%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}

// Make this thread's generic-proxy shared-memory writes visible to the async
// proxy (tcgen05.cp, TMA) before another thread hands them over.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, single CTA.
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void umma_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when every tcgen05 operation issued so far by this
// thread has completed.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// ---------------------------------------------------------------- CTA pairs
// Two CTAs of a cluster of two (ranks 0 and 1) run one tcgen05.mma with
// .cta_group::2: rank 0 issues it, each CTA supplies half of A (M/2 rows) and
// half of B (N/2 columns) from the same shared-memory offsets and holds its
// M/2 rows of the accumulator in its own TMEM.
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Shared::cluster address of the variable at shared::cta address `addr` in
// the CTA of cluster rank `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// All threads of both CTAs (release / acquire at cluster scope).
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}
// Tiled loads into this CTA's shared memory whose completion is counted on
// an mbarrier of either CTA of the pair (`bar`: shared::cluster address).
__device__ __forceinline__ void tma_load_3d_pair(const CUtensorMap* map, uint32_t bar,
                                                 uint32_t dst, int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z)
      : "memory");
}
__device__ __forceinline__ void tma_load_4d_pair(const CUtensorMap* map, uint32_t bar,
                                                 uint32_t dst, int x, int y, int z, int w) {
  asm volatile(
      "cp.async.bulk.tensor.4d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z), "r"(w)
      : "memory");
}
// Warp-wide, one warp in each CTA of the pair together: the same `ncols`
// TMEM columns in both CTAs, address written to each CTA's smem `dst`.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T over the pair (issued by rank 0).
__device__ __forceinline__ void umma_f16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                              uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on the mbarrier at shared offset `bar` in both CTAs of the
// pair when this thread's tcgen05 operations so far have completed.
__device__ __forceinline__ void umma_commit_pair_both(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar), "h"(static_cast<uint16_t>(3))
      : "memory");
}
// The same on this CTA's barrier only.
__device__ __forceinline__ void umma_commit_pair_local(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}
// Named barrier over `nthreads` threads (a multiple of 32) of this CTA.
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Warp-wide TMEM -> registers: 32 lanes x 32 consecutive 32-bit columns.
// Thread i of the warp receives lane (taddr.lane + i), columns col..col+31.
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr));
}
// Warp-wide TMEM -> registers: 32 lanes x 8 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld_32x32b_x8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// tcgen05.wait::ld that also names the two 8-column loads it completes, so no
// use of their registers can be scheduled above the wait.
__device__ __forceinline__ void tmem_ld_wait_x8x2(uint32_t (&a)[8], uint32_t (&b)[8]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(a[0]), "+r"(a[1]), "+r"(a[2]), "+r"(a[3]), "+r"(a[4]), "+r"(a[5]),
                 "+r"(a[6]), "+r"(a[7]), "+r"(b[0]), "+r"(b[1]), "+r"(b[2]), "+r"(b[3]),
                 "+r"(b[4]), "+r"(b[5]), "+r"(b[6]), "+r"(b[7])
               :
               : "memory");
}

// ---------------------------------------------------------------- misc
// silu(g) = g / (1 + e^-g).  The fast division (2 ulp of fp32 for divisors
// below 2^126) replaces the IEEE one: the result is rounded to bf16 or
// e4m3 next, and the division was the costliest step of the gate/up
// epilogue.  -g is clamped at 80 so the divisor stays in that range; below
// g = -80 the result is under 2^-100 * |g| either way.
__device__ __forceinline__ float silu_f(float g) {
  return __fdividef(g, 1.0f + __expf(fminf(-g, 80.0f)));
}

// Gate activation of the gated MLP, `act` a moe_activation value (uniform
// across the kernel, so the branch never diverges): silu, exact GELU
// x/2 (1 + erf(x / sqrt 2)), or max(x, 0).
__device__ __forceinline__ float gate_act(float g, int act) {
  if (act == MOE_ACT_SILU) return silu_f(g);
  if (act == MOE_ACT_GELU) return 0.5f * g * (1.0f + erff(g * 0.70710678118654752f));
  return fmaxf(g, 0.0f);
}

// Smallest power of two >= q (q > 0, fp32), read from q's bits (exact, no
// log2); *stored gets the biased exponent byte b of the UE8M0 form, scale
// 2^(b-127).  b is capped at 254 (255 is not a scale).
__device__ __forceinline__ float ue8m0_ceil(float q, uint32_t* stored) {
  const uint32_t bits = __float_as_uint(q);
  int b = static_cast<int>((bits >> 23) & 0xFFu) + ((bits & 0x7FFFFFu) != 0u ? 1 : 0);
  b = b > 254 ? 254 : b;
  *stored = static_cast<uint32_t>(b);
  return b == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(static_cast<uint32_t>(b) << 23);
}

// e4m3 scale of one block from its absolute maximum: amax/448 (IEEE fp32
// division) or the smallest power of two >= that quotient; amax = 0 -> 1.
// Returns the scale value and its stored form (fp32 bits or exponent byte).
__device__ __forceinline__ float block_scale(float amax, bool ue8m0, uint32_t* stored) {
  if (amax == 0.f) {
    *stored = ue8m0 ? 127u : __float_as_uint(1.0f);
    return 1.0f;
  }
  const float q = amax / 448.0f;
  if (!ue8m0) {
    *stored = __float_as_uint(q);
    return q;
  }
  return ue8m0_ceil(q, stored);
}

// Two fp32 values -> e4m3 codes (round to nearest even, saturating), lo in
// the low byte.
__device__ __forceinline__ uint16_t e4m3x2(float lo, float hi) {
  return static_cast<uint16_t>(__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3));
}

// Fire-and-forget fp32 reductions into global memory (no value returned,
// so the L2 answers nothing back): the combine of the down projections.
__device__ __forceinline__ void red_add_v4(float* p, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c),
               "f"(d)
               : "memory");
}
__device__ __forceinline__ void red_add_f32(float* p, float a) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(p), "f"(a) : "memory");
}
// L2 policies: lines kept in preference to others (evict_last), or the
// first to go (evict_first).
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
// The reductions above with an L2 policy for the accumulator lines.
__device__ __forceinline__ void red_add_v4_hint(float* p, float a, float b, float c, float d,
                                                uint64_t pol) {
  asm volatile("red.global.add.L2::cache_hint.v4.f32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p),
               "f"(a), "f"(b), "f"(c), "f"(d), "l"(pol)
               : "memory");
}
__device__ __forceinline__ void red_add_f32_hint(float* p, float a, uint64_t pol) {
  asm volatile("red.global.add.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(p), "f"(a), "l"(pol)
               : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Exclusive scan of one value per thread; blockDim.x must be 1024 and all
// threads must call it.
__device__ __forceinline__ int block_exclusive_scan(int v, int* s_warp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = s_warp[lane];
    int ws = w;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, ws, off);
      if (lane >= off) ws += y;
    }
    s_warp[lane] = ws - w;  // exclusive prefix of warp totals
    if (lane == 31) s_warp[32] = ws;
  }
  __syncthreads();
  const int res = s_warp[warp] + x - v;
  *total = s_warp[32];
  __syncthreads();
  return res;
}

}  // namespace moe
