// moe_dispatch_noalloc: the dispatch entry point for callers that cannot
// allocate device memory.
//
// Some callers have no way to hand us a workspace: a serving runtime that
// reserves all device memory once at start-up and forbids any later
// cudaMalloc (which can fail mid-request and synchronises the device), or a
// plugin interface whose per-call hook must not allocate.  For them the
// dispatch scratch (per-chunk expert counts, the m-tile prefix, the touched
// list and the error word) lives in one file-scope device array of fixed
// size instead of a caller buffer.  The array is part of the library image:
// every GPU that loads the library holds it until the process exits.
//
// The host never uses the array's name as an address (in host code it only
// names a host-side shadow).  The device address is looked up with
// cudaGetSymbolAddress once per device, with that device current, on the
// first call made on it; that first call should therefore come before any
// stream capture.
//
// Every call shares the one array, and it keeps the previous call's
// contents: the error word is cleared at the start of each call, and all
// other scratch is fully rewritten before it is read.  Calls whose work
// overlaps on the GPU (different streams, or different host threads without
// ordering) race on the array and give wrong results.
#include <cuda_runtime.h>

#include <mutex>

#include "moe_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = MOE_DISPATCH_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_dispatch_scratch[kNoAllocScratchBytes];

// Largest dispatch scratch any accepted size needs: the error-word block,
// the m-tile prefix and the touched list (E+1 ints each), and the per-chunk
// expert counts (at most 128 chunks of E ints), each region 1024-byte
// aligned.  The fixed array covers it, so the size check below is only a
// guard against a future change of that layout.
constexpr size_t align1k(size_t x) { return (x + 1023) / 1024 * 1024; }
constexpr size_t kMaxDispatchScratch = align1k(sizeof(moe::WsHeader)) +
                                       2 * align1k((moe::kMaxE + 1) * 4) +
                                       align1k(128 * static_cast<size_t>(moe::kMaxE) * 4);
static_assert(kMaxDispatchScratch <= kNoAllocScratchBytes,
              "the fixed dispatch scratch must hold every accepted size");

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once
// per device).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> g(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_dispatch_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" {

moe_status moe_dispatch_noalloc(const int32_t* topk_idx, int T, int E, int k, int32_t* counts,
                                int32_t* offsets, int32_t* sorted_f, int32_t* row_of,
                                void* stream) {
  if (T < 0 || E < 1 || k < 1)
    return moe::set_last_error(MOE_ERR_INVALID_ARG, "moe_dispatch_noalloc: bad sizes");
  if (E > moe::kMaxE)
    return moe::set_last_error(MOE_ERR_UNSUPPORTED, "moe_dispatch_noalloc: E must be in [1, %d]",
                               moe::kMaxE);
  if (k > E || k > moe::kMaxK)
    return moe::set_last_error(MOE_ERR_UNSUPPORTED,
                               "moe_dispatch_noalloc: k must be in [1, min(E, %d)]", moe::kMaxK);
  if (static_cast<long>(T) * k > 0x7FFFFFFFL)
    return moe::set_last_error(MOE_ERR_UNSUPPORTED, "moe_dispatch_noalloc: T*k exceeds int32");
  const size_t need = moe_dispatch_workspace_size(T, E, k);
  if (need > kNoAllocScratchBytes)
    return moe::set_last_error(MOE_ERR_UNSUPPORTED,
                               "moe_dispatch_noalloc: these sizes need %zu bytes of scratch, more "
                               "than the fixed %zu; use moe_dispatch with a workspace",
                               need, kNoAllocScratchBytes);
  void* scratch = nullptr;
  cudaError_t e = scratch_address(&scratch);
  if (e != cudaSuccess)
    return moe::set_last_error(MOE_ERR_CUDA, "moe_dispatch_noalloc: cudaGetSymbolAddress failed: %s",
                               cudaGetErrorString(e));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The error word must start at zero; everything else is rewritten.
  e = cudaMemsetAsync(scratch, 0, sizeof(moe::WsHeader), s);
  if (e != cudaSuccess)
    return moe::set_last_error(MOE_ERR_CUDA,
                               "moe_dispatch_noalloc: clearing the error word failed: %s",
                               cudaGetErrorString(e));
  return moe_dispatch(topk_idx, T, E, k, counts, offsets, sorted_f, row_of, scratch,
                      kNoAllocScratchBytes, stream);
}

}  // extern "C"
