/*
 * moe_experts.h - C ABI of the GB300 (sm_103a) routed top-k Mixture-of-Experts
 * experts forward.
 *
 * What is computed (Hugging Face Transformers "Experts backends" page,
 * introduction): every token is sent to the k experts its router ranks
 * highest; its hidden state goes through each of those experts' gated MLP
 * (fused gate/up projection, SwiGLU, down projection; backends table, deepgemm_megamoe row,
 * and the SonicMoE section's silu -> SwiGLU mapping) and the k results are
 * summed with the routing weights.  Tokens are ordered by selected expert
 * before the expert GEMMs (backends table, grouped_mm and deepgemm rows).  FP8
 * experts carry float32 or UE8M0 block scales (paragraph after the backends
 * table), FP4 experts are int8-packed e2m1 codes with UE8M0 scales, and
 * activations are quantised dynamically per row ("FP8 and FP4 quantized
 * experts" section).
 *
 * Conventions shared by every entry point:
 *   - All pointers named as device buffers must point to device memory of the
 *     current CUDA device; the caller owns every buffer.  The library
 *     allocates no device memory: scratch lives in a caller-provided
 *     workspace sized by moe_workspace_size().
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Work is
 *     queued asynchronously on it; MOE_OK means "validated and launched".
 *   - Row-major layouts everywhere.  bf16 buffers are passed as void*.
 *   - Every device buffer must be 16-byte aligned.
 *   - On a non-OK status nothing was launched (argument errors) or a CUDA
 *     launch failed (MOE_ERR_CUDA); moe_last_error() gives a message.
 *   - Errors are loud: an unsupported shape or format is rejected, never
 *     computed approximately (the page's note on Blackwell scale formats
 *     prefers a clear error to a wrong result).
 */
#ifndef MOE_EXPERTS_H
#define MOE_EXPERTS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,  /* null pointer, bad size, misaligned buffer      */
  MOE_ERR_UNSUPPORTED = 2,  /* shape or format outside the supported set      */
  MOE_ERR_CUDA = 3,         /* a CUDA runtime/driver call failed              */
  MOE_ERR_TIMEOUT = 4,      /* a device-side bounded wait expired             */
  MOE_ERR_WORKSPACE = 5     /* workspace missing or smaller than required     */
} moe_status;

typedef enum { MOE_W_BF16 = 0, MOE_W_FP8_E4M3 = 1, MOE_W_FP4_E2M1 = 2 } moe_wdtype;

/* Block-scale format of FP8 weights (and of the dynamic activation scales,
 * which always use the weights' format): MOE_SCALE_F32 stores float32 scales,
 * MOE_SCALE_UE8M0 stores one byte b per block with scale 2^(b-127). */
typedef enum { MOE_SCALE_NONE = 0, MOE_SCALE_F32 = 1, MOE_SCALE_UE8M0 = 2 } moe_scale_fmt;

/* Library version (major*10000 + minor*100 + patch). */
int moe_version(void);

/* Message for the last non-OK status returned on this host thread. */
const char* moe_last_error(void);

/*
 * moe_route - router top-k (introduction of the page: per token the router
 * picks k experts).
 *   logits   device fp32 [T, E]
 *   topk_idx device int32 [T, k]  out: selected experts, slot j ordered by
 *            descending logit, equal logits by ascending expert index
 *   topk_w   device fp32 [T, k]   out: softmax over all E renormalised over
 *            the k selected = exp(l_j - l_max) / sum over the selected; a row
 *            whose largest logit is -inf gets 1/k in every slot
 * Logits must not be NaN (not checked).  1 <= k <= min(E, 32), E <= 1024.
 * T = 0 is a no-op.
 */
moe_status moe_route(const float* logits, int T, int E, int k,
                     int32_t* topk_idx, float* topk_w, void* stream);

/*
 * moe_dispatch - order the T*k routing entries by expert (grouped_mm /
 * deepgemm rows of the backends table).  Flat entry f = t*k + j.
 *   counts   device int32 [E]    rows routed to each expert
 *   offsets  device int32 [E+1]  exclusive scan of counts, offsets[E] = T*k
 *   sorted_f device int32 [T*k]  row r of the expert-contiguous order holds
 *            entry sorted_f[r]; within an expert entries ascend in f (stable)
 *   row_of   device int32 [T*k]  inverse permutation
 *   ws       device scratch of at least moe_dispatch_workspace_size() bytes
 * topk_idx values must lie in [0, E); an out-of-range entry is reported as
 * MOE_ERR_INVALID_ARG by the next moe_workspace_status() on this ws.
 */
size_t moe_dispatch_workspace_size(int T, int E, int k);
moe_status moe_dispatch(const int32_t* topk_idx, int T, int E, int k,
                        int32_t* counts, int32_t* offsets, int32_t* sorted_f,
                        int32_t* row_of, void* ws, size_t ws_bytes, void* stream);

/*
 * moe_workspace_size - bytes of device scratch moe_experts_forward needs for
 * these sizes and this weight type.
 */
size_t moe_workspace_size(int T, int H, int I, int E, int k, moe_wdtype wdtype);

/*
 * moe_workspace_accumulator_offset - byte offset, inside a workspace sized
 * by moe_workspace_size() with the same arguments, of the fp32 accumulator
 * [T, H] into which the grouped paths sum the weighted expert outputs before
 * the single rounding to bf16.  After such a forward (every path except the
 * small-token GEMVs: bf16 with T*k <= moe_get_decode_rows(), FP4 with
 * T*k <= moe_get_fp4_gemv_rows()) and until the next call on the workspace,
 * it holds the un-rounded output, and out is its round-to-nearest-even bf16
 * image.  Meant for checking results; 0 for invalid sizes.
 */
size_t moe_workspace_accumulator_offset(int T, int H, int I, int E, int k, moe_wdtype wdtype);

/*
 * moe_experts_forward - routed experts forward (introduction: expert
 * outputs weighted by the routing weights and summed; gated MLP of the
 * deepgemm_megamoe row).
 *   hidden      device bf16 [T, H]
 *   topk_idx    device int32 [T, k], values in [0, E)
 *   topk_w      device fp32 [T, k]
 *   w_gate_up   device [E, 2I, H]: rows 0..I-1 of each expert are the gate
 *               projection, rows I..2I-1 the up projection
 *   w_down      device [E, H, I]
 *   wdtype      MOE_W_BF16: weights are bf16, scales must be NULL and
 *               sfmt MOE_SCALE_NONE.
 *               MOE_W_FP8_E4M3: weights are e4m3 bytes with 128x128 block
 *               scales scale_gate_up [E, 2I/128, H/128] and scale_down
 *               [E, H/128, I/128], float32 or UE8M0 bytes per sfmt; the
 *               activations (hidden rows and the SwiGLU output) are quantised
 *               on the fly per row in 1x128 blocks with the same format.
 *               There is no static activation scale.
 *               MOE_W_FP4_E2M1: weights are e2m1 codes packed two per byte,
 *               the even element in the low nibble: w_gate_up [E, 2I, H/2],
 *               w_down [E, H, I/2] bytes, with one UE8M0 byte per 1x32 block
 *               along the contraction axis: scale_gate_up [E, 2I, H/32],
 *               scale_down [E, H, I/32]; sfmt must be MOE_SCALE_UE8M0.  The
 *               hidden rows and the SwiGLU output are quantised on the fly to
 *               e4m3 in 1x32 UE8M0 blocks.  Block-scaled tensor-core GEMMs
 *               run these forwards (they need H % 256 == 0 and 32-byte
 *               aligned weight buffers, else MOE_ERR_UNSUPPORTED /
 *               MOE_ERR_INVALID_ARG); CUDA-core GEMVs take batches of at most
 *               64 routed rows when H % 256 != 0, or up to the threshold
 *               moe_set_fp4_gemv_rows sets.
 *   out         device bf16 [T, H]: out[t] = sum_j topk_w[t,j] *
 *               down(silu(gate x_t) * up x_t) of expert topk_idx[t,j],
 *               accumulated in fp32 and rounded once to bf16
 *   ws          device scratch, >= moe_workspace_size() bytes, 256-B aligned;
 *               its first 256 bytes must be zero before the first forward
 *               that uses it (they hold the device error word and two
 *               counters of the small-token decode kernel; the library
 *               leaves them zero after every call, and moe_workspace_status
 *               resets them after an error)
 * Requirements: H % 128 == 0 (H % 256 == 0 for FP8 weights), I % 128 == 0,
 * 1 <= k <= min(E, 32), E <= 1024, T >= 0 (T = 0 is a no-op).  Other
 * shapes: MOE_ERR_UNSUPPORTED.
 * FP8 weights with MOE_SCALE_NONE, FP4 weights without MOE_SCALE_UE8M0:
 * MOE_ERR_INVALID_ARG.
 * Inputs are never written; out is fully overwritten.
 * Calls that share one ws must be ordered (same stream or synchronised).
 */
moe_status moe_experts_forward(const void* hidden, int T, int H,
                               const int32_t* topk_idx, const float* topk_w,
                               int E, int k, int I,
                               const void* w_gate_up, const void* w_down,
                               moe_wdtype wdtype,
                               const void* scale_gate_up, const void* scale_down,
                               moe_scale_fmt sfmt,
                               void* out, void* ws, size_t ws_bytes, void* stream);

/*
 * Gate activation of the gated expert MLP (SonicMoE section: silu, gelu and
 * relu map to SwiGLU, GeGLU and ReGLU): h = act(gate x) * (up x).
 *   MOE_ACT_SILU  silu(x) = x / (1 + e^-x)            (SwiGLU)
 *   MOE_ACT_GELU  exact GELU x/2 (1 + erf(x / sqrt 2)) (GeGLU)
 *   MOE_ACT_RELU  max(x, 0)                            (ReGLU)
 */
typedef enum { MOE_ACT_SILU = 0, MOE_ACT_GELU = 1, MOE_ACT_RELU = 2 } moe_activation;

/*
 * moe_experts_forward_act - moe_experts_forward with the gate activation as
 * an argument; moe_experts_forward is this call with MOE_ACT_SILU.  Every
 * path (token-row, swap-AB and CTA-pair grouped GEMMs, FP8, FP4, decode)
 * applies it in the gate/up epilogue.  An activation outside moe_activation:
 * MOE_ERR_INVALID_ARG.  Everything else as moe_experts_forward.
 */
moe_status moe_experts_forward_act(const void* hidden, int T, int H,
                                   const int32_t* topk_idx, const float* topk_w,
                                   int E, int k, int I,
                                   const void* w_gate_up, const void* w_down,
                                   moe_wdtype wdtype,
                                   const void* scale_gate_up, const void* scale_down,
                                   moe_scale_fmt sfmt, moe_activation act,
                                   void* out, void* ws, size_t ws_bytes, void* stream);

/*
 * moe_quantize_fp8_blocks - quantise bf16 matrices into e4m3 codes with one
 * scale per 128x128 block (the FP8 expert format of the "FP8 and FP4
 * quantized experts" section).  Scale s = amax/448 (float32 division) for
 * MOE_SCALE_F32, or the smallest power of two >= that quotient for
 * MOE_SCALE_UE8M0 (stored as the biased exponent byte); amax = 0 gives
 * s = 1; code = e4m3(x * (1/s)), round to nearest even, saturated to +-448.
 *   w      device bf16 [nmat, rows, cols], rows % 128 == 0, cols % 128 == 0
 *   q      device uint8 [nmat, rows, cols]
 *   scale  device fp32 or uint8 [nmat, rows/128, cols/128]
 */
moe_status moe_quantize_fp8_blocks(const void* w, int nmat, int rows, int cols,
                                   moe_scale_fmt sfmt, uint8_t* q, void* scale,
                                   void* stream);

/*
 * moe_quantize_fp4_blocks - quantise bf16 matrices into packed e2m1 codes
 * with one UE8M0 scale per 1x32 block along each row (the FP4 expert format
 * of the "FP8 and FP4 quantized experts" section).  Scale s = the smallest
 * power of two >= amax/6 (float32 division; amax = 0 gives s = 1), stored
 * as the biased exponent byte b, s = 2^(b-127); code = the e2m1 value
 * nearest to x * (1/s) (0, 0.5, 1, 1.5, 2, 3, 4, 6 and their negatives),
 * ties to the even code, saturated to +-6; two codes per byte, the even
 * element in the low nibble.  Inputs must be finite.
 *   w      device bf16 [nmat, rows, cols], cols % 32 == 0
 *   q      device uint8 [nmat, rows, cols/2]
 *   scale  device uint8 [nmat, rows, cols/32]
 */
moe_status moe_quantize_fp4_blocks(const void* w, int nmat, int rows, int cols,
                                   uint8_t* q, uint8_t* scale, void* stream);

/*
 * moe_workspace_status - synchronise `stream`, read and clear the device
 * error word at the head of `ws`.  Returns MOE_ERR_TIMEOUT if a bounded
 * device wait expired in a kernel that used this workspace,
 * MOE_ERR_INVALID_ARG if a kernel met an out-of-range expert index, MOE_OK
 * otherwise.
 */
moe_status moe_workspace_status(void* ws, void* stream);

/*
 * moe_set_decode_rows - route bf16 forwards with T*k <= rows through the
 * small-token decode path (weight streaming over the touched experts only,
 * the page's "Decode-stage switching" idea); larger ones through the grouped
 * tensor-core path.  rows < 0 restores the default (16, the measured
 * crossover); values are clamped to 2048 (the decode path's workspace is
 * sized up to that many rows).
 * Process-wide setting; moe_get_decode_rows returns the threshold in use.
 */
void moe_set_decode_rows(int rows);
int moe_get_decode_rows(void);

/*
 * moe_set_swap_rows - choose the orientation of the bf16 grouped GEMMs.
 * With T*k <= rows_per_expert * E (few routed rows per expert) the expert's
 * weight rows are the MMA's M side and its tokens the N side (tokens padded
 * to 16, "swap AB"); otherwise 128 token rows are the M side.  After a call
 * with rows_per_expert >= 0 the rule applies to both GEMMs (0: token rows
 * always).  The default (rows_per_expert < 0) applies it with 128 rows per
 * expert to the gate/up GEMM and uses swap AB for the down GEMM at every
 * size, the fastest combination measured on the benchmark workloads.
 * Process-wide setting; moe_get_swap_rows returns the threshold in use.
 */
void moe_set_swap_rows(int rows_per_expert);
int moe_get_swap_rows(void);

/*
 * moe_set_down_phases - tile order of the down GEMMs (bf16 on CTA pairs
 * and swap-AB, block-scaled and float32-scale FP8).  Their combine adds every routed row into the fp32
 * accumulator [T, H] of its token; when that accumulator is larger than L2,
 * a token's k contributions, made by different experts at different times,
 * find its lines evicted.  With P phases the output columns are cut into P
 * slices run one after the other, each over all experts, so only a
 * [T, H/P] slice is live at a time (the h rows are read once per phase).
 * phases < 0 (the default): the smallest P that divides the number of
 * 256-column blocks and brings the slice to at most 40 MB; 0 or 1: one
 * phase; P > 1: at least P (rounded up to such a divisor).  Process-wide;
 * moe_get_down_phases returns the setting (-1 = automatic).
 */
void moe_set_down_phases(int phases);
int moe_get_down_phases(void);

/*
 * moe_set_pair_gemm - bf16 grouped GEMMs (forwards above the decode
 * threshold) on CTA pairs: tcgen05.mma.cta_group::2, 256 weight rows (128
 * per SM) against up to 256 of an expert's tokens.  mask bit 0: the gate/up
 * GEMM, bit 1: the down GEMM (only where H % 256 == 0; else the one-CTA
 * kernel runs); mask < 0 restores the default: gate/up on pairs where
 * H >= 4096 (measured faster at DeepSeek-V3 width, slower at H = 2048), the
 * down GEMM on pairs where T*k >= 8*E, i.e. at least 8 routed rows per
 * expert on average (measured faster there; the one-CTA swap-AB kernel is
 * faster for smaller batches).
 * Process-wide; moe_get_pair_gemm returns the mask set (-1 = the default).
 */
void moe_set_pair_gemm(int mask);
int moe_get_pair_gemm(void);

/*
 * moe_set_down_l2_hints - L2 policies of the down GEMMs (bf16 on CTA pairs
 * and swap-AB, block-scaled and float32-scale FP8; bit 1 only swap-AB and
 * block-scaled): bit 0 = the fp32 accumulator's reductions evict_last (its
 * lines kept in preference to streaming data), bit 1 = the W_down tile
 * loads evict_first.  0: no policy; bits < 0 restore the default, 1 (the
 * accumulator evict_last, measured 1-3 % faster; bit 1 measured no faster).
 * Process-wide; moe_get_down_l2_hints returns the bits in use.
 */
void moe_set_down_l2_hints(int bits);
int moe_get_down_l2_hints(void);

/*
 * moe_set_tile_group - tile order of the token-row gate/up GEMMs (bf16,
 * block-scaled and float32-scale FP8; for the CTA-pair kernel, its 256-token
 * tiles).  Inside an expert the 128-row m-tiles run in groups of m_tiles:
 * every n-tile of one group (m fastest), then the next group, so that an expert with many rows
 * re-reads one group's activation tiles per n-tile instead of all of them.
 * 0 puts all of an expert's m-tiles in one group; m_tiles < 0 restores the
 * default (4, measured 2 % faster than one group on the skewed
 * DeepSeek-V3-shaped layer).  Process-wide; moe_get_tile_group returns the
 * setting in use.
 */
void moe_set_tile_group(int m_tiles);
int moe_get_tile_group(void);

/*
 * moe_set_decode_single - bf16 forwards with at most 64 routed rows on the
 * small-token path run as one cooperative kernel (on != 0: the gate/up
 * GEMV, then the down GEMV and combine, whose weight loads start before the
 * last h values are ready) or as two kernels (on == 0, the default, measured
 * faster).  If the GPU cannot hold the single kernel's grid at once, the two
 * kernels run.
 * Process-wide; moe_get_decode_single returns the setting.
 */
void moe_set_decode_single(int on);
int moe_get_decode_single(void);

/*
 * moe_set_block_scaled_mma - how UE8M0 block scales of FP8 experts are
 * applied.  on != 0 (the default): by the tensor core's block scaling
 * (tcgen05.mma kind::mxf8f6f4, one UE8M0 byte per 32-wide K sub-block of
 * every row and column), so no software promotion runs; on == 0: by the
 * software promotion kernel that float32 scales always use.  Both give the
 * same mathematics (scales are powers of two; only the fp32 summation order
 * differs).  Process-wide; moe_get_block_scaled_mma returns the setting.
 */
void moe_set_block_scaled_mma(int on);
int moe_get_block_scaled_mma(void);

/*
 * moe_set_fp4_gemv_rows - FP4 forwards with T*k <= rows run on the
 * CUDA-core GEMVs (small-token path), larger ones on the block-scaled
 * tensor-core GEMMs.  rows < 0 restores the default (0: the GEMMs at every
 * size, measured faster than the GEMVs down to one token); values are
 * clamped to 64.  Process-wide; moe_get_fp4_gemv_rows returns the threshold
 * in use.
 */
void moe_set_fp4_gemv_rows(int rows);
int moe_get_fp4_gemv_rows(void);

/*
 * Stage timing: between moe_profile_begin() and moe_profile_end() every
 * launch of moe_experts_forward records a CUDA event pair on its stream
 * around each stage.  moe_profile_end() synchronises those events and writes
 * up to `n` entries: the summed milliseconds and launch count per stage
 * (index = moe_stage); it returns the number of stages.  Not thread-safe.
 */
typedef enum {
  MOE_STAGE_DISPATCH = 0, /* histogram, scan, permute, sorted-row copy    */
  MOE_STAGE_GEMM1 = 1,    /* gate/up projection + SwiGLU                   */
  MOE_STAGE_GEMM2 = 2,    /* down projection + weighted combine             */
  MOE_STAGE_FINISH = 3,   /* fp32 -> bf16 output                            */
  MOE_STAGE_COUNT = 4
} moe_stage;
moe_status moe_profile_begin(void);
int moe_profile_end(float* stage_ms, int* stage_launches, int n);

/*
 * moe_profile_read - the same report as moe_profile_end() without ending the
 * session or releasing its events.  Meant for forwards captured in a CUDA
 * graph while profiling was on: every replay re-records the captured event
 * pairs, so reading after each replay gives that replay's stage times.
 * Synchronises the events; returns the number of stages.  Not thread-safe.
 */
int moe_profile_read(float* stage_ms, int* stage_launches, int n);

/*
 * moe_dispatch_noalloc - moe_dispatch for callers that cannot allocate
 * device memory.  The page has no counterpart to this entry point; it exists
 * for integration only.
 *
 * Some callers cannot provide a workspace: serving runtimes that reserve all
 * device memory at start-up and forbid later cudaMalloc calls (which can fail
 * mid-request and synchronise the device), or plugin hooks that must not
 * allocate.  This variant keeps its scratch in a fixed device array inside
 * the library (MOE_DISPATCH_NOALLOC_SCRATCH_BYTES, held on every GPU that
 * loads the library until the process exits) and allocates nothing.  The
 * caller still passes the inputs and the four outputs, with the same meaning
 * and layout as moe_dispatch.
 *   - E, k and T*k have the same limits as moe_dispatch (E <= 1024,
 *     k <= min(E, 32), T*k < 2^31) and are checked first.  Every size those
 *     limits accept needs at most about 535 KB of scratch, so the fixed
 *     array always suffices; its size check (MOE_ERR_UNSUPPORTED when
 *     moe_dispatch_workspace_size(T, E, k) exceeds it, before anything is
 *     launched) is only a guard.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.
 *   - All calls share the one array, which keeps the last call's contents;
 *     each call clears the error word and rewrites the rest.  Calls that
 *     overlap on the GPU (other streams, unordered host threads) race and
 *     give wrong results.
 *   - Out-of-range expert indices are skipped; the caller sees them as
 *     offsets[E] < T*k.
 */
#define MOE_DISPATCH_NOALLOC_SCRATCH_BYTES (1u << 20)
moe_status moe_dispatch_noalloc(const int32_t* topk_idx, int T, int E, int k,
                                int32_t* counts, int32_t* offsets, int32_t* sorted_f,
                                int32_t* row_of, void* stream);

/*
 * moe_launch_count - number of kernels this library has launched in this
 * process (all entry points, all devices).  Driver memsets are not counted.
 */
long long moe_launch_count(void);

/*
 * moe_selftest_wait_timeout - launch one kernel that waits on a device
 * barrier nothing will ever complete, with a wait limit of `limit_us`
 * microseconds; the kernel gives up, records MOE_ERR_TIMEOUT in the error
 * word at the head of `ws` and returns, leaving the context usable.  Used to
 * test the timeout path without hanging a GPU.
 */
moe_status moe_selftest_wait_timeout(void* ws, size_t ws_bytes, int limit_us, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_EXPERTS_H */
