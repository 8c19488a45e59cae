/*
 * moe.h -- C ABI of libmoe, the GB300 (sm_103a) MXFP4 mixture-of-experts FFN
 * layer with softmax top-K routing.
 *
 * The layer, in order (one call per step, all on one CUDA stream):
 *   moe_route    softmax top-K routing of router logits; the shared expert is
 *                appended as slot K (expert id E, weight 1)
 *   moe_permute  stable counting sort of the (token, slot) pairs by expert,
 *                each expert's bucket padded to a multiple of tile_m rows
 *   moe_ffn      grouped gate_up GEMM with a SwiGLU epilogue, grouped down
 *                GEMM scaled by the routing weight, slot-ordered combine
 *
 * Sources (web pages on the method):
 *   [IX]  InferenceX, "MI355X Qwen3.5-397B SGLang" blog, section on the
 *         optimisations: PR #21421 (softmax-scored fused top-K at E=512,
 *         K=10) and PR #20736 (shared expert fused as routed expert top-K+1
 *         when its width equals the routed width).
 *   [VS]  VibeSys, "Qwen3.5-397B serving engine on 4x MI300A": section
 *         "baseline" (fused MoE kernel dequantising MXFP4 in registers),
 *         section "kernels and graph capture", section "cheaper prefill and
 *         collectives" (32-row tiles in the MoE kernel).
 *   [VL]  vLLM, "MiniMax M3 on MI355X": section "local shape and tiling"
 *         (small-M vs large-M launcher regimes, grouped-MoE program order)
 *         and section "shared expert fusion".
 * The pages do not print the weight format; this library reads MXFP4 as E2M1
 * codes, two per byte (low nibble = even k), with one E8M0 scale byte
 * (2^(s-127)) per 32 consecutive k.
 *
 * Conventions for every call:
 *   - Every pointer is a caller-owned DEVICE pointer (cudaMalloc or
 *     equivalent) unless stated.  No call allocates memory or synchronises
 *     the host with the device.  The library's only state is: two device
 *     error words per kernel file (read and cleared by moe_device_error),
 *     the fixed scratch array of moe_ffn_noalloc, and host-side caches (the
 *     per-device SM count and per-kernel shared-memory limits, the scratch
 *     address per CUDA context).  Results never depend on that state.
 *   - Work is enqueued on `stream` (0 = legacy default stream).  Calls are
 *     asynchronous; read outputs only after the stream has completed.
 *   - Arguments and shapes are checked on the host before any launch.  A
 *     rejected call launches nothing and returns MOE_ERR_INVALID_ARG (NULL
 *     pointer, negative size, misaligned pointer) or MOE_ERR_UNSUPPORTED_SHAPE
 *     (a size outside the documented limits).  A failed launch returns
 *     MOE_ERR_CUDA (the CUDA error is left for cudaGetLastError).
 *   - Tensors are dense row-major.  bf16 tensors are passed as uint16_t bit
 *     patterns.  Sizes are in elements unless stated.
 */
#ifndef LIBMOE_MOE_H
#define LIBMOE_MOE_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,
    MOE_ERR_UNSUPPORTED_SHAPE = 2,
    MOE_ERR_WORKSPACE_TOO_SMALL = 3,
    MOE_ERR_CUDA = 4,
    MOE_ERR_INTERNAL = 5
} moe_status_t;

/* Which moe_ffn kernels run: AUTO picks by the mean rows per expert. */
typedef enum {
    MOE_PATH_AUTO = 0,
    MOE_PATH_DECODE = 1, /* small M: weights streamed through registers, mma.sync */
    MOE_PATH_PREFILL = 2, /* large M: TMA + tcgen05 MMA with TMEM accumulators */
    /* large M on the block-scaled tensor cores (tcgen05.mma kind::mxf8f6f4):
     * the E2M1 weights as stored, each bf16 activation as two E4M3 terms */
    MOE_PATH_PREFILL_FP8X2 = 3
} moe_path_t;

/* Static string for a status code (never NULL). */
const char* moe_status_string(moe_status_t status);

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int moe_version(void);

/*
 * moe_route -- softmax top-K routing [IX, PR #21421].
 *
 *   logits     fp32 [T, E] router logits.
 *   topk_ids   int32 [T, Kt] out, Kt = K + (with_shared ? 1 : 0).
 *   topk_w     fp32  [T, Kt] out.
 * For each token: p = softmax over all E logits (fp32, expf); the K experts
 * with the largest logits, in descending order, equal logits ordered by lower
 * expert index (+0 and -0 compare equal); weights p[id] renormalised to sum
 * to 1 over the K selected when `renormalize` is nonzero, else p[id].  With
 * `with_shared` nonzero, slot K holds expert id E with weight 1 [IX, PR #20736].
 * Limits: 1 <= K <= min(E, 32), 1 <= E <= 1024, T >= 0 (T = 0 is a no-op).
 * Preconditions (not checked): no NaN logits and at least one finite logit
 * per token; otherwise the outputs for that token are unspecified.
 * Ids are bit-exact with the plain definition; weights agree with it to a few
 * fp32 ulp (the summation order of the softmax denominator differs).
 */
moe_status_t moe_route(const float* logits, int T, int E, int K, int with_shared, int renormalize,
                       int32_t* topk_ids, float* topk_w, cudaStream_t stream);

/*
 * moe_route_ex -- moe_route with a per-token weight for the shared slot.
 *
 *   shared_w   fp32 [T] or NULL: the weight of slot K for each token (for
 *              models that gate the shared expert per token, e.g. by a
 *              sigmoid of a gate logit computed by the caller); NULL means
 *              weight 1 as in moe_route.  Only allowed with with_shared.
 * The pages fix the shared expert's weight only for the fused equal-width
 * case [IX, PR #20736]; the gate itself is the caller's.  Everything else as
 * moe_route; the routed slots do not depend on shared_w.
 */
moe_status_t moe_route_ex(const float* logits, const float* shared_w, int T, int E, int K,
                          int with_shared, int renormalize, int32_t* topk_ids, float* topk_w,
                          cudaStream_t stream);

/*
 * moe_permute_capacity -- number of int32 entries of `sorted_pairs`:
 *   cap = T*Kt + Et*(tile_m - 1); max_tiles = cap / tile_m entries of
 *   `tile_expert`.  Returns 0 for invalid sizes.
 */
size_t moe_permute_capacity(int T, int Kt, int Et, int tile_m);
size_t moe_permute_max_tiles(int T, int Kt, int Et, int tile_m);

/*
 * moe_permute -- group the T*Kt (token, slot) pairs by expert [VS, 32-row
 * tiles in the MoE kernel].
 *
 *   topk_ids        int32 [T, Kt]; pair q = t*Kt + j names expert topk_ids[q].
 *   sorted_pairs    int32 [cap] out: bucket e holds the pairs of expert e in
 *                   increasing q, starting at expert_offsets[e]; every other
 *                   position (bucket padding, tail) holds -1.
 *   expert_offsets  int32 [Et+1] out: offsets[e] = sum over e' < e of
 *                   count(e') rounded up to a multiple of tile_m;
 *                   offsets[Et] = rows in use.
 *   inv_pairs       int32 [T*Kt] out: position of pair q in sorted_pairs.
 *   tile_expert     int32 [max_tiles] out: tile i (rows [i*tile_m,
 *                   (i+1)*tile_m)) belongs to expert tile_expert[i]; tiles from
 *                   num_tiles on hold -1.
 *   num_tiles       int32 [1] out: offsets[Et] / tile_m (stays on the device).
 * Limits: 1 <= Kt <= 33, 1 <= Et <= 1025, 1 <= tile_m <= 256, cap < 2^31.
 * Output is bit-exact (a deterministic function of topk_ids).  Ids outside
 * [0, Et) are a precondition violation: such pairs are dropped and their
 * inv_pairs entry is -1.  Small batches sort in one CTA; batches of at least
 * 8192 pairs with at least 8 pairs per expert use a four-launch multi-block
 * version of the same stable sort (count, scan, scatter, inverse map), with
 * identical output.
 */
moe_status_t moe_permute(const int32_t* topk_ids, int T, int Kt, int Et, int tile_m,
                         int32_t* sorted_pairs, int32_t* expert_offsets, int32_t* inv_pairs,
                         int32_t* tile_expert, int32_t* num_tiles, cudaStream_t stream);

/*
 * moe_route_permute -- moe_route_ex followed by moe_permute (Kt = K + shared,
 * Et = E + shared), bit-identical to the two calls.  For T up to
 * MOE_ROUTE_PERMUTE_FUSED_MAX_T both run in one launch of one block (tiny
 * batches are bound by launch latency, not by this work [VS, "kernels and
 * graph capture"]); above it one block would route too many tokens per warp,
 * so the two kernels run.  Arguments, limits and errors are those of the two
 * calls.
 */
#define MOE_ROUTE_PERMUTE_FUSED_MAX_T 32
moe_status_t moe_route_permute(const float* logits, const float* shared_w, int T, int E, int K,
                               int with_shared, int renormalize, int tile_m, int32_t* topk_ids,
                               float* topk_w, int32_t* sorted_pairs, int32_t* expert_offsets,
                               int32_t* inv_pairs, int32_t* tile_expert, int32_t* num_tiles,
                               cudaStream_t stream);

/*
 * moe_ffn_workspace_size -- bytes of device workspace moe_ffn needs:
 * the 16-bit SwiGLU intermediate [cap, I], the weighted fp32 per-pair expert
 * outputs [T*Kt, H], x as f16 rows [T, H], when tile_m is a prefill tile
 * height (32, 64, 96, 128, 256) their tile-ordered copy [cap, H], T + cap fp32
 * row factors, cap fp32 position weights and, for prefill tile heights, the
 * shift bytes of the staged y [ceil(cap/32), (H rounded up to 128) / 8] and
 * the scale bytes of h's two E4M3 terms [2 cap, I/32] (MOE_PATH_PREFILL_FP8X2);
 * each 256-byte aligned.
 */
size_t moe_ffn_workspace_size(int T, int H, int I, int Et, int Kt, int tile_m);

/*
 * moe_ffn -- the expert FFN of every (token, slot) pair and the combine
 * [VS, fused MXFP4 MoE kernel; IX/VL, shared expert in the same dispatch].
 *
 *   x        bf16 [T, H] activations.
 *   w13      uint8 [Et, 2I, H/2] packed E2M1 codes of gate (rows 0..I-1) and
 *            up (rows I..2I-1) projections; s13 uint8 [Et, 2I, H/32] E8M0.
 *   w2       uint8 [Et, H, I/2] codes of the down projection; s2 [Et, H, I/32].
 *   topk_w, sorted_pairs, expert_offsets, inv_pairs, tile_expert, num_tiles:
 *            as produced by moe_route / moe_permute with the same T, Kt, Et
 *            and tile_m.
 *   out      bf16 [T, H] out.
 *   workspace / ws_bytes: device scratch of at least moe_ffn_workspace_size().
 * For each pair (t, j) with e = topk_ids[t, j]:
 *   g = W_gate[e] x_t, u = W_up[e] x_t (fp32 accumulation of exact
 *   products), h = bf16(silu(g) * u), y = W2[e] h (fp32);
 *   out_t = bf16(sum over j ascending of topk_w[t, j] * y_tj).
 * Both paths carry x and h into the MMAs as f16 scaled per row by a power
 * of two (largest magnitude in [2^14, 2^15)): elements at least 2^-29 of
 * their row's largest magnitude stay exact, smaller ones move by less than
 * 2^-39 of it.  The prefill path hands y from the down GEMM to the combine
 * as f16 scaled by a power of two per (8 output rows, 32 sorted positions):
 * relative error at most 2^-11 per element (elements more than 2^28 below
 * their group's largest move by less than 2^-38 of it).
 * Result tolerance against the plain fp32 definition: per element
 * |out - ref| <= 1e-2 * (|ref| + rms(ref)) and relative L2 error <= 2e-3
 * (the GEMM summation order differs; SwiGLU bf16 roundings may flip by 1 ulp).
 * Weights are exact: the decode path applies each E8M0 scale as an exact
 * power-of-two factor for scale bytes 7..247 (2^-120..2^120); the prefill
 * path stores each weight row in f16 relative to its largest scale, exact
 * for every group whose scale is within 2^36 of that largest (groups further
 * below are rounded, at most 2^-37 of the row's largest weight).
 * MOE_PATH_PREFILL_FP8X2 carries x and h instead as two E4M3 terms per
 * value with an E8M0 scale per 32 values and term: per block of 32 with
 * largest magnitude amax (biased fp32 exponent b), s_hi = max(b - 7, 0),
 * s_lo = max(s_hi - 5, 0), u = v * 2^(127 - s_hi), hi = E4M3(u) and
 * lo = E4M3((u - hi) * 2^(s_hi - s_lo)), nearest even (moe_split_e4m3x2):
 * exact for every element within 2^14 of amax, smaller ones move by less
 * than 2^-21 amax.  Its y goes to the combine as on the prefill path.
 * Limits: H % 32 == 0, I % 32 == 0, H, I <= 65536; the decode path needs
 * tile_m in {8, 16, 32, 64}, the prefill path tile_m in {32, 64, 128, 256},
 * MOE_PATH_PREFILL_FP8X2 tile_m in {32, 64, 96, 128} and H % 512 == I % 512 == 0.
 * Pointers 16-byte aligned.
 */
moe_status_t moe_ffn(const uint16_t* x, const uint8_t* w13, const uint8_t* s13, const uint8_t* w2,
                     const uint8_t* s2, const float* topk_w, const int32_t* sorted_pairs,
                     const int32_t* expert_offsets, const int32_t* inv_pairs,
                     const int32_t* tile_expert, const int32_t* num_tiles, int T, int H, int I,
                     int Et, int Kt, int tile_m, uint16_t* out, void* workspace, size_t ws_bytes,
                     cudaStream_t stream);

/* moe_ffn with an explicit path choice (MOE_PATH_AUTO behaves like moe_ffn). */
moe_status_t moe_ffn_path(const uint16_t* x, const uint8_t* w13, const uint8_t* s13,
                          const uint8_t* w2, const uint8_t* s2, const float* topk_w,
                          const int32_t* sorted_pairs, const int32_t* expert_offsets,
                          const int32_t* inv_pairs, const int32_t* tile_expert,
                          const int32_t* num_tiles, int T, int H, int I, int Et, int Kt,
                          int tile_m, uint16_t* out, void* workspace, size_t ws_bytes,
                          moe_path_t path, cudaStream_t stream);

/*
 * The three steps of moe_ffn as separate calls; moe_ffn runs exactly these,
 * in this order, on one workspace (at least moe_ffn_workspace_size() bytes):
 *   h  [cap, I] at byte 0, y fp32 [T*Kt, H] at moe_ffn_y_offset(), then
 *   the activation area (x as scaled f16 rows, and for prefill tile heights
 *   their tile-ordered copy) and the fp32 row factors of x and of h.
 * `path` must resolve to the same path for both GEMM calls (AUTO always does
 * for the same sizes).
 *
 * moe_ffn_gate_up: h[p, n] = bf16(silu(g) * u) for every sorted position p
 *   that holds a pair (pads are not written), then each such row re-encoded
 *   in place as f16 times a power of two per row (the row factors after the
 *   activation area), the form the down GEMMs read.  On
 *   MOE_PATH_PREFILL_FP8X2 h is written instead as its two E4M3 terms (see
 *   moe_ffn): the h area holds 2 tile_m rows of I bytes per tile (the tile's
 *   high terms, then its low terms) and their scale bytes follow the shifts
 *   of the staged y; x's terms are written in the same form into the area of
 *   the tile-ordered copy, their scale bytes into the y area.
 * moe_ffn_down:    y[q, m] = topk_w[q] * (W2[e] h_p)[m] for every pair q at
 *   position p (the routing-weighted expert outputs).
 * moe_combine:     out[t, m] = bf16(sum over j = 0..Kt-1, ascending, of
 *   y[t*Kt + j, m]); out is bf16 [T, H].
 */
moe_status_t moe_ffn_gate_up(const uint16_t* x, const uint8_t* w13, const uint8_t* s13,
                             const int32_t* sorted_pairs, const int32_t* tile_expert,
                             const int32_t* num_tiles, int T, int H, int I, int Et, int Kt,
                             int tile_m, void* workspace, size_t ws_bytes, moe_path_t path,
                             cudaStream_t stream);
moe_status_t moe_ffn_down(const uint8_t* w2, const uint8_t* s2, const float* topk_w,
                          const int32_t* sorted_pairs, const int32_t* tile_expert,
                          const int32_t* num_tiles, int T, int H, int I, int Et, int Kt,
                          int tile_m, void* workspace, size_t ws_bytes, moe_path_t path,
                          cudaStream_t stream);
moe_status_t moe_combine(const float* y, int T, int H, int Kt, uint16_t* out, cudaStream_t stream);

/*
 * moe_ffn_down_combine -- moe_ffn_down followed by moe_combine, in one call
 * (moe_ffn runs gate_up and then this).  The decode path gives the same
 * results bit for bit.  The prefill and two-term paths write y by sorted position
 * ([cap][H rounded up to 128]) as f16 times a power of two per (8 output
 * rows, 32 sorted positions), with the shift bytes after the position
 * weights; the combine undoes the shift exactly, multiplies by the routing
 * weight and sums each token's Kt positions (inv_pairs) in slot order.  The
 * one rounding to f16 (at most 2^-11 relative) is the only difference from
 * moe_ffn_down + moe_combine; the result meets moe_ffn's tolerance.  The
 * workspace's y is not the [T*Kt, H] array of moe_ffn_down after this call.
 */
moe_status_t moe_ffn_down_combine(const uint8_t* w2, const uint8_t* s2, const float* topk_w,
                                  const int32_t* sorted_pairs, const int32_t* inv_pairs,
                                  const int32_t* tile_expert, const int32_t* num_tiles, int T, int H,
                                  int I, int Et, int Kt, int tile_m, uint16_t* out, void* workspace,
                                  size_t ws_bytes, moe_path_t path, cudaStream_t stream);

/* moe_combine plus one more fp32 [T, H] term added last (NULL: none). */
moe_status_t moe_combine_ex(const float* y, const float* y_extra, int T, int H, int Kt,
                            uint16_t* out, cudaStream_t stream);

/*
 * moe_ffn_dense_shared -- the layer with a shared expert whose width Is
 * differs from the routed experts' I, run as a separate dense MXFP4 MLP over
 * every token: the pages fuse the shared expert into the routed dispatch only
 * when the widths are equal [IX, PR #20736], and describe the unfused shared
 * expert as a separate dense MLP path [VL, "shared expert fusion"].
 *
 *   x, w13, s13, w2, s2, topk_w, sorted_pairs, ..., num_tiles, T, H, I, Et,
 *            Kt, tile_m: the routed layer as for moe_ffn (routed with
 *            with_shared = 0, or with a fused shared slot of its own).
 *   w13s     uint8 [1, 2*Is, H/2], s13s [1, 2*Is, H/32], w2s [1, H, Is/2],
 *            s2s [1, H, Is/32]: the shared expert, same format.
 *   shared_w fp32 [T] per-token weight of the shared expert, or NULL for 1.
 *   workspace: at least moe_ffn_dense_shared_workspace_size() bytes.
 * out_t = bf16(sum over the routed slots j ascending of topk_w[t,j] * y_tj,
 *              then + shared_w[t] * y_shared_t), each y as in moe_ffn (fp32),
 * with y_shared = W2s bf16(silu(W_gate_s x_t) * (W_up_s x_t)).  With Is = I
 * and the shared weights stored as expert E this equals the fused layer
 * (shared slot last) bit for bit.  Limits: those of moe_ffn for both (I, Et,
 * Kt) and (Is, 1, 1); the path of each part is chosen as by MOE_PATH_AUTO.
 */
size_t moe_ffn_dense_shared_workspace_size(int T, int H, int I, int Et, int Kt, int Is, int tile_m);
moe_status_t moe_ffn_dense_shared(const uint16_t* x, const uint8_t* w13, const uint8_t* s13,
                                  const uint8_t* w2, const uint8_t* s2, const float* topk_w,
                                  const int32_t* sorted_pairs, const int32_t* expert_offsets,
                                  const int32_t* inv_pairs, const int32_t* tile_expert,
                                  const int32_t* num_tiles, int T, int H, int I, int Et, int Kt,
                                  int tile_m, const uint8_t* w13s, const uint8_t* s13s,
                                  const uint8_t* w2s, const uint8_t* s2s, int Is,
                                  const float* shared_w, uint16_t* out, void* workspace,
                                  size_t ws_bytes, cudaStream_t stream);

/* Byte offset of y inside the moe_ffn workspace (h [cap, I], 16-bit, comes first). */
size_t moe_ffn_y_offset(int T, int I, int Et, int Kt, int tile_m);

/*
 * moe_device_error -- reads (and with `clear` nonzero resets) the library's
 * device error flags.  *flag receives a bit set: bit 0 (value 1) when one of
 * the kernels' bounded mbarrier waits (2 s each) gave up (the kernel then
 * skips its output, releases its tensor memory and exits instead of
 * hanging); bit 1 (value 2) when a kernel met an index outside its inputs'
 * range -- a tile's expert outside [0, Et), a pair index >= T*Kt, a tile
 * count above the buffers' -- and skipped that work instead of reading or
 * writing out of bounds (inputs not produced by moe_permute for these
 * sizes).  0 means no error.  Bit 0 is sticky: while it is set, the
 * kernels' waits give up at once (so one failure cannot stall later grids),
 * so clear it before relying on further results.  This call synchronises the
 * current device.
 */
moe_status_t moe_device_error(int* flag, int clear);

/*
 * moe_selftest_wait_timeout -- diagnostic: launches one block that waits on
 * an mbarrier nothing arrives at, through the same bounded wait the GEMM
 * kernels use, with a limit of limit_us microseconds (1..10^6).  The wait
 * gives up, raises the device error flag (value 1 of moe_device_error) and the
 * kernel returns; the context stays usable.  It lets a test drive the
 * failure path without faulting or hanging the GPU.  The pages have no
 * counterpart.
 */
moe_status_t moe_selftest_wait_timeout(int limit_us, cudaStream_t stream);

/*
 * moe_set_gemm_events -- profiling hook: from this call on (process-wide,
 * until changed), every FFN call (moe_ffn*, moe_ffn_gate_up, moe_ffn_down,
 * moe_ffn_down_combine, moe_ffn_mxfp4act*) records `before` on its stream
 * right before launching its grouped GEMM kernel and `after` right after,
 * so cudaEventElapsedTime(before, after) is that kernel's duration (each call
 * re-records the pair; set a fresh pair per call to time several).  Both
 * events are caller-created CUDA events of the current device; pass two
 * nulls to switch the hook off.  MOE_ERR_INVALID_ARG when only one is null.
 * A failed record returns MOE_ERR_CUDA from the FFN call.  The pages have no
 * counterpart.
 */
moe_status_t moe_set_gemm_events(cudaEvent_t before, cudaEvent_t after);

/*
 * moe_selftest_wait_split -- diagnostic: one block of two warps whose bounded
 * waits end differently.  Warp 0 waits on an mbarrier nothing arrives at
 * (limit_us microseconds, 1..10^6), warp 1 on one that has already
 * completed.  Each warp makes its outcome uniform across its lanes, the two
 * warps reduce it with AND at a named barrier, and they meet at that barrier
 * again only if both succeeded -- the pattern the GEMM epilogues use before
 * their own named barriers, so a failure seen by one warp cannot leave
 * another waiting there without a limit.
 *   outcome  device int32 [2], 4-byte aligned: written with the outcome each
 *            warp acted on (0 = stopped; both are 0 after a correct run).
 * Raises device error bit 1 (moe_device_error) like moe_selftest_wait_timeout.
 * MOE_ERR_INVALID_ARG for a limit outside 1..10^6 or a null/misaligned
 * outcome.  The pages have no counterpart.
 */
moe_status_t moe_selftest_wait_split(int limit_us, int32_t* outcome, cudaStream_t stream);

/*
 * moe_ffn_noalloc -- moe_ffn for callers that cannot allocate device memory
 * (no cudaMalloc allowed where they run: inside a stream capture that must
 * not allocate, or in a runtime or plugin that only owns fixed, pre-assigned
 * device memory).  The paper has no counterpart; this is a deployment
 * convenience.
 *
 * Same arguments, results and limits as moe_ffn, minus the workspace: the
 * scratch (the whole moe_ffn workspace, moe_ffn_workspace_size() bytes) lives
 * in a fixed device array of MOE_NOALLOC_SCRATCH_BYTES inside the library,
 * which every GPU that loads libmoe holds until the process exits.  The call
 * allocates nothing (no cudaMalloc, cudaFree or allocating library routine).
 *   - Sizes whose moe_ffn_workspace_size() exceeds MOE_NOALLOC_SCRATCH_BYTES
 *     are rejected with MOE_ERR_UNSUPPORTED_SHAPE before any launch (the
 *     64-token decode step of a 4096/1024, 513-expert, top-10+1 layer needs
 *     about 20 MiB with tile_m = 8).
 *   - The first call in each CUDA context looks up the array's device
 *     address there (cudaGetSymbolAddress) and caches it under the context's
 *     ID (cuCtxGetId, never reused within a process), so a context created
 *     again after cudaDeviceReset, or a caller's own non-primary context,
 *     gets its own lookup.  Make the first call in a context before any
 *     stream capture.
 *   - Every call on a device shares the one array, and it keeps the last
 *     call's contents.  Nothing in it needs to start at zero.  Calls whose
 *     kernels overlap on the GPU (different streams without ordering, or
 *     different host threads) race on the scratch and corrupt each other's
 *     results: order them on one stream.
 */
#define MOE_NOALLOC_SCRATCH_BYTES (64u * 1024u * 1024u)
moe_status_t moe_ffn_noalloc(const uint16_t* x, const uint8_t* w13, const uint8_t* s13,
                             const uint8_t* w2, const uint8_t* s2, const float* topk_w,
                             const int32_t* sorted_pairs, const int32_t* expert_offsets,
                             const int32_t* inv_pairs, const int32_t* tile_expert,
                             const int32_t* num_tiles, int T, int H, int I, int Et, int Kt,
                             int tile_m, uint16_t* out, cudaStream_t stream);

/*
 * ---------------------------------------------- MXFP4-quantised activations
 * The layer variant whose GEMMs run MXFP4 x MXFP4 on the block-scaled tensor
 * cores: x and the SwiGLU output are quantised to MXFP4 before the GEMM that
 * reads them.  [OR] OpenRelay, "Gemma 4 31B from B200 to MI355X": section
 * "optimisation 4" (a fused activation + up projection + MXFP4 quantisation
 * kernel) and section "how far from the ceiling" (the matmuls measured
 * against the MXFP4 peak).  The pages print no rounding rule; this library
 * uses the OCP Microscaling v1.0 conversion, per 32 consecutive values:
 *   e      = floor(log2(max |v|)) - 2, clamped to e >= -127
 *   scale  = E8M0 byte e + 127 (byte 0 when every value is zero)
 *   code_k = E2M1 nearest to v_k / 2^e, ties to the even code, magnitudes
 *            above 6 saturating to 6, the sign of v_k kept
 * codes packed two per byte, element 2i in the low nibble.
 */

/*
 * moe_split_e4m3x2 -- the two-term E4M3 encoding MOE_PATH_PREFILL_FP8X2 gives
 * its activations, of a bf16 matrix row by row (see moe_ffn):
 *   x      bf16 [rows, cols] in (cols a multiple of 32).
 *   q_hi, q_lo  uint8 [rows, cols] out: the E4M3 bytes of the two terms.
 *   s_hi, s_lo  uint8 [rows, cols/32] out: their E8M0 scale bytes.
 * x[r, c] == e4m3(q_hi) * 2^(s_hi - 127) + e4m3(q_lo) * 2^(s_lo - 127)
 * exactly whenever |x[r, c]| >= 2^-14 of its block's largest magnitude.
 * Device pointers; x, q_hi and q_lo 16-byte aligned.  Asynchronous on stream.
 */
moe_status_t moe_split_e4m3x2(const uint16_t* x, int rows, int cols, uint8_t* q_hi, uint8_t* q_lo,
                              uint8_t* s_hi, uint8_t* s_lo, cudaStream_t stream);

/*
 * moe_quantize_mxfp4 -- MXFP4 encoding of a bf16 matrix, row by row.
 *   x      [rows, cols] bf16 (16-byte aligned), cols a multiple of 32.
 *   codes  [rows, cols/2] (16-byte aligned), scales [rows, cols/32]: written.
 * Bit-exact with the rule above.  MOE_ERR_UNSUPPORTED_SHAPE when cols % 32.
 */
moe_status_t moe_quantize_mxfp4(const uint16_t* x, int rows, int cols, uint8_t* codes,
                                uint8_t* scales, cudaStream_t stream);

/*
 * moe_ffn_mxfp4act_workspace_size -- bytes of device workspace the calls
 * below need: x codes [T, H/2] and scales [T, H/32], both again in tile
 * order [cap, ...], h codes [cap, I/2] and scales [cap, I/32], the routing
 * weight of each sorted position fp32 [cap], y as f16 rows by sorted
 * position [cap, H] and its shift bytes [ceil(cap/32), H/8] (one power of
 * two per 8 output rows and 32 positions), as moe_ffn_down_combine's
 * prefill path stages it.
 */
size_t moe_ffn_mxfp4act_workspace_size(int T, int H, int I, int Et, int Kt, int tile_m);

/*
 * moe_ffn_mxfp4act -- the expert FFN and combine with MXFP4 activations.
 * Arguments, grouping and output as for moe_ffn; per pair (t, j), e = the
 * pair's expert:
 *   xq  = decode(quantise(x_t))                  (blocks of 32 along H)
 *   g_n = W13[e][n] . xq,  u_n = W13[e][I+n] . xq (fp32 accumulation)
 *   h   = decode(quantise(silu(g) * u))          (fp32 SwiGLU, blocks of 32 along I)
 *   y   = topk_w[t, j] * (W2[e] . h)             (fp32; W2[e] . h passes to the
 *                                                 combine as f16 scaled by a power
 *                                                 of two, at most 2^-11 relative)
 *   out_t = bf16(sum over j ascending of y)
 * Both GEMMs are tcgen05 block-scaled MXFP4 x MXFP4 contractions; the scales
 * of weights and activations are applied inside the MMA.
 * Limits: H % 128 == 0, I % 128 == 0, tile_m in {32, 64, 128, 256}, plus
 * moe_ffn's limits; MOE_ERR_UNSUPPORTED_SHAPE otherwise.
 * Numerics: x's encoding is exact (its inputs are bf16).  h's encoding is
 * decided on fp32 values: the GEMM's fp32 sums (exact for the configured
 * scale ranges, whose products and partial sums fit 24 bits) and silu
 * computed with the fast exponential and division, a few ulp from the
 * correctly rounded result, so an element lying within that distance of an
 * E2M1 decision boundary may land on the neighbouring code.
 */
moe_status_t moe_ffn_mxfp4act(const uint16_t* x, const uint8_t* w13, const uint8_t* s13,
                              const uint8_t* w2, const uint8_t* s2, const float* topk_w,
                              const int32_t* sorted_pairs, const int32_t* expert_offsets,
                              const int32_t* inv_pairs, const int32_t* tile_expert,
                              const int32_t* num_tiles, int T, int H, int I, int Et, int Kt,
                              int tile_m, uint16_t* out, void* workspace, size_t ws_bytes,
                              cudaStream_t stream);

/*
 * The two steps of moe_ffn_mxfp4act (it runs exactly these on one workspace):
 *   moe_ffn_mxfp4act_gate_up: quantises x, gathers its code rows into tile
 *     order and writes h's encoding for every sorted position p of the used
 *     tiles (codes row p, scales row p; padding positions encode zeros);
 *   moe_ffn_mxfp4act_down: the down GEMM from that encoding, scaled by the
 *     routing weight, and the combine into out (inv_pairs: the position of
 *     each pair, from moe_permute).
 * moe_ffn_mxfp4act_h_offsets gives the byte offsets of h's codes [cap, I/2]
 * and scales [cap, I/32] inside the workspace, so a caller can inspect h or
 * supply its own.
 */
moe_status_t moe_ffn_mxfp4act_gate_up(const uint16_t* x, const uint8_t* w13, const uint8_t* s13,
                                      const int32_t* sorted_pairs, const int32_t* tile_expert,
                                      const int32_t* num_tiles, int T, int H, int I, int Et,
                                      int Kt, int tile_m, void* workspace, size_t ws_bytes,
                                      cudaStream_t stream);
moe_status_t moe_ffn_mxfp4act_down(const uint8_t* w2, const uint8_t* s2, const float* topk_w,
                                   const int32_t* sorted_pairs, const int32_t* inv_pairs,
                                   const int32_t* tile_expert, const int32_t* num_tiles, int T,
                                   int H, int I, int Et, int Kt, int tile_m, uint16_t* out,
                                   void* workspace, size_t ws_bytes, cudaStream_t stream);
moe_status_t moe_ffn_mxfp4act_h_offsets(int T, int H, int I, int Et, int Kt, int tile_m,
                                        size_t* codes_offset, size_t* scales_offset);

/* The regime MOE_PATH_AUTO picks for these sizes [VL, small-M vs large-M]:
 * MOE_PATH_DECODE or MOE_PATH_PREFILL (the large-M regime, whichever of its
 * two paths moe_ffn_auto_path_shape names). */
moe_path_t moe_ffn_auto_path(int T, int Kt, int Et, int tile_m);

/* The path MOE_PATH_AUTO runs for these sizes: in the large-M regime
 * MOE_PATH_PREFILL_FP8X2 where its widths and tile heights allow (it is the
 * faster of the two there), else MOE_PATH_PREFILL; the MOE_FORCE_PATH
 * environment override (decode, prefill, prefill_fp8x2) applies as it does
 * to the FFN calls.  Returns MOE_PATH_AUTO for sizes no path supports. */
moe_path_t moe_ffn_auto_path_shape(int T, int H, int I, int Et, int Kt, int tile_m);

#ifdef __cplusplus
}
#endif

#endif /* LIBMOE_MOE_H */
