/*
 * moe_route.h -- C ABI of the GB300 (sm_103a) MoE routing + FP8 quantisation
 * hot path.
 *
 * Five operations, in the order a MoE layer runs them:
 *
 *   moe_topk_gate        scores [T,E] f32  -> topk_idx [T,k] i32, topk_weights [T,k] f32
 *   moe_route_map        topk_idx          -> counts [E], offsets [E+1], pos [T,k], sorted_src [T*k]
 *   moe_expand_cast_fp8  x [T,H] bf16, pos -> out [R,H] E4M3 bytes, out_sf [R,H/128] f32
 *   swiglu_cast_fp8      x [M,2N] bf16     -> out [M,N] E4M3 bytes, out_sf [M,N/128] f32
 *   moe_combine          y [R,H] bf16, topk_weights, pos -> out [T,H] bf16 or f32
 *
 * and their widened forms: the padded expert layout (moe_route_map_aligned,
 * moe_expand_cast_fp8_padded), the scale options and SwiGLU variants
 * (moe_expand_cast_fp8_ex, swiglu_cast_fp8_ex), the FP4 E2M1 casts
 * (moe_expand_cast_fp4, swiglu_cast_fp4), steps 1-3 in one call with a fused
 * decode launch (moe_route_expand_cast_fp8), and the route map without a
 * workspace (moe_route_map_noalloc).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Pointers are DEVICE pointers into memory the caller owns (allocated by the
 *   caller, e.g. through PyTorch).  The library allocates no device memory and
 *   keeps no per-call state; a caller-provided workspace is the only scratch.
 * - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *   stream).  Every call only enqueues work on it and returns at once; no call
 *   synchronises except moe_get_device_status.
 * - Tensors are dense row-major with the shapes given; bf16 is passed as raw
 *   16-bit patterns, E4M3 (OCP E4M3FN: bias 7, max 448, no infinities) as raw
 *   bytes.
 * - Arguments are checked on the host BEFORE anything is launched.  A bad
 *   argument returns MOE_ERR_INVALID_ARG (or MOE_ERR_UNSUPPORTED for a valid
 *   but unimplemented option) and launches nothing.  A zero-sized problem
 *   returns MOE_OK and launches no kernel (moe_route_map with T == 0 still
 *   zero-fills counts and offsets with cudaMemsetAsync).
 * - Conditions only the data can reveal (an expert index outside [0,E), a
 *   pos row outside [0,num_rows)) are not memory errors: the kernel skips the
 *   offending access, and sets a bit in a device-side error word that
 *   moe_get_device_status reports and clears.
 * - A launch failure returns MOE_ERR_CUDA; moe_last_cuda_error_string gives
 *   the CUDA text.  No C++ exception crosses this boundary.
 * - Calls on distinct streams may run concurrently; the device error word is
 *   shared by all of them.
 * - Inputs must not contain NaN.  Results for NaN inputs are unspecified.
 *
 * Sources (page title, section):
 *   [TK]  "DeepSeek open-sources TileKernels: GPU operators written in Python
 *         approach hardware limits" (itsolotime.com): 2.1 Top-K Gating,
 *         2.2 Fused Expand, 3.1 quantisation config, 3.2 per-token cast,
 *         3.3 SwiGLU + quantisation, and the routing chain opening section 2.
 *   [PX]  "CuTeDSL at Perplexity" (perplexity.ai blog): MoE dispatch and
 *         combine, the TP=1 local kernel.
 */
#ifndef MOE_ROUTE_H
#define MOE_ROUTE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_ROUTE_ABI_VERSION 1

/* Largest supported expert count and top-k. */
#define MOE_MAX_EXPERTS 1024
#define MOE_MAX_TOPK 32
/* The FP8 casts' scaling group: one fp32 scale per 128 channels (the FP4
 * casts take 16, 32, 64 or 128). */
#define MOE_CAST_GROUP 128

typedef enum moe_status {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1, /* bad pointer, size, alignment or range       */
    MOE_ERR_UNSUPPORTED = 2, /* valid request this library does not implement */
    MOE_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed          */
    MOE_ERR_DEVICE = 4       /* a kernel flagged bad data (see error bits)    */
} moe_status_t;

typedef enum moe_weight_mode {
    MOE_WEIGHTS_NONE = 0,        /* write topk_idx only                         */
    MOE_WEIGHTS_SOFTMAX_TOPK = 1 /* softmax over the k selected scores          */
} moe_weight_mode_t;

typedef enum moe_out_dtype {
    MOE_OUT_BF16 = 0,
    MOE_OUT_F32 = 1
} moe_out_dtype_t;

/* Scale options of the *_ex cast calls (bit flags). */
#define MOE_SF_COLMAJOR 0x1u /* scales transposed: [G][sf_ld] (TMA-aligned column-major) */
#define MOE_SF_POW2 0x2u     /* round_sf: smallest power of two >= the plain scale      */
#define MOE_SF_UE8M0 0x4u    /* store the power-of-two scale as its biased exponent
                                byte; requires MOE_SF_POW2.  Row-major: [rows][G] u8;
                                with MOE_SF_COLMAJOR: [ceil(G/4)][sf_ld] u32, four
                                consecutive groups of a row per word (group 4i+j in
                                byte j)                                                 */

/* Bits of the device error word (moe_get_device_status). */
#define MOE_DEVERR_EXPERT_RANGE 0x1u /* route_map: topk_idx outside [0, E)      */
#define MOE_DEVERR_POS_RANGE 0x2u    /* expand/combine: pos >= num_rows         */
#define MOE_DEVERR_DUPLICATE_EXPERT 0x4u /* route_map: a token names an expert twice */
#define MOE_DEVERR_ROWS_SHORT 0x8u   /* route_map_aligned: num_rows < padded total */
#define MOE_DEVERR_TIMEOUT 0x10u     /* fused decode path: a bounded wait ran out */
#define MOE_DEVERR_BOUNDS 0x20u      /* debug-bounds library only: an internal index
                                        or alignment check failed, access skipped */

/* Paths of moe_route_expand_cast_fp8. */
#define MOE_PATH_AUTO 0       /* the library's choice (see moe_route_expand_cast_fp8)     */
#define MOE_PATH_FUSED 1      /* one cooperative launch (decode shapes only)              */
#define MOE_PATH_SEPARATE 2   /* moe_topk_gate + moe_route_map + moe_expand_cast_fp8     */
#define MOE_PATH_REPLICATED 3 /* one ordinary launch, routing repeated per block (small T) */
#define MOE_PATH_CHAINED 4    /* three launches: top-k + chunk ranks, a scan, the expand   */
#define MOE_AUTO_REPLICATED_MAX_TOKENS 1024 /* AUTO's switch from REPLICATED to SEPARATE  */

/*
 * moe_topk_gate -- [TK] 2.1 Top-K Gating, plus the "Weight Normalization" that
 * closes [TK]'s routing chain, read as the softmax over the selected scores.
 *
 * For every token t the k experts with the largest scores[t, :], in
 * descending score order; equal scores go to the lower expert index (so the
 * result is unique).  -0.0 and +0.0 compare equal; +-inf are ordinary values.
 *   scores       [T, E] f32, read-only.
 *   topk_idx     [T, k] i32 out (the page's int64 narrowed: E <= 1024).
 *   topk_weights [T, k] f32 out, may be NULL when weight_mode is
 *                MOE_WEIGHTS_NONE; with MOE_WEIGHTS_SOFTMAX_TOPK,
 *                w[t,j] = exp(s_j - s_0) / sum_i exp(s_i - s_0) over the k
 *                selected scores s_0 >= s_1 >= ... (fp32, expf); scores must
 *                be finite.
 * Requires 1 <= E <= MOE_MAX_EXPERTS, 1 <= k <= min(E, MOE_MAX_TOPK), T >= 0,
 * scores 4-byte aligned.
 */
moe_status_t moe_topk_gate(const float *scores, int64_t num_tokens,
                           int32_t num_experts, int32_t num_topk,
                           int32_t *topk_idx, float *topk_weights,
                           int32_t weight_mode, void *stream);

/*
 * moe_route_map_workspace_bytes -- device scratch moe_route_map needs for a
 * problem of this size: a histogram row of E int32 per chunk of consecutive
 * tokens (chunks of a multiple of 32 tokens, at most 512, aiming at about 128
 * chunks), rounded up to 256 bytes.  0 when num_tokens == 0 or k is out of
 * range.  Pure host function.
 */
size_t moe_route_map_workspace_bytes(int64_t num_tokens, int32_t num_experts,
                                     int32_t num_topk);

/*
 * moe_route_map -- [PX] local dispatch: "count the tokens assigned to each
 * expert and give each token a unique index in its expert's list", made
 * stable and deterministic (the page's shared-memory atomics are not):
 *   counts[e]     = #{(t,j) : topk_idx[t,j] == e}                 [E]   i32
 *   offsets[e]    = sum_{e' < e} counts[e'], offsets[E] = T*k     [E+1] i32
 *   pos[t,j]      = offsets[e] + #{(t',j') before (t,j) in row-major
 *                   order with topk_idx[t',j'] == e}              [T,k] i32
 *   sorted_src[r] = t*k + j for r = pos[t,j]   (inverse of pos)   [T*k] i32
 * Rows of one expert are therefore in ascending token order.
 *   workspace: at least moe_route_map_workspace_bytes(...) bytes of device
 *   memory, 16-byte aligned; contents on entry are ignored; it is busy until
 *   the work enqueued on `stream` completes.  (For T <= 1024, E <= 256 and
 *   T*k <= 16384 the map is built in one launch in which every block builds
 *   it in shared memory and writes its own tokens' entries; the workspace is
 *   then not touched.  Otherwise a histogram launch and a rank launch.)
 * Each token's k experts must be distinct (as moe_topk_gate produces them); a
 * repeated expert sets MOE_DEVERR_DUPLICATE_EXPERT and leaves that token's
 * results unspecified (no write leaves the output buffers).  An index outside
 * [0, E) sets MOE_DEVERR_EXPERT_RANGE; that copy is not counted, its pos is
 * -1, and sorted_src keeps holes at its end.
 * Requires the same E and k limits as moe_topk_gate and T*k < 2^31.
 */
moe_status_t moe_route_map(const int32_t *topk_idx, int64_t num_tokens,
                           int32_t num_experts, int32_t num_topk,
                           int32_t *counts, int32_t *offsets, int32_t *pos,
                           int32_t *sorted_src, void *workspace,
                           size_t workspace_bytes, void *stream);

/*
 * moe_route_map_aligned -- the route map into a padded expert layout, for an
 * expert GEMM that wants every expert's rows to start on a tile boundary
 * ([PX] dispatch: "tokens are optionally copied into padded buffers for the
 * MoE GEMM"; [TK] 2.2: rows no token lands on are zero-filled by the expand).
 * As moe_route_map, except that each expert's segment is rounded up to a
 * multiple of `align` rows:
 *   offsets[e+1]  = offsets[e] + align * ceil(counts[e] / align)
 *   pos[t,j]      = offsets[e] + rank of the copy among e's copies
 *   sorted_src[r] = t*k + j for r = pos[t,j]; -1 for every other row of
 *                   [0, num_rows) (padding rows and the tail)   [num_rows] i32
 * counts[e] is the unpadded count.  align == 1 gives moe_route_map's results
 * (with a -1 tail when num_rows > T*k).
 *   num_rows: rows of the padded buffers; T*k + E*(align-1) always suffices.
 *   If it is smaller than offsets[E] the kernel sets MOE_DEVERR_ROWS_SHORT and
 *   drops the copies that would land at or past num_rows (their pos is -1).
 * Requires 1 <= align <= 4096, T*k + E*(align-1) < 2^31 and num_rows < 2^31;
 * the workspace is moe_route_map_workspace_bytes(T, E, k).
 */
moe_status_t moe_route_map_aligned(const int32_t *topk_idx, int64_t num_tokens,
                                   int32_t num_experts, int32_t num_topk,
                                   int32_t align, int64_t num_rows, int32_t *counts,
                                   int32_t *offsets, int32_t *pos, int32_t *sorted_src,
                                   void *workspace, size_t workspace_bytes,
                                   void *stream);

/*
 * moe_route_map_noalloc -- moe_route_map for callers that cannot allocate
 * device memory.  The pages have no counterpart: it exists for callers such
 * as engine plugins or runtimes that hand out every device buffer from their
 * own arena and forbid allocation while they run, so they cannot provide the
 * workspace moe_route_map needs.  Same arguments and results as
 * moe_route_map, minus the workspace; its histogram lives instead in one
 * static device array of MOE_ROUTE_NOALLOC_SCRATCH_BYTES that every GPU
 * loading this library holds until the process exits.
 * - Allocates nothing (no cudaMalloc, cudaFree or allocating library call).
 * - Returns MOE_ERR_UNSUPPORTED, launching nothing, when the problem needs
 *   more than that: moe_route_map_workspace_bytes(T, E, k) >
 *   MOE_ROUTE_NOALLOC_SCRATCH_BYTES.  Every problem with T <= 65536 fits
 *   (any E, k); larger ones fit while ceil(T / 512) * E <= 2^18.
 * - The first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current; make that first call
 *   before any stream capture.
 * - All calls share the one array.  Nothing in it needs clearing (each call
 *   writes every entry it reads), but calls that overlap on the GPU (other
 *   streams, other threads) race on it and give wrong results: serialise them.
 * - Argument checks, including 4-byte alignment of every array, and data
 *   errors are those of moe_route_map: an expert index outside [0, E) or a
 *   token naming one expert twice sets its bit in the device error word that
 *   moe_get_device_status reports.
 */
#define MOE_ROUTE_NOALLOC_SCRATCH_BYTES (1u << 20)
moe_status_t moe_route_map_noalloc(const int32_t *topk_idx, int64_t num_tokens,
                                   int32_t num_experts, int32_t num_topk,
                                   int32_t *counts, int32_t *offsets,
                                   int32_t *pos, int32_t *sorted_src,
                                   void *stream);

/*
 * moe_expand_cast_fp8 -- [TK] 3.2 per_token_cast fused with [TK] 2.2
 * expand_to_fused.  For every token t and 128-channel group g of x[t, :]:
 *   amax   = max |x| over the group (bf16 widened exactly to f32)
 *   sf     = max(amax, 1e-4f) / 448   (f32, IEEE round-to-nearest-even;
 *            1e-4 is [TK] 3.1's E4M3 clamp_min_value)
 *   sf_inv = 1 / sf                   (f32, IEEE; "multiply by the inverse")
 *   q      = E4M3(x * sf_inv)         (f32 product, round to nearest even,
 *            saturating to +-448; the sign of zero is kept)
 * and for every j with pos[t,j] >= 0 the row of codes goes to
 * out[pos[t,j], :] and the group scales to out_sf[pos[t,j], :].  pos[t,j] < 0
 * means "no copy" ([TK] 2.2).  Rows of out no pos names are not written.
 *   x       [T, H] bf16, 16-byte aligned.      pos [T, k] i32.
 *   out     [num_rows, H] u8, 16-byte aligned. out_sf [num_rows, H/128] f32.
 * Requires H % 128 == 0, 1 <= k <= MOE_MAX_TOPK, num_rows < 2^31, group ==
 * 128 and T * H/128 < 2^31 (else MOE_ERR_UNSUPPORTED).  pos >= num_rows sets
 * MOE_DEVERR_POS_RANGE and is skipped.
 */
moe_status_t moe_expand_cast_fp8(const void *x, int64_t num_tokens,
                                 int32_t hidden, int32_t num_topk,
                                 const int32_t *pos, int64_t num_rows,
                                 uint8_t *out, float *out_sf, int32_t group,
                                 void *stream);

/*
 * moe_expand_cast_fp8_padded -- moe_expand_cast_fp8 into a padded layout,
 * zero-filling in the same launch every row r < num_rows with
 * sorted_src[r] < 0 ([TK] 2.2: the expand kernel's grid covers max(T, rows)
 * so that the invalid rows are zeroed without another launch).  Those rows get
 * all-zero codes and all-zero scales; rows named by pos are written as
 * moe_expand_cast_fp8 writes them.  sorted_src: [num_rows] i32 as
 * moe_route_map_aligned returns it.  Same requirements and error bits as
 * moe_expand_cast_fp8.
 */
moe_status_t moe_expand_cast_fp8_padded(const void *x, int64_t num_tokens,
                                        int32_t hidden, int32_t num_topk,
                                        const int32_t *pos, const int32_t *sorted_src,
                                        int64_t num_rows, uint8_t *out, float *out_sf,
                                        int32_t group, void *stream);

/*
 * moe_expand_cast_fp8_ex -- moe_expand_cast_fp8 with the scale options of
 * [TK] 3.1 (round_sf, packed UE8M0) and [TK] 2.2 (TMA-aligned column-major
 * scales), and optionally the zero-fill of moe_expand_cast_fp8_padded.
 *   sf_flags: 0 or a combination of MOE_SF_COLMAJOR, MOE_SF_POW2,
 *             MOE_SF_UE8M0 (which requires MOE_SF_POW2):
 *     0                      out_sf [num_rows][G] f32 (moe_expand_cast_fp8's)
 *     COLMAJOR               out_sf [G][sf_ld] f32
 *     POW2 (| COLMAJOR)      as above, scale = smallest power of two >=
 *                            max(amax, 1e-4)/448 (codes use its exact inverse)
 *     UE8M0|POW2             out_sf [num_rows][G] u8: biased exponent (value
 *                            2^(byte-127)) of the power-of-two scale
 *     UE8M0|POW2|COLMAJOR    out_sf [ceil(G/4)][sf_ld] u32, group 4i+j of row r
 *                            in byte j of word [i][r]
 *   sf_ld: column-major leading dimension, >= num_rows and a multiple of 4
 *          (16-byte aligned columns for TMA); ignored without COLMAJOR.
 *   sorted_src: NULL, or [num_rows] i32 to zero-fill the rows with a negative
 *          entry (codes 0, scales 0.0 or byte 0) in the same launch.
 *   workspace, workspace_bytes: NULL / 0, or device memory (16-byte aligned)
 *          of at least moe_expand_cast_fp8_ex_workspace_bytes(num_tokens,
 *          hidden, sf_flags) bytes.  With a column-major layout, sorted_src
 *          and a workspace, each token's scales are staged there once and a
 *          second kernel writes the column-major buffer row by row from
 *          sorted_src, in whole 128-byte lines; sorted_src must then be pos's
 *          inverse (as moe_route_map / moe_route_map_aligned return it), and
 *          a sorted_src entry >= num_tokens * num_topk sets
 *          MOE_DEVERR_POS_RANGE and gives that row zero scales.  Otherwise each copy's scales are
 *          stored directly (the same values; every store then writes part of
 *          an L2 sector, which at large num_rows is much slower).  Unused for
 *          row-major layouts.
 * Requirements and error bits as moe_expand_cast_fp8; out_sf 4-byte aligned
 * (1-byte for row-major UE8M0).
 */
moe_status_t moe_expand_cast_fp8_ex(const void *x, int64_t num_tokens, int32_t hidden,
                                    int32_t num_topk, const int32_t *pos,
                                    const int32_t *sorted_src, int64_t num_rows,
                                    uint8_t *out, void *out_sf, uint32_t sf_flags,
                                    int64_t sf_ld, void *workspace, size_t workspace_bytes,
                                    int32_t group, void *stream);

/* Workspace bytes moe_expand_cast_fp8_ex stages column-major scales in:
 * num_tokens * G * 4 (f32) or num_tokens * ceil(G/4) * 4 (packed UE8M0),
 * G = hidden / 128, rounded up to 256; 0 for row-major layouts. */
size_t moe_expand_cast_fp8_ex_workspace_bytes(int64_t num_tokens, int32_t hidden,
                                              uint32_t sf_flags);

/*
 * moe_expand_cast_fp4 -- expand + per-group FP4 E2M1 cast: [TK] 3.1
 * (CastOutputConfig with the float4_e2m1fn output type, clamp_min_value =
 * max_value * 2^-126 = 6 * 2^-126), 3.2 (per-group absmax -> scale ->
 * multiply by the scale's inverse, num_per_channels channels per group) and
 * 2.2 (copy to the rows pos names).
 *   scale of a group: fl32(max(amax, 6 * 2^-126) / 6), or the smallest power
 *   of two >= it under MOE_SF_POW2; code = E2M1(fl32(x * fl32(1 / scale))),
 *   round to nearest, ties to the even code, saturating at +-6, the sign kept
 *   (also for zero).  E2M1 (OCP MX FP4): sign bit 3, exponent bits 2..1 with
 *   bias 1, mantissa bit 0; magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6.
 *   out: [num_rows][H/2] u8, two codes per byte, element 2i in the low nibble.
 *   out_sf, sf_flags, sf_ld, sorted_src, workspace: as moe_expand_cast_fp8_ex,
 *   with G = H / group scales per row.
 *   group: 16, 32, 64 or 128 channels per scale.
 * Requires H % 32 == 0, H % group == 0, H <= 16384, 1 <= k <= MOE_MAX_TOPK,
 * num_rows < 2^31, x and out 16-byte aligned.  Error bits as
 * moe_expand_cast_fp8.
 */
moe_status_t moe_expand_cast_fp4(const void *x, int64_t num_tokens, int32_t hidden,
                                 int32_t num_topk, const int32_t *pos, const int32_t *sorted_src,
                                 int64_t num_rows, uint8_t *out, void *out_sf, uint32_t sf_flags,
                                 int64_t sf_ld, void *workspace, size_t workspace_bytes,
                                 int32_t group, void *stream);

/* Workspace bytes moe_expand_cast_fp4 stages column-major scales in: as
 * moe_expand_cast_fp8_ex_workspace_bytes with G = hidden / group. */
size_t moe_expand_cast_fp4_workspace_bytes(int64_t num_tokens, int32_t hidden, int32_t group,
                                           uint32_t sf_flags);

/*
 * swiglu_cast_fp8 -- [TK] 3.3, plain form (no clamp, no top-k weight).  For
 * each row r and channel c < N, in f32:
 *   g = x[r, c] (left half, the gate), u = x[r, N + c] (right half, up)
 *   v = g / (1 + exp(-g)) * u
 * then the per-128-channel cast of moe_expand_cast_fp8 on v.
 *   x [M, 2N] bf16, 16-byte aligned; out [M, N] u8, 16-byte aligned;
 *   out_sf [M, N/128] f32.
 * Requires N % 128 == 0, group == 128 and M * N/128 < 2^31 (else
 * MOE_ERR_UNSUPPORTED).  exp and the division use the GPU's exp2 and
 * reciprocal units (__expf, __fdividef), so v is within a few ulps of the
 * correctly rounded f32 value, and an E4M3 code can differ by one step from a
 * host evaluation when v / sf lies that close to a rounding midpoint.
 */
moe_status_t swiglu_cast_fp8(const void *x, int64_t num_rows, int32_t n,
                             uint8_t *out, float *out_sf, int32_t group,
                             void *stream);

/*
 * swiglu_cast_fp8_ex -- swiglu_cast_fp8 with the variants of [TK] 3.3 and the
 * scale options of moe_expand_cast_fp8_ex:
 *   has_clamp, clamp: if has_clamp, g = min(g, clamp) and u = min(max(u,
 *              -clamp), clamp) before the activation (clamp >= 0, finite);
 *   weights:   NULL, or [M] f32: v = g / (1 + exp(-g)) * u * weights[r] (the
 *              routed copy's top-k weight, in expert-sorted row order);
 *   clamp_count: NULL, or one u64 in device memory to which the number of
 *              inputs the clamp changed is ADDED (zero it to count one call);
 *   sf_flags, sf_ld: as moe_expand_cast_fp8_ex, over M rows.
 * Requirements as swiglu_cast_fp8.
 */
moe_status_t swiglu_cast_fp8_ex(const void *x, int64_t num_rows, int32_t n, uint8_t *out,
                                void *out_sf, uint32_t sf_flags, int64_t sf_ld,
                                int32_t has_clamp, float clamp, const float *weights,
                                uint64_t *clamp_count, int32_t group, void *stream);

/*
 * swiglu_cast_fp4 -- swiglu_cast_fp8_ex with the FP4 E2M1 output of
 * moe_expand_cast_fp4: the same SwiGLU values (clamp, weight, clamp count),
 * cast per group of `group` channels (16, 32, 64 or 128) with scale
 * max(amax, 6 * 2^-126) / 6 (or its power-of-two round-up), codes packed two
 * per byte, element 2i in the low nibble: out [M][N/2] u8; scales as
 * swiglu_cast_fp8_ex with G = N / group.
 * Requires N % group == 0, N % 32 == 0, x and out 16-byte aligned.
 */
moe_status_t swiglu_cast_fp4(const void *x, int64_t num_rows, int32_t n, uint8_t *out,
                             void *out_sf, uint32_t sf_flags, int64_t sf_ld, int32_t has_clamp,
                             float clamp, const float *weights, uint64_t *clamp_count,
                             int32_t group, void *stream);

/*
 * moe_combine -- [PX] combine: "accumulate in registers using the token
 * positions, then write the final tokens".  For every token t:
 *   out[t, c] = sum_{j=0..k-1, pos[t,j] >= 0} topk_weights[t,j] * y[pos[t,j], c]
 * accumulated in f32 in slot order j = 0..k-1 (fused multiply-add), then
 * rounded to nearest even bf16 (MOE_OUT_BF16) or kept f32 (MOE_OUT_F32).
 *   y   [num_rows, H] bf16, 16-byte aligned (the expert outputs in the
 *       expert-sorted layout moe_route_map produced)
 *   topk_weights [T, k] f32, pos [T, k] i32
 *   out [T, H] bf16 or f32, 16-byte aligned
 * Requires H % 8 == 0 and T * H/8 < 2^31 (else MOE_ERR_UNSUPPORTED).
 * pos >= num_rows sets MOE_DEVERR_POS_RANGE and that copy contributes nothing.
 */
moe_status_t moe_combine(const void *y, const float *topk_weights,
                         const int32_t *pos, int64_t num_tokens, int32_t hidden,
                         int32_t num_topk, int64_t num_rows, void *out,
                         int32_t out_dtype, void *stream);

/*
 * moe_route_expand_cast_fp8 -- steps 1-3 of the path in one call: top-k gate +
 * softmax weights, route map, expand + per-token E4M3 cast, with exactly the
 * results of moe_topk_gate (MOE_WEIGHTS_SOFTMAX_TOPK), moe_route_map and
 * moe_expand_cast_fp8 (num_rows = T*k).
 *
 * The FUSED path is the decode specialisation of "CuTeDSL at Perplexity"
 * (prefill/decode kernels; MoE dispatch): one cooperative launch of one block
 * per SM.  Every warp selects its tokens' experts and every block casts its
 * tokens into shared memory; block 0 then builds the route map once all
 * blocks have arrived on a counter, and signals the others, which write their
 * rows.  Each wait is bounded (1 s); one that runs out sets
 * MOE_DEVERR_TIMEOUT.  It applies to T <= 2048, 32 < E <= 256, k <= 32,
 * T*k <= 16384, H <= 16384 (shared-memory staging permitting).  The
 * REPLICATED path has no wait on another block and no cooperative launch:
 * every block builds the whole route map in its own shared memory, then casts
 * and writes its own tokens' rows (and their pos and sorted_src entries).  For
 * T <= 32 it is one launch in which every block also selects the experts of
 * all T tokens (block 0 writes idx, w, counts and offsets); above, the top-k
 * kernel runs first and a second launch does the rest.  It applies to
 * T <= 2048, T*k <= 16384, 32 < E <= 256, k <= 32, H <= 8192.  The SEPARATE
 * path is the launches of the individual calls (three or four: the route map
 * is one launch for T <= 1024).  The CHAINED path is three launches: the
 * top-k kernel, one CTA per chunk of 16 to 64 consecutive tokens, also counts
 * each chunk's copies per expert and ranks every copy among its expert's
 * copies in the chunk; a scan turns the counts into per-chunk bases, the
 * counts and the offsets; the expand kernel places every copy itself (expert
 * offset + chunk base + rank), writing pos and sorted_src, then stores the
 * rows.  It applies to
 * 32 < E <= 256, k <= 32, H <= 16384 with H/128 % 4 == 0 and 16-byte aligned
 * out and out_sf.
 *   scores [T,E] f32; x [T,H] bf16; topk_idx [T,k] i32; topk_weights [T,k]
 *   f32; counts [E], offsets [E+1], pos [T,k], sorted_src [T*k] i32;
 *   out [T*k,H] u8; out_sf [T*k,H/128] f32.
 *   workspace: at least moe_route_expand_cast_fp8_workspace_bytes(T,E,k)
 *   bytes, 16-byte aligned.  Its first 256 bytes hold the FUSED and CHAINED
 *   paths' control words (the fused launch's arrival counters; the chained
 *   scan's count of finished CTAs): ZERO them once before the first call
 *   (each call leaves them zero; after a MOE_DEVERR_TIMEOUT, zero them
 *   again).  One workspace must not be used by two calls in flight at once.
 *   mode: MOE_PATH_AUTO, MOE_PATH_FUSED, MOE_PATH_REPLICATED or
 *   MOE_PATH_CHAINED (MOE_ERR_UNSUPPORTED where they do not apply) or
 *   MOE_PATH_SEPARATE.  AUTO
 *   takes the path measured fastest on GB300 for the shape: REPLICATED for
 *   T <= MOE_AUTO_REPLICATED_MAX_TOKENS where it applies (E = 256, k = 8,
 *   H = 4096, one call: 8.8 against 14.0 us at T = 16, 12.9 against 14.0 at
 *   T = 256, 15.0 against 16.0 at T = 512, 17.0 against 18.0 at T = 768,
 *   20.1 against 20.1 at T = 1024 (14.2 against 14.6 back to back); at
 *   T = 2048 the separate launches are faster back to back), else SEPARATE
 *   (the separate launches, chained by programmatic dependent launch, were
 *   as fast as the FUSED launch for T <= 64 and faster above: its single
 *   routing block and the cooperative launch cost more than the gaps they
 *   remove; and 1-2 % faster than CHAINED at T = 1024 to 65536: the chained
 *   top-k kernel, the scan and the expand's placement step take longer than
 *   the route map's two launches they replace).
 * Requirements as the individual calls; group == 128.
 */
moe_status_t moe_route_expand_cast_fp8(const float *scores, int64_t num_tokens,
                                       int32_t num_experts, int32_t num_topk, const void *x,
                                       int32_t hidden, int32_t *topk_idx, float *topk_weights,
                                       int32_t *counts, int32_t *offsets, int32_t *pos,
                                       int32_t *sorted_src, uint8_t *out, float *out_sf,
                                       void *workspace, size_t workspace_bytes, int32_t mode,
                                       int32_t group, void *stream);

/* 256 + moe_route_map_workspace_bytes(T, E, k). */
size_t moe_route_expand_cast_fp8_workspace_bytes(int64_t num_tokens, int32_t num_experts,
                                                 int32_t num_topk);

/* Test hooks of the fused path, process-wide, read at each launch:
 *   MOE_DEBUG_WAIT_TIMEOUT_NS: the bound of every wait (default 1e9 ns);
 *   MOE_DEBUG_SKIP_ROUTE_SIGNAL: nonzero = block 0 never signals "routed", so
 *   the copy blocks' waits run out (the failure path, without a fault).
 * Returns MOE_ERR_INVALID_ARG for an unknown key or a value out of range. */
#define MOE_DEBUG_WAIT_TIMEOUT_NS 1
#define MOE_DEBUG_SKIP_ROUTE_SIGNAL 2
moe_status_t moe_debug_set(int32_t key, int64_t value);

/*
 * moe_debug_cvt -- the device's value conversions on arbitrary f32 input, for
 * tests: out[i] = the E4M3FN code (MOE_DEBUG_CVT_E4M3: round to nearest even,
 * saturating at +-448, NaN -> NaN) or the E2M1 code in the low nibble
 * (MOE_DEBUG_CVT_E2M1: round to nearest even, saturating at +-6) of in[i],
 * exactly as the cast kernels convert x * (1 / scale).
 *   in [n] f32, out [n] u8, both 16-byte aligned; n % 4 == 0.
 */
#define MOE_DEBUG_CVT_E4M3 0
#define MOE_DEBUG_CVT_E2M1 1
moe_status_t moe_debug_cvt(int32_t format, const float *in, uint8_t *out, int64_t n,
                           void *stream);

/*
 * moe_peak_copy -- a plain 16-byte vectorised device-to-device copy of
 * `bytes` bytes (a multiple of 16; both pointers 16-byte aligned), used to
 * measure the HBM bandwidth the kernels above are held against.
 */
moe_status_t moe_peak_copy(const void *src, void *dst, size_t bytes, void *stream);

/*
 * moe_get_device_status -- synchronises `stream`, then reads and clears the
 * current device's error word.  Returns MOE_OK when no bit was set,
 * MOE_ERR_DEVICE when one was (the bits go to *error_bits if non-NULL), or
 * MOE_ERR_CUDA if synchronising failed.
 */
moe_status_t moe_get_device_status(void *stream, uint32_t *error_bits);

/* Static description of a status code (never NULL). */
const char *moe_status_string(moe_status_t status);

/* Text of the last CUDA error seen by this library on the calling thread. */
const char *moe_last_cuda_error_string(void);

/* MOE_ROUTE_ABI_VERSION of the loaded library. */
int32_t moe_abi_version(void);

/* Number of kernels this library has launched in this process so far. */
uint64_t moe_kernel_launch_count(void);

/*
 * Debug-bounds build.  The same sources compiled with MOE_DEBUG_BOUNDS
 * defined give libmoe_route_debug.so (the Python binding loads it when the
 * environment variable MOE_DEBUG_BOUNDS is 1).  Its kernels check, before the
 * access each guards, invariants that the normal build takes from the kernels'
 * construction: the alignment, size and shared-memory source of every TMA bulk
 * copy, the alignment of wide scale stores, the shared-memory extent of the
 * staging slots, and the sorted_src row of every copy the decode kernels
 * place.  A failed check skips that access and sets MOE_DEVERR_BOUNDS; no
 * kernel traps.  Results are otherwise identical to the normal build's.
 *
 * moe_debug_bounds_enabled: 1 in the debug-bounds library, 0 otherwise.
 * moe_debug_bounds_selftest: in the debug-bounds library, launches one
 *   kernel whose single check is false by construction (it guards no memory
 *   access), so that the next moe_get_device_status reports
 *   MOE_DEVERR_BOUNDS; returns MOE_OK, or MOE_ERR_CUDA if the launch failed.
 *   In the normal library: MOE_ERR_UNSUPPORTED, nothing launched.
 */
int32_t moe_debug_bounds_enabled(void);
moe_status_t moe_debug_bounds_selftest(void *stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_ROUTE_H */
