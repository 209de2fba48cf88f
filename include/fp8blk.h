/*
 * fp8blk.h -- C ABI of libfp8blk: the GB300 (sm_103a) FP8 block-scaled decode
 * GEMV, its fused greedy argmax, and the NVFP4 routed-expert dequant + GEMV.
 *
 * Conventions for every entry point
 *   - Plain C types only.  `stream` is a cudaStream_t passed as void*
 *     (NULL = the legacy default stream).
 *   - Device pointers are CUDA device (or managed) memory owned by the caller.
 *     The library allocates nothing, frees nothing and never synchronizes:
 *     every GPU entry point only enqueues kernels on `stream` and returns.
 *     Buffers must stay alive until that work has run.
 *   - Arguments are checked on the host before anything is enqueued; on any
 *     error nothing is launched and the return value says why.
 *   - Matrices are row-major and dense (row stride = number of columns).
 *   - Integer sizes are int64_t; the product rows * cols may exceed 2^31.
 *   - Launch contract for e4m3 weight codes (fp8blk_gemv, fp8blk_gemv_argmax,
 *     fp8blk_gemv_argmax_noalloc): kernels are launched with programmatic
 *     dependent launch and start copying the weight codes as soon as they are
 *     resident, which can be before the kernel launched just before them on
 *     the same stream has finished; x, scales and outputs are touched only
 *     after that kernel has completed.  So the codes must not be written by
 *     that immediately preceding kernel (nor by a kernel it lets run
 *     concurrently by triggering its dependents before waiting on its own
 *     predecessors; the library's kernels never do).  Codes written by a copy,
 *     a memset, or any earlier kernel are safe -- weights loaded once at start
 *     up, as the pages' engine keeps them ("Module dsv4_gpu" page, struct
 *     Fp8Dense), always are.  fp8blk_set_launch_tuning(.., use_pdl = 0, ..)
 *     turns the early start off.  bf16 and FP4 weights are read only after
 *     the preceding kernel has completed (the bf16 GEMV's weights can be the
 *     dequant kernel's output).
 *
 * Return codes (int): FP8BLK_OK on success, otherwise one of the codes below;
 * fp8blk_strerror() names them.
 */
#ifndef FP8BLK_H
#define FP8BLK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define FP8BLK_OK 0
#define FP8BLK_EINVAL 1  /* null pointer, size <= 0, m outside [1, 8], column count not a
                            multiple of the format's granule, bad or repeated expert id */
#define FP8BLK_EALIGN 2  /* a pointer is not aligned as documented */
#define FP8BLK_ESCALE 3  /* e8m0 code 0xFF, or an NVFP4 global scale that is not a finite
                            nonzero power of two (the bf16 dequant would not be exact) */
#define FP8BLK_EWS 4     /* workspace missing or smaller than the *_ws_bytes() answer */
#define FP8BLK_ECUDA 5   /* the CUDA runtime refused a launch or attribute call */
#define FP8BLK_ERANGE 6  /* a size is beyond what the kernels index (rows >= 2^31, ...) */

#define FP8BLK_MAX_M 8      /* activation rows per call: 1 (decode) .. 8 (batched verify) */
#define FP8BLK_BLOCK 128    /* side of a square scale block */

/* Bits of the device status word (see fp8blk_device_status). */
#define FP8BLK_STATUS_WAIT_TIMEOUT 1u /* a kernel gave up waiting for a weight tile (bounded
                                         wait, about one second); its outputs are invalid */
#define FP8BLK_STATUS_BAD_EXPERT 2u   /* an expert GEMV met a device-side expert id outside
                                         [0, n_experts) or a global scale that is not a power
                                         of two in [2^-100, 2^100]; that slot's outputs are NaN */

/* Version of this ABI; bumped on any incompatible change. */
int fp8blk_abi_version(void);

/* Human-readable name of a return code (static storage). */
const char *fp8blk_strerror(int code);

/*
 * fp8blk_scales_from_e8m0 -- HOST function: decode an e8m0 block-scale grid
 * to f32, out[k] = 2^(codes[k] - 127).  Source: "Module dsv4_gpu" page,
 * struct Fp8Dense (the 128x128 block-scale grid is decoded to f32 on the host;
 * every e8m0 code is a power of two; 0xFF is refused at load).
 *   codes      host, n bytes
 *   out        host, n floats (code 0 decodes to the f32 subnormal 2^-127)
 *   bad_index  host, optional: on FP8BLK_ESCALE receives the first 0xFF index
 * Returns FP8BLK_ESCALE on any 0xFF code (out is then unspecified), EINVAL on
 * null codes/out with n > 0.
 */
int fp8blk_scales_from_e8m0(const uint8_t *codes, size_t n, float *out, size_t *bad_index);

/*
 * fp8blk_gemv -- y[i][r] = sum_c e4m3(W[r][c]) * S[r/128][c/128] * x[i][c]
 * for i < m, r < rows.  Source: "Module dsv4_gpu" page, struct Fp8Dense (the
 * device GEMV decodes e4m3(code) * scale in-register) and "Struct Dsv4Gpu"
 * page, field dense_fp8 (decode and verify read the FP8-blk linears as stored)
 * and method verify_batch_dev (m = T = k+1 verify rows).
 *   w_codes  device, uint8 e4m3 codes [rows, cols], 16-byte aligned.  NaN codes
 *            (0x7F, 0xFF) are not refused; they make the affected outputs NaN.
 *   scales   device, f32 grid [ceil(rows/128), ceil(cols/128)], 4-byte aligned
 *            (normally the output of fp8blk_scales_from_e8m0).
 *   x        device, f32 activations [m, cols], 16-byte aligned; used as f32.
 *   y        device, f32 outputs [m, rows], 4-byte aligned; fully overwritten.
 *            Must not overlap any input.
 *   m        1..8;  rows >= 1;  cols >= 16 and a multiple of 16.
 * Accumulation is f32 in a fixed order (results are deterministic run to
 * run); each product is formed as e4m3 * (x * S), exact unless x * S leaves
 * the f32 range.  Error bound versus the exact sum: |err| <= 1e-5 * sum|w x|
 * + 1e-6 per output.
 * Errors: EINVAL, EALIGN, ERANGE (rows or cols >= 2^31), ECUDA.
 */
int fp8blk_gemv(const uint8_t *w_codes, const float *scales, const float *x, float *y, int m,
                int64_t rows, int64_t cols, void *stream);

/*
 * fp8blk_gemv_argmax_ws_bytes -- workspace size (bytes) that
 * fp8blk_gemv_argmax needs for this shape.  Returns 0 for invalid shapes.
 */
size_t fp8blk_gemv_argmax_ws_bytes(int m, int64_t rows, int64_t cols);

/*
 * fp8blk_gemv_argmax -- the same GEMV fused with a greedy argmax per
 * activation row: tokens[i] = min{ r : y[i][r] = max_r' y[i][r'] }.
 * Source: "Struct Dsv4Gpu" page, method decode_step_greedy (the argmax runs on
 * the device and only 4 bytes cross back) and method verify_batch_dev (a
 * per-position argmax [T]); "dflash.rs source" page, fn dflash2_walk_greedy
 * (ascending scan with a strict '>': the lowest index wins ties).
 * NaN never wins; -0 and +0 tie; a row with nothing above -inf gives token 0.
 * The token is the argmax of the f32 logits this call computes (the same
 * values written to `logits` when it is given).
 *   logits   device, optional (NULL = not written): f32 [m, rows], 4-aligned
 *   tokens   device, uint32 [m], 4-byte aligned; the caller copies it back
 *   ws       device workspace of at least fp8blk_gemv_argmax_ws_bytes(m, rows,
 *            cols) bytes, 16-byte aligned.  It must be zero-filled once
 *            before its first use; every call leaves it ready for the next.
 *            Calls that share a workspace must be ordered (same stream).
 *   others   as fp8blk_gemv.
 * Errors: as fp8blk_gemv, plus EWS.
 */
int fp8blk_gemv_argmax(const uint8_t *w_codes, const float *scales, const float *x,
                       float *logits, uint32_t *tokens, void *ws, size_t ws_bytes, int m,
                       int64_t rows, int64_t cols, void *stream);

/*
 * fp8blk_gemv_argmax_noalloc -- fp8blk_gemv_argmax for callers that cannot
 * allocate device memory.  No counterpart in the paper: the pages' engine
 * preallocates its own arenas.  This entry point serves callers that cannot
 * hand the library a workspace: code running while a CUDA graph is being
 * captured (no cudaMalloc then), serving loops that must not call
 * cudaMalloc/cudaFree because those synchronize the device, and plain C hosts
 * or plugins that own no allocator.  It computes exactly what
 * fp8blk_gemv_argmax computes, with the workspace placed in a fixed array of
 * fp8blk_noalloc_scratch_bytes() bytes (64.25 KiB) in the library's own device
 * memory; every GPU that loads the library holds that array until the process
 * exits.  It allocates nothing, and calls no cudaMalloc or cudaFree.
 *   Arguments as fp8blk_gemv_argmax, without ws / ws_bytes.
 *   Size limit: the workspace fp8blk_gemv_argmax_ws_bytes(m, rows, cols) must
 *   fit in the array -- any m <= 8 with cols <= 4096; wider rows only for
 *   tiny rows x m.  Larger shapes return FP8BLK_ERANGE.
 *   Set-up: the first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current; make that first call
 *   before any stream capture.
 *   Sharing: every call uses the same array, which keeps the last call's
 *   contents; each call clears the part that must start at zero with a
 *   stream-ordered memset.  Calls whose GPU work overlaps (different streams,
 *   or different host threads) race on the array: serialize them.
 * Errors: as fp8blk_gemv_argmax, with ERANGE in place of EWS.
 */
int fp8blk_gemv_argmax_noalloc(const uint8_t *w_codes, const float *scales, const float *x,
                               float *logits, uint32_t *tokens, int m, int64_t rows, int64_t cols,
                               void *stream);

/* Size in bytes of the fixed device array fp8blk_gemv_argmax_noalloc uses. */
size_t fp8blk_noalloc_scratch_bytes(void);

/*
 * fp8blk_bf16_gemv -- y[i][r] = sum_c bf16(B[r][c]) * x[i][c], f32
 * accumulation.  The GEMV that follows the per-expert dequant.  Source:
 * "Module dsv4_gpu" page, module header (bf16 GEMMs with f32 accumulation)
 * and enum ExpertArm (Bf16Dequant).  x stays f32.
 *   w_bf16   device, bf16 bit patterns [rows, cols], 16-byte aligned
 *   x, y, m  as fp8blk_gemv;  cols >= 16 and a multiple of 16.
 * Errors: EINVAL, EALIGN, ERANGE, ECUDA.
 */
int fp8blk_bf16_gemv(const uint16_t *w_bf16, const float *x, float *y, int m, int64_t rows,
                     int64_t cols, void *stream);

/*
 * nvfp4_expert_dequant -- dequantise one NVFP4 expert to bf16:
 *   out[r][c] = bf16( e2m1(q[r][c]) * e4m3(s[r][c/16]) * g[e] ),
 * exact in bf16 (the host refuses global scales for which it would not be).
 * Source: "Module dsv4_gpu" page, module header and enum ExpertArm (routed
 * experts stay NVFP4 as stored and each activated expert is dequantised into a
 * reused bf16 scratch, exact in bf16) and enum ExpertKind (trunk = NVFP4).
 *   codes        device, uint8 [n_experts, rows, cols/2], two e2m1 codes per
 *                byte, column 2j in the LOW nibble; 16-byte aligned
 *   scales       device, uint8 e4m3 [n_experts, rows, cols/16], 2-byte aligned
 *   gscale_host  HOST, f32 [n_experts]: per-expert global scale, each a finite
 *                nonzero power of two (else ESCALE)
 *   expert_id    0 <= expert_id < n_experts
 *   out          device, uint16 bf16 bits [rows, cols], 16-byte aligned
 *   cols         a multiple of 32.
 * Errors: EINVAL, EALIGN, ESCALE, ERANGE, ECUDA.
 */
int nvfp4_expert_dequant(const uint8_t *codes, const uint8_t *scales, const float *gscale_host,
                         int n_experts, int expert_id, uint16_t *out, int64_t rows, int64_t cols,
                         void *stream);

/*
 * nvfp4_expert_dequant_gemv -- for k < n_active: dequantise expert
 * ids_host[k] into the reused bf16 scratch, then y[k] = scratch x.
 * Same sources as nvfp4_expert_dequant.  The scratch is reused in stream
 * order; when the call's work has run it holds the LAST active expert.
 *   ids_host     HOST, int32 [n_active], distinct, each in [0, n_experts)
 *   n_active     >= 1
 *   x            device, f32 [cols], 16-byte aligned
 *   y            device, f32 [n_active, rows], 4-byte aligned
 *   bf16_scratch device, uint16 [rows, cols], 16-byte aligned
 *   others       as nvfp4_expert_dequant.
 * Errors: as nvfp4_expert_dequant.
 */
int nvfp4_expert_dequant_gemv(const uint8_t *codes, const uint8_t *scales,
                              const float *gscale_host, int n_experts, const int32_t *ids_host,
                              int n_active, const float *x, float *y, uint16_t *bf16_scratch,
                              int64_t rows, int64_t cols, void *stream);

/*
 * nvfp4_expert_gemv -- y[k] = W(ids[k]) x for k < n_active in ONE launch,
 * with no bf16 scratch:
 *   y[k][r] = sum_c bf16(e2m1(q[e][r][c]) * e4m3(s[e][r][c/16]) * g[e]) * x[c],
 *   e = ids[k]; every product is exact, so the weights take the same values
 *   as nvfp4_expert_dequant writes; the sum is in f32.  Two kernels
 *   (fp8blk_set_fp4_kernel; by shape, the tensor cores from 12288 active rows
 *   on): the CUDA cores decode the weights in registers; the tensor cores take
 *   the codes as stored, x as five e4m3 planes per 16-column block (2^-20 of
 *   each element), and apply the block scales to the f32 block sums.  Both
 *   meet the GEMV error bound and are bit-identical run to run.
 * Source: "Module dsv4_gpu" page, module header (routed experts stay NVFP4 as
 * stored; one-launch-per-projection indirect expert dispatch) and enum
 * ExpertArm.  The router's output stays on the device: ids and global scales
 * are read by the kernel, so the host checks neither.
 *   codes, scales as nvfp4_expert_dequant, but scales 16-byte aligned
 *   gscale       DEVICE, f32 [n_experts], 4-byte aligned: per-expert global
 *                scale, a power of two in [2^-100, 2^100]
 *   ids          DEVICE, int32 [n_active], 4-byte aligned; repeats allowed
 *   n_active     1 .. 65536
 *   x            device, f32 [cols], 16-byte aligned
 *   y            device, f32 [n_active, rows], 4-byte aligned
 *   cols         a multiple of 256 (so every scale row starts on 16 bytes).
 * An id outside [0, n_experts) or an unusable global scale sets
 * FP8BLK_STATUS_BAD_EXPERT in the device status word and makes y[k] NaN.
 * An inf or NaN in x: the CUDA cores give the IEEE result, the tensor cores
 * NaN in every output.
 * Errors: EINVAL, EALIGN, ERANGE, ECUDA.
 */
int nvfp4_expert_gemv(const uint8_t *codes, const uint8_t *scales, const float *gscale, int n_experts,
                      const int32_t *ids, int n_active, const float *x, float *y, int64_t rows, int64_t cols,
                      void *stream);

/*
 * mxfp4_expert_gemv -- as nvfp4_expert_gemv, for OCP MXFP4 experts (the MTP
 * block's routed experts, "Module dsv4_gpu" page, enum ExpertKind):
 *   y[k][r] = sum_c e2m1(q[e][r][c]) * 2^(s[e][r][c/32] - 127) * x[c], e = ids[k].
 * Same two kernels and routing as nvfp4_expert_gemv (fp8blk_set_fp4_kernel);
 * on the tensor cores x is split into five e4m3 planes per 32-column block and
 * each 32-column block sum is scaled by its e8m0 factor.
 * The page names the format only; the layout is read from the OCP MX format:
 *   codes        device, uint8 [n_experts, rows, cols/2], two e2m1 codes per
 *                byte, column 2j in the LOW nibble; 16-byte aligned
 *   scales       device, uint8 e8m0 [n_experts, rows, cols/32], 16-byte
 *                aligned; code 0xFF is the MX NaN (its block's weights are NaN)
 *   ids          DEVICE, int32 [n_active]; repeats allowed
 *   cols         a multiple of 512 (so every scale row starts on 16 bytes).
 * No global scale.  An id outside [0, n_experts) sets
 * FP8BLK_STATUS_BAD_EXPERT and makes y[k] NaN.  An inf or NaN in x: the
 * CUDA cores give the IEEE result, the tensor cores NaN in every output.
 * Errors: EINVAL, EALIGN, ERANGE, ECUDA.
 */
int mxfp4_expert_gemv(const uint8_t *codes, const uint8_t *scales, int n_experts, const int32_t *ids,
                      int n_active, const float *x, float *y, int64_t rows, int64_t cols, void *stream);

/*
 * fp8blk_set_launch_tuning -- process-wide launch-shape knobs for the
 * streaming GEMV kernels.  They change speed only: every output is reduced in
 * an order fixed by the column panel layout, so results are bit-identical
 * under any setting.  Pass 0 for a knob's default.
 *   target_stage_bytes  weight bytes per shared-memory pipeline stage (32 KiB)
 *   ctas_per_sm         resident CTAs per SM, 1..4 (2 for m <= 4, else 1)
 *   use_pdl             programmatic dependent launch on (nonzero) or off
 *   l2_prefetch         L2 prefetch, before the grid dependency wait, of the
 *                       stages after the first ring (e4m3) or of the first
 *                       stages (bf16), and of each CTA's first 192 KiB of
 *                       weight rows (tensor-core kernel), on (nonzero) or off
 *   max_stages          pipeline depth cap, 2..8 (8)
 * Not thread-safe against concurrent calls of the other entry points.
 * Errors: EINVAL.
 */
int fp8blk_set_launch_tuning(int target_stage_bytes, int ctas_per_sm, int use_pdl, int l2_prefetch,
                             int max_stages);

/*
 * fp8blk_set_wait_limit -- process-wide limit (nanoseconds, 0 ..
 * FP8BLK_WAIT_LIMIT_DEFAULT_NS) on how long a kernel thread of the CUDA-core
 * GEMVs (fp8blk_gemv / fp8blk_gemv_argmax below the tensor-core thresholds,
 * fp8blk_bf16_gemv, nvfp4_expert_gemv, mxfp4_expert_gemv) waits for a weight
 * tile before it gives up, sets FP8BLK_STATUS_WAIT_TIMEOUT and returns.  The
 * default is about one second; a healthy tile lands in microseconds, so any
 * shorter limit is for exercising the failure path (0 gives up on the first
 * tile that has not landed yet).  After a give-up the CTA still waits, with
 * the fixed one-second bound, for the copies it has in flight before it
 * exits, and still takes part in the argmax hand-off, so the workspace stays
 * consistent; the outputs of that call are invalid.  The tensor-core kernel
 * and the dequant kernel keep the fixed bound.  Not thread-safe against
 * concurrent calls of the other entry points.  Errors: EINVAL.
 */
#define FP8BLK_WAIT_LIMIT_DEFAULT_NS 1000000000ll
int fp8blk_set_wait_limit(int64_t limit_ns);

/*
 * fp8blk_set_m1_kernel -- which kernel serves m = 1 (speed only; results are
 * identical to within the stated error bound, and bit-identical run to run):
 *   choice 0 = by size (e4m3 from the tensor-core threshold of
 *   fp8blk_set_tensor_core_min_m, 48 MiB by default: the tensor-core kernel;
 *   otherwise -- below it, or a shape the tensor-core kernel does not take --
 *   row-per-warp when rows * cols * bytes_per_weight >= rowwarp_min_bytes,
 *   0 = default 96 MiB; the team kernel below that),
 *   1 = always row-per-warp, 2 = always the team kernel (both skip the tensor
 *   cores).  Errors: EINVAL.
 */
int fp8blk_set_m1_kernel(int choice, int64_t rowwarp_min_bytes);

/*
 * fp8blk_set_fp4_kernel -- which kernel serves nvfp4_expert_gemv and
 * mxfp4_expert_gemv (speed only;
 * both are within the stated error bound, each bit-identical run to run):
 *   0 = by shape: the tensor cores from 12288 active rows (n_active x rows)
 *   on, the CUDA cores below; 1 = CUDA cores (weights decoded to f32 in
 *   registers, one f32 FMA each); 2 = tensor cores (the e2m1 codes fed to
 *   tcgen05.mma kind::f8f6f4 as stored, x as five e4m3 planes per scale
 *   block -- 16 columns NVFP4, 32 MXFP4 -- the block scales applied to the
 *   f32 block sums).  The tensor cores also need 32-byte-aligned codes and
 *   room in shared memory for x's planes (16 bytes per column) beside four
 *   code stages (cols up to 4608 with 128-row slabs, more with shorter ones),
 *   else the CUDA cores serve the call; with an inf or NaN in x they return
 *   NaN in every output, the CUDA cores the IEEE result.
 *   Errors: EINVAL.
 */
int fp8blk_set_fp4_kernel(int choice);

/*
 * fp8blk_set_tensor_core_min_m -- route e4m3 GEMVs with m >= min_m activation
 * rows (1..8; 9 = never; 0 = the library default, 1) and at least min_bytes
 * of weights (rows * cols; 1 = any size; 0 = the library default, which
 * depends on m: 24 MiB for m >= 5, 32 MiB for m = 3..4, 48 MiB for m = 1..2) to
 * the tensor-core kernel ("Struct Dsv4Gpu" page, verify_batch_dev: the k+1
 * rows of a speculative verify; decode_step_greedy: the vocab head).  That
 * kernel feeds the stored e4m3 codes to the tensor cores unchanged, splits
 * x * S (S the 128-row tile's block scale) into five e4m3 planes with one
 * exponent per activation row and tile, and accumulates in f32 in tensor
 * memory.  The result stays within the e4m3 GEMV error bound but is not
 * bit-identical to the CUDA-core kernels.  Only for 128 <= cols <= 32768.
 * Speed only; process-wide; not thread-safe against concurrent calls of the
 * other entry points.  Errors: EINVAL.
 */
int fp8blk_set_tensor_core_min_m(int min_m, int64_t min_bytes);

/*
 * fp8blk_plan_query -- HOST, no CUDA calls: the launch geometry the streaming
 * GEMV would use for this shape on a device with the given SM count and
 * shared-memory limits (bytes), for inspection and bounds checks.
 *   bytes_per_weight  1 (e4m3) or 2 (bf16)
 *   out  host int64[13]: panels, panel_cols, team_warps, teams, row_batches,
 *        rows_per_batch, stage_rows, stage_bytes, stages, ctas_per_sm,
 *        n_groups, dynamic_smem_bytes, kernel (0 = team kernel, 1 = row-per-warp
 *        kernel (m = 1, large matrices); for kernel 1, stage_bytes and stages
 *        describe each warp's private ring and teams = warps per CTA)
 * Errors: EINVAL (bad shape or device facts).
 */
int fp8blk_plan_query(int m, int64_t rows, int64_t cols, int bytes_per_weight, int sms,
                      int smem_per_sm, int smem_per_block, int64_t *out);

/*
 * fp8blk_device_status -- read (and optionally clear) the library's device
 * status word on the current device (FP8BLK_STATUS_* bits; 0 = healthy).
 * SYNCHRONIZES the current device.  status_out is a host pointer.
 * Errors: EINVAL, ECUDA.
 */
int fp8blk_device_status(uint32_t *status_out, int clear);

#ifdef __cplusplus
}
#endif

#endif /* FP8BLK_H */
