/*
 * sage_gb300.h - C ABI of the GB300 (sm_103a) quantized attention library.
 *
 * The library computes the data-parallel hot path of SageAttention-2-style
 * quantized attention and of int8 KV-cache prompt attention.  Everything runs
 * in the library's own CUDA kernels on the caller's stream.
 *
 * Conventions for every entry point:
 *  - All tensor pointers are DEVICE pointers owned by the caller.  The library
 *    allocates no device memory and never synchronises the stream.  Scratch
 *    memory, where an entry point needs some, is passed in by the caller; its
 *    size comes from the matching *_workspace() query.  The one exception,
 *    sage_quantize_qk_noalloc, uses a fixed scratch array held by the library.
 *  - `stream` is a cudaStream_t passed as an opaque pointer (NULL = the legacy
 *    default stream).  Work is enqueued asynchronously.
 *  - Argument errors are detected on the host before anything is launched and
 *    are returned as SAGE_ERR_INVALID_ARG or SAGE_ERR_UNSUPPORTED; nothing is
 *    written in that case.  A failed launch returns SAGE_ERR_CUDA.
 *  - `status_dev`, where present, may be NULL.  Otherwise it is a device int32
 *    that kernels set (atomically, never clear) to a non-zero sage_status when
 *    they detect a condition on the device, e.g. SAGE_ERR_TIMEOUT when a
 *    bounded wait inside a kernel ran out.  The caller zeroes it and reads it
 *    after synchronising.
 *  - Head dimension d must be 128.  Element strides describe [B, H, N, d]
 *    tensors whose channel stride is 1; every stride and base pointer must be
 *    16-byte aligned (strides are multiples of 8 elements for bf16).
 *  - Inputs must be finite.  The functions hold no global state (except the
 *    scratch array of sage_quantize_qk_noalloc, and the six CUDA events that
 *    sage_attention_host creates per calling thread and device context on its
 *    first call and reuses afterwards) and may be called from several host
 *    threads.
 *
 * Citations name the page and its section that defines each operation.
 */
#ifndef SAGE_GB300_H
#define SAGE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int sage_status;
#define SAGE_OK 0
#define SAGE_ERR_INVALID_ARG 1  /* null/misaligned pointer, bad size or stride   */
#define SAGE_ERR_UNSUPPORTED 2  /* d != 128, block size not 64/128, and the like  */
#define SAGE_ERR_CUDA 3         /* a CUDA call or kernel launch failed            */
#define SAGE_ERR_WORKSPACE 4    /* workspace smaller than the *_workspace() size  */
#define SAGE_ERR_TIMEOUT 5      /* device side: a bounded wait ran out            */
#define SAGE_ERR_TOO_LARGE 6    /* beyond the fixed scratch of sage_quantize_qk_noalloc */
#define SAGE_ERR_NONFINITE 7    /* device side: a non-finite input or scale       */

#define SAGE_DTYPE_BF16 0
#define SAGE_DTYPE_F32 1

/* Element strides of a [B, H, N, 128] tensor (channel stride is 1). */
typedef struct {
    int64_t b, h, n;
} sage_strides;

/* Human-readable name of a status code (static storage, never NULL). */
const char *sage_status_string(sage_status s);

/* Version of this ABI (bumped on any incompatible change). */
int sage_abi_version(void);

/* ------------------------------------------------------------------------
 * sage_quantize_qk - K smoothing, then INT8 per-block quantisation of Q and
 * of the smoothed K.
 *
 * Defines: "H3 Performance Roadmap", section "Measured GB10 Baseline", table
 * "SageAttention 2.2.0 internals" (rows "Q/K INT8 quantization" and "K
 * smoothing"), and section "Phase 4: Dense Sage-Compatible Attention", items
 * 2-3 (keep the per-block INT8 Q/K policy and K smoothing).
 *
 * Computes, per (b, h):
 *   k_mean[c]  = mean of K[t, c] over t < Nk: tokens summed in ascending
 *                order in fp32 inside chunks of 256, chunk sums added in
 *                ascending order in fp32, the total divided by Nk;
 *   Ks         = fl(K - k_mean)  (fp32);
 *   per block of `q_block` (`k_block`) tokens, the last one partial:
 *   scale      = fl(amax / 127), amax = max |x| over the block;
 *   code       = clamp(rint_even(fl(x * fl(127 / amax))), -127, 127),
 *                0 everywhere when amax = 0.
 * Inputs : q_bf16 [B,H,Nq,128] with strides qs; k_bf16 [B,H,Nk,128] with ks.
 * Outputs (contiguous): q_codes int8 [B,H,Nq,128]; q_scales fp32
 *   [B,H,ceil(Nq/q_block)]; k_codes int8 [B,H,Nk,128]; k_scales fp32
 *   [B,H,ceil(Nk/k_block)]; k_mean fp32 [B,H,128].
 * q_block, k_block in {64, 128}.  Nq, Nk >= 1.  Workspace: at least
 * sage_quantize_qk_workspace(B, H, Nk) bytes, 16-byte aligned.
 * ---------------------------------------------------------------------- */
size_t sage_quantize_qk_workspace(int B, int H, int Nk);
sage_status sage_quantize_qk(const void *q_bf16, sage_strides qs, const void *k_bf16, sage_strides ks,
                             int B, int H, int Nq, int Nk, int d, int q_block, int k_block,
                             int8_t *q_codes, float *q_scales, int8_t *k_codes, float *k_scales,
                             float *k_mean, void *workspace, size_t workspace_bytes, void *stream);

/* ------------------------------------------------------------------------
 * sage_quantize_qk_noalloc - the same computation and outputs as
 * sage_quantize_qk, for callers that cannot allocate device memory.
 *
 * The pages have no counterpart of this entry point; it exists for callers
 * that must not allocate: a serving engine that reserves all of HBM at start
 * and hands out fixed buffers, a plug-in whose host framework owns every
 * device allocation, or a latency-bound loop where a cudaMalloc (which may
 * synchronise the device) is not allowed.  Such a caller still passes its
 * inputs and outputs; only the scratch is taken care of here.
 *
 * Scratch: a static device array of SAGE_QK_NOALLOC_SCRATCH_BYTES (8 MiB)
 * inside the library, held by every GPU that loads the library until the
 * process exits.  It holds the K-mean chunk partials, B*H*ceil(Nk/256)*128
 * fp32 values, so B*H*ceil(Nk/256) <= 16384 (for example 24 heads up to
 * 174,848 keys); larger problems return SAGE_ERR_TOO_LARGE and launch nothing.
 * Each call writes every partial it later reads, so nothing needs clearing
 * between calls.  All calls on a device share the one array: calls whose
 * kernels overlap on the GPU (different streams, or different host threads)
 * race on it and must be serialised by the caller.
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current), and so does the first
 * call after the device's context was destroyed and created anew (e.g. by
 * cudaDeviceReset, which reloads the library's device code); make those
 * calls before any stream capture.  Allocates nothing: no cudaMalloc or
 * cudaFree.
 * ---------------------------------------------------------------------- */
#define SAGE_QK_NOALLOC_SCRATCH_BYTES (8u << 20)
sage_status sage_quantize_qk_noalloc(const void *q_bf16, sage_strides qs, const void *k_bf16,
                                     sage_strides ks, int B, int H, int Nq, int Nk, int d, int q_block,
                                     int k_block, int8_t *q_codes, float *q_scales, int8_t *k_codes,
                                     float *k_scales, float *k_mean, void *stream);

/* ------------------------------------------------------------------------
 * sage_quantize_qkv - the whole preparation of the dense path (what
 * sage_quantize_qk and sage_quantize_v compute) in three launches for all
 * heads: one reduction pass over K and V (K chunk sums, V channel maxima),
 * one finalisation (K mean, V scales), one encoding pass over Q, K and V.
 *
 * Defines: the same steps as sage_quantize_qk and sage_quantize_v ("H3
 * Performance Roadmap", table "SageAttention 2.2.0 internals"), fused as
 * "Phase 4: Dense Sage-Compatible Attention", item 4 asks (fuse the Q/K/V
 * preparation where profitable).
 *
 * Codes, scales, the K mean and the V codes are bit for bit those of the two
 * separate entry points.  qk_format selects how the Q/K codes are stored:
 *   SAGE_QK_INT8: int8 [B,H,N,128] (as sage_quantize_qk);
 *   SAGE_QK_F16:  the codes' exact fp16 images [B,H,N,128] (every code is
 *                 an integer of magnitude <= 127), the operand layout the
 *                 attention's tensor cores read: sage_attn_fwd_f16 takes
 *                 them with no conversion pass.
 * q_out, k_out: contiguous, int8 or fp16 as selected; q_scales, k_scales,
 * k_mean, v_codes, v_scales as in sage_quantize_qk / sage_quantize_v.
 * Workspace: at least sage_quantize_qkv_workspace(B, H, Nk) bytes.
 * ---------------------------------------------------------------------- */
#define SAGE_QK_INT8 0
#define SAGE_QK_F16 1
size_t sage_quantize_qkv_workspace(int B, int H, int Nk);
sage_status sage_quantize_qkv(const void *q_bf16, sage_strides qs, const void *k_bf16, sage_strides ks,
                              const void *v_bf16, sage_strides vs, int B, int H, int Nq, int Nk, int d, int q_block,
                              int k_block, int qk_format, void *q_out, float *q_scales, void *k_out, float *k_scales,
                              float *k_mean, uint8_t *v_codes, float *v_scales, void *workspace,
                              size_t workspace_bytes, void *stream);

/* ------------------------------------------------------------------------
 * sage_quantize_v - FP8 E4M3 per-channel quantisation of V, written
 * transposed for the P.V product.
 *
 * Defines: "H3 Performance Roadmap", section "Measured GB10 Baseline", table
 * "SageAttention 2.2.0 internals" (row "V FP8 quantization") and the
 * uninstrumented phase list of the Sage2 decomposition ("V transpose/
 * quantization").
 *
 * Per (b, h, channel c): amax_c = max_t |V[t, c]|; v_scales[c] = fl(amax_c/448);
 * code = e4m3_rn_satfinite(fl(V * fl(448/amax_c))) (OCP E4M3, largest finite
 * 448), 0 when amax_c = 0.
 * Input : v_bf16 [B,H,Nk,128] with strides vs.
 * Outputs (contiguous): v_codes uint8 [B,H,128,Nk_pad] with
 *   Nk_pad = ceil(Nk/128)*128 and codes 0 for tokens >= Nk;
 *   v_scales fp32 [B,H,128].
 * Workspace: at least sage_quantize_v_workspace(B, H, Nk) bytes.
 * ---------------------------------------------------------------------- */
size_t sage_quantize_v_workspace(int B, int H, int Nk);
sage_status sage_quantize_v(const void *v_bf16, sage_strides vs, int B, int H, int Nk, int d,
                            uint8_t *v_codes, float *v_scales, void *workspace,
                            size_t workspace_bytes, void *stream);

/* ------------------------------------------------------------------------
 * sage_attn_fwd - non-causal quantized attention forward over the outputs of
 * sage_quantize_qk / sage_quantize_v.
 *
 * Defines: "Sage2 SM89 Temporal Pair Experiment", section "Candidate" (per
 * KV tile the order QK -> online-softmax update of m, d, O -> accumulate the
 * denominator -> scores to FP8 -> PV; V scale fused into the epilogue, kernel
 * name "..._fuse_v_scale_attn_inst_buf"), and "H3 Performance Roadmap",
 * section "Phase 4: Dense Sage-Compatible Attention".
 *
 * For each query row i and 128-key tile (ascending):
 *   S = q_codes . k_codes (exact int32), s = S * fl(fl(sq*sk) * C) with
 *   C = fl(sm_scale * log2 e); m' = max(m, max s); alpha = 2^(m - m');
 *   p = 2^(s - m'); l = alpha*l + sum p (fp32 p); P = e4m3(448 p);
 *   O = alpha*O + P.V (fp32 accumulate); out = bf16(O / l * v_scale / 448).
 * Inputs: codes/scales as written by the two quantisers (q_block, k_block
 *   must match), Nk_pad as there.  sm_scale <= 0 selects 1/sqrt(128).
 * Output: out_bf16 [B,H,Nq,128] with element strides os.
 * Workspace: at least sage_attn_fwd_workspace(B, H, Nq, Nk) bytes (fp16
 *   images of the int8 codes for the tensor cores).
 * ---------------------------------------------------------------------- */
size_t sage_attn_fwd_workspace(int B, int H, int Nq, int Nk);
sage_status sage_attn_fwd(const int8_t *q_codes, const float *q_scales, const int8_t *k_codes,
                          const float *k_scales, const uint8_t *v_codes, const float *v_scales,
                          int B, int H, int Nq, int Nk, int d, int q_block, int k_block,
                          float sm_scale, void *out_bf16, sage_strides os, void *workspace,
                          size_t workspace_bytes, int32_t *status_dev, void *stream);

/* ------------------------------------------------------------------------
 * sage_attn_fwd_ex - sage_attn_fwd with two options the pages name as the
 * next steps of the dense path ("H3 Performance Roadmap", "Phase 4: Dense
 * Sage-Compatible Attention"): a causal mask and the per-row log-sum-exp.
 *   causal: 0 or 1.  With 1, query i sees keys j <= i + (Nk - Nq) (the last
 *           query sees every key; for Nq == Nk, j <= i).  Requires Nq <= Nk,
 *           else SAGE_ERR_UNSUPPORTED.
 *   lse:    NULL, or fp32 [B][H][Nq] (contiguous, 4-byte aligned): the natural
 *           log of sum_j exp(s_ij) over the row's visible keys, s the scaled
 *           logits sm_scale * q.k of the quantized program.
 * Everything else as sage_attn_fwd (which equals causal = 0, lse = NULL).
 * ---------------------------------------------------------------------- */
sage_status sage_attn_fwd_ex(const int8_t *q_codes, const float *q_scales, const int8_t *k_codes,
                             const float *k_scales, const uint8_t *v_codes, const float *v_scales,
                             int B, int H, int Nq, int Nk, int d, int q_block, int k_block, float sm_scale,
                             int causal, void *out_bf16, sage_strides os, float *lse, void *workspace,
                             size_t workspace_bytes, int32_t *status_dev, void *stream);

/* ------------------------------------------------------------------------
 * sage_attn_fwd_f16 - sage_attn_fwd_ex over the exact fp16 images of the
 * Q/K codes (as sage_quantize_qkv writes them with SAGE_QK_F16) instead of
 * the int8 codes: the same attention kernel and result, without the two
 * conversion passes and without a workspace.  Page and computation as
 * sage_attn_fwd ("Sage2 SM89 Temporal Pair Experiment", section
 * "Candidate").
 *   q_f16 [B,H,Nq,128], k_f16 [B,H,Nk,128]: contiguous fp16 images, 16-byte
 *   aligned; everything else as sage_attn_fwd_ex.
 * ---------------------------------------------------------------------- */
sage_status sage_attn_fwd_f16(const void *q_f16, const float *q_scales, const void *k_f16, const float *k_scales,
                              const uint8_t *v_codes, const float *v_scales, int B, int H, int Nq, int Nk, int d,
                              int q_block, int k_block, float sm_scale, int causal, void *out_bf16, sage_strides os,
                              float *lse, int32_t *status_dev, void *stream);

/* ------------------------------------------------------------------------
 * sage_attention - the dense path (sage_quantize_qk, sage_quantize_v,
 * sage_attn_fwd_ex) in one call on device buffers, for callers that do not
 * keep the codes: the three steps in a row on one stream, their
 * intermediates in the workspace.  The result is bit for bit that of the
 * three entry points called in a row.  The steps are those of the table
 * "SageAttention 2.2.0 internals" ("H3 Performance Roadmap", section
 * "Measured GB10 Baseline": K smoothing, Q/K INT8 quantization, V FP8
 * quantization, attention forward).
 *   q, k, v, out, strides, sizes, blocks, sm_scale, causal, lse: as in
 *     sage_quantize_qk, sage_quantize_v and sage_attn_fwd_ex.
 *   workspace: device memory of sage_attention_workspace(B, H, Nq, Nk)
 *     bytes: codes, scales and means of all heads and the three entry
 *     points' own workspaces.
 * Errors as the three entry points, all checked before the first step is
 * enqueued.
 * ---------------------------------------------------------------------- */
size_t sage_attention_workspace(int B, int H, int Nq, int Nk);
sage_status sage_attention(const void *q_bf16, sage_strides qs, const void *k_bf16, sage_strides ks,
                           const void *v_bf16, sage_strides vs, int B, int H, int Nq, int Nk, int d, int q_block,
                           int k_block, float sm_scale, int causal, void *out_bf16, sage_strides os, float *lse,
                           void *workspace, size_t workspace_bytes, int32_t *status_dev, void *stream);

/* ------------------------------------------------------------------------
 * sage_attention_host - the dense path (sage_quantize_qk, sage_quantize_v,
 * sage_attn_fwd_ex) on HOST buffers, with the host<->device copies and the
 * quantizers of one group of heads overlapped with the attention of another.
 * The (batch, head) problems are independent ("H3 Performance Roadmap",
 * section "Phase 4: Dense Sage-Compatible Attention": one dense attention per
 * head), so the B*H heads are cut into chunks of up to head_chunk heads
 * (1, 2, 4, ... at the start and the end); the copy stream moves chunk c+2
 * in, chunk c out and quantizes chunk c+2 while the compute stream runs the
 * attention of chunk c+1.
 *   q_host, out_host: bf16 [B][H][Nq][128] contiguous; k_host, v_host: bf16
 *     [B][H][Nk][128] contiguous.  Page-locked memory lets the copies overlap
 *     the kernels (pageable memory works, without overlap).
 *   head_chunk >= 1: heads per chunk (the last chunk may be smaller).
 *   causal: 0 or 1 as in sage_attn_fwd_ex (no lse here).
 *   workspace: device memory of sage_attention_host_workspace(B, H, Nq, Nk,
 *     head_chunk) bytes (double-buffered bf16 chunks, codes, scales and
 *     quantizer workspaces, one attention workspace); shared by successive
 *     calls.
 *   compute_stream, copy_stream: two different streams (the copy stream
 *     also runs the quantizer kernels).  Everything is
 *     enqueued asynchronously; out_host is complete once compute_stream has
 *     reached the end of the call (it waits for the last copy).  The copies
 *     start after the work already queued on compute_stream.  The two streams
 *     are ordered by six events that the calling thread keeps for its current
 *     device context (created by the first call, reused by every later one).
 * Errors as the three entry points; SAGE_ERR_INVALID_ARG for a null pointer,
 * head_chunk < 1 or equal streams.  After an error, work already enqueued may
 * still run: synchronise both streams before reusing the buffers.
 * ---------------------------------------------------------------------- */
size_t sage_attention_host_workspace(int B, int H, int Nq, int Nk, int head_chunk);
sage_status sage_attention_host(const void *q_host, const void *k_host, const void *v_host, void *out_host, int B,
                                int H, int Nq, int Nk, int d, int q_block, int k_block, float sm_scale, int causal,
                                int head_chunk, void *workspace, size_t workspace_bytes, int32_t *status_dev,
                                void *compute_stream, void *copy_stream);

/* ------------------------------------------------------------------------
 * sage_attn_fwd_scores_dump - sage_attn_fwd that also writes, for checking,
 * every exact integer score S = q_codes . k_codes^T the tensor cores produced
 * for the attention (the Q.K^T of the defining passage above), as int32 into
 * s_dump [B*H][Nq_pad][Nk_pad] with Nq_pad = ceil(Nq/256)*256 and
 * Nk_pad = ceil(Nk/128)*128 (entries past Nq or Nk are scores against zero
 * rows).  Diagnostic only: the dump costs a full write of S and is meant for
 * small problems.  s_dump must be 16-byte aligned.
 * ---------------------------------------------------------------------- */
sage_status sage_attn_fwd_scores_dump(const int8_t *q_codes, const float *q_scales, const int8_t *k_codes,
                                      const float *k_scales, const uint8_t *v_codes, const float *v_scales,
                                      int B, int H, int Nq, int Nk, int d, int q_block, int k_block,
                                      float sm_scale, void *out_bf16, sage_strides os, void *workspace,
                                      size_t workspace_bytes, int32_t *status_dev, int32_t *s_dump,
                                      void *stream);

/* ------------------------------------------------------------------------
 * sage_attn_fwd_fault_test - exercises the failure detection of
 * sage_attn_fwd: the same launch, except that the kernel's load warp stops
 * early, so the other warps' bounded waits run out after wait_limit_ns.
 *   mode 1: the load warp issues no copy at all;
 *   mode 2: it loads the query tiles and the first key tile, then stops, so
 *           copies and MMAs are issued before the waits give up.
 * Every CTA then stops its loops, waits for the copies and MMAs it already
 * issued, frees its tensor memory and returns; the kernel sets *status_dev
 * to SAGE_ERR_TIMEOUT.  Nothing faults, traps or hangs, and the CUDA context
 * stays usable.  The output is not written.  status_dev must not be NULL;
 * wait_limit_ns > 0; mode 1 or 2.  Test hook only.
 * ---------------------------------------------------------------------- */
sage_status sage_attn_fwd_fault_test(const int8_t *q_codes, const float *q_scales, const int8_t *k_codes,
                                     const float *k_scales, const uint8_t *v_codes, const float *v_scales,
                                     int B, int H, int Nq, int Nk, int d, int q_block, int k_block,
                                     float sm_scale, void *out_bf16, sage_strides os, void *workspace,
                                     size_t workspace_bytes, int32_t *status_dev, uint64_t wait_limit_ns,
                                     int mode, void *stream);

/* ------------------------------------------------------------------------
 * int8kv_prompt_attn - causal prompt attention of bf16 queries over an int8
 * KV cache with per-token fp16 scales, grouped-query heads.
 *
 * Defines: "Strata PR #2092" (sm_75 v2 int8 prompt attention), its
 * description (chunked prompt attention over the int8 KV cache, per-chunk
 * K/V staging with their scales) and its table "qsa_prompt_attn_parity (int8
 * KV), ms per chunk and error against FP64"; "Strata PR #2146" (the same
 * kernel in one stage).
 *
 * Query i (absolute position q_pos0 + i) of query head h reads kv head
 * g = h / (Hq / Hkv) and keys j <= q_pos0 + i:
 *   s_ij = sm_scale * ks_j * sum_c q_ic kc_jc;  p = softmax_j(s) in fp32;
 *   out_ic = sum_j p_ij * vs_j * vc_jc.
 * Layouts: q_bf16 [Nq, Hq, 128] with element strides q_tok_stride (between
 *   tokens) and q_head_stride (between heads); k_cache, v_cache int8
 *   [Hkv, Nk, 128] with kv_head_stride elements between heads and 128 between
 *   tokens; k_scale_f16, v_scale_f16 fp16 [Hkv, Nk] with scale_head_stride;
 *   out_bf16 [Nq, Hq, 128] with o_tok_stride, o_head_stride.
 * Requires Hq % Hkv == 0, 1 <= Nq, q_pos0 >= 0, q_pos0 + Nq <= Nk.  Cache
 * positions q_pos0 + Nq .. Nk - 1 are visible to no query and never read, so
 * a chunk may attend within a longer, partly filled cache.
 * sm_scale <= 0 selects 1/sqrt(128).  Workspace: at least
 * int8kv_prompt_attn_workspace(Nq, Hq, Hkv, Nk) bytes.
 * ---------------------------------------------------------------------- */
size_t int8kv_prompt_attn_workspace(int Nq, int Hq, int Hkv, int Nk);
sage_status int8kv_prompt_attn(const void *q_bf16, int64_t q_tok_stride, int64_t q_head_stride,
                               const int8_t *k_cache, const void *k_scale_f16, const int8_t *v_cache,
                               const void *v_scale_f16, int64_t kv_head_stride,
                               int64_t scale_head_stride, int Nq, int q_pos0, int Nk, int Hq,
                               int Hkv, int d, float sm_scale, void *out_bf16, int64_t o_tok_stride,
                               int64_t o_head_stride, void *workspace, size_t workspace_bytes,
                               int32_t *status_dev, void *stream);

/* ------------------------------------------------------------------------
 * int8kv_prompt_attn_fault_test - exercises the failure detection of
 * int8kv_prompt_attn: the same launch, except that the kernel's load warp
 * stops early, so the other warps' bounded waits run out after
 * wait_limit_ns.
 *   mode 1: the load warp issues no copy at all;
 *   mode 2: it loads the query tile and the first two key tiles, then
 *           stops, so copies and Q.K^T MMAs are issued before the waits give
 *           up and must complete before the kernel frees its memory.
 * The kernel sets *status_dev to SAGE_ERR_TIMEOUT, lets every warp pass the
 * barriers its group shares (they cannot time out), waits for what was
 * issued, frees its tensor memory and returns; nothing faults, traps or
 * hangs and the CUDA context stays usable.  The output is not meaningful.
 * status_dev must not be NULL; wait_limit_ns > 0; mode 1 or 2, else
 * SAGE_ERR_INVALID_ARG.  Other arguments as int8kv_prompt_attn.
 * ---------------------------------------------------------------------- */
sage_status int8kv_prompt_attn_fault_test(const void *q_bf16, int64_t q_tok_stride, int64_t q_head_stride,
                                          const int8_t *k_cache, const void *k_scale_f16, const int8_t *v_cache,
                                          const void *v_scale_f16, int64_t kv_head_stride,
                                          int64_t scale_head_stride, int Nq, int q_pos0, int Nk, int Hq, int Hkv,
                                          int d, float sm_scale, void *out_bf16, int64_t o_tok_stride,
                                          int64_t o_head_stride, void *workspace, size_t workspace_bytes,
                                          int32_t *status_dev, uint64_t wait_limit_ns, int mode, void *stream);

/* ------------------------------------------------------------------------
 * int8kv_cache_write - quantizes N new K and V rows per kv head into the
 * int8 KV cache read by int8kv_prompt_attn, at cache positions
 * pos0 .. pos0+N-1.  Page: "Strata PR #2092" (an int8 K/V cache with
 * per-token fp16 scales, written upstream of the prompt attention).  Per row
 * of 128 channels of one (kv head, token):
 *   scale = fp16_rn(fl(amax / 127)),
 *   code  = clamp(rint_even(fl(x / float(scale))), -127, 127), 0 where the
 *           fp16 scale is 0.
 *
 * k_src, v_src: [N][Hkv][128] with element strides src_tok_stride,
 *   src_head_stride (channel stride 1), type src_dtype (SAGE_DTYPE_BF16 or
 *   SAGE_DTYPE_F32); bf16 rows need 8-byte alignment (strides multiples of
 *   4), fp32 rows 16-byte alignment (strides multiples of 4).
 * k_cache, v_cache: int8 [Hkv][Ncache][128], head stride cache_head_stride
 *   elements (>= Ncache*128, a multiple of 16), 16-byte aligned.
 * k_scale_f16, v_scale_f16: fp16 [Hkv][Ncache], head stride
 *   scale_head_stride (>= Ncache).
 * Requires d == 128, N >= 1, Hkv >= 1, 0 <= pos0, pos0 + N <= Ncache.  Only
 * the N new rows (codes and scales) are written.  If an fp16 scale is not
 * finite (amax/127 beyond 65504) *status_dev becomes SAGE_ERR_NONFINITE and
 * that row's codes are undefined.  Inputs must be finite.
 * ---------------------------------------------------------------------- */
sage_status int8kv_cache_write(const void *k_src, const void *v_src, int src_dtype, int64_t src_tok_stride,
                               int64_t src_head_stride, int N, int Hkv, int d, int pos0, int8_t *k_cache,
                               int8_t *v_cache, int64_t cache_head_stride, int Ncache, void *k_scale_f16,
                               void *v_scale_f16, int64_t scale_head_stride, int32_t *status_dev, void *stream);

/* ------------------------------------------------------------------------
 * sage_conversion_check - check hook: applies, on the device, the four
 * number-format conversions the kernels use to every fp32 x[i]:
 *   e4m3[i] = OCP E4M3 code, round to nearest even, saturating to +-448
 *             (cvt.rn.satfinite.e4m3x2.f32: the V codes and the FP8 P of
 *             "Sage2 SM89 Temporal Pair Experiment", section "Candidate");
 *   i8[i]   = round to nearest even integer, clamped to [-127, 127] (the
 *             Q/K codes and the int8 cache codes);
 *   bf16[i] = bf16 bits, round to nearest even (the attention outputs);
 *   f16[i]  = fp16 bits, round to nearest even (the int8 cache scales).
 * n even and >= 2; every pointer 16-byte aligned device memory of n
 * elements.  Enqueued on `stream`; for tests that sweep fp32 bit patterns.
 * ---------------------------------------------------------------------- */
sage_status sage_conversion_check(const float *x, int64_t n, uint8_t *e4m3, int8_t *i8, uint16_t *bf16,
                                  uint16_t *f16, void *stream);

/* ------------------------------------------------------------------------
 * sage_probe_rates - measurement hook for the roofline of the attention
 * kernels: runs one CTA per SM (grid = the device's SM count), each doing a
 * fixed amount of one kind of work, and writes the SM clock cycles (clock64)
 * that CTA took to cycles[cta]:
 *   kind 0: iters blocks of 128 x 128 x 128 MACs as tcgen05.mma kind::f16
 *           M128 N128 K16 (8 per block), operands in shared memory, fp32
 *           accumulators in TMEM: the Q.K^T instruction of the dense path;
 *   kind 1: the same blocks as kind::f8f6f4 E4M3 M128 N128 K32 (4 per
 *           block): the P.V instruction of the dense path;
 *   kind 2: iters x 64 x 8 ex2.approx.f32 on each of 384 threads (MUFU):
 *           the softmax's exponentials.
 * MACs (or ex2) per clock per SM = work / cycles; with the call's duration
 * (CUDA events) cycles also give the SM clock of the run.
 * cycles: device memory of at least SM-count entries; sink: one device fp32
 * (never written in practice); status_dev: device int32, SAGE_ERR_TIMEOUT if
 * the bounded wait for the MMA chain ran out.  kind in 0..2, 1 <= iters <=
 * 2^20.  Not part of the attention path; called by the benchmark.
 * ---------------------------------------------------------------------- */
sage_status sage_probe_rates(int kind, int iters, unsigned long long *cycles, float *sink, int32_t *status_dev,
                             void *stream);

/* ------------------------------------------------------------------------
 * sage_shard_range - the contiguous range [*begin, *end) of `units`
 * independent problems that rank `rank` of `world` processes: the first
 * units % world ranks take ceil(units / world) units, the others
 * floor(units / world), in rank order (so no rank holds more than
 * ceil(units / world), and a rank with nothing to do gets begin == end).
 *
 * Defines the head partition of a multi-GPU run: every (batch, head)
 * attention problem is independent, and the Ulysses layout the pages name
 * for distributed execution ("H3 Performance Roadmap", section "Phase 3:
 * NVFP4 Fused Projection Prototype", the paragraph on the direct-layout
 * target: QKV tiles land in rank-destined Ulysses buffers) puts whole heads
 * on ranks.  Units are the B*H heads of the dense path, the Hkv kv-head
 * groups of int8kv_prompt_attn, or the tokens of a sequence-sharded tensor.
 * Host only, no CUDA call.  SAGE_ERR_INVALID_ARG for units < 0, world < 1,
 * rank outside [0, world) or a NULL output pointer.
 * ---------------------------------------------------------------------- */
sage_status sage_shard_range(int64_t units, int world, int rank, int64_t *begin, int64_t *end);

/* ------------------------------------------------------------------------
 * sage_debug_bounds - the bounds record of the debug build.
 *
 * Not an operation of the method: a checking aid that stands in for a
 * memory sanitizer.  The library can be built a second time with
 * -DSAGE_DEBUG_BOUNDS (the package's build(debug_bounds=True) writes
 * libsage_gb300_debug.so beside the normal library).  In that build every
 * global load or store whose index a kernel computes is guarded: when the
 * index falls outside the tensor it belongs to (per the sizes and layouts
 * documented above), the access is skipped and the first such site is
 * recorded on the device; nothing traps.  Accesses made by the TMA engine
 * are bounds-checked by the hardware and are not instrumented.
 *
 * sage_debug_bounds synchronises the current device, stores in *site the
 * first recorded site since the previous call (0 if none; otherwise kernel
 * file id * 100000 + source line: 1 quant.cu, 2 prepare.cu, 3 kvcache.cu,
 * 4 attn_dense.cu, 5 attn_int8kv.cu, 6 check.cu) and clears the records.
 * In the normal build there are no checks and *site is always 0.
 * SAGE_ERR_INVALID_ARG for a NULL site, SAGE_ERR_CUDA if the device could
 * not be read.
 * sage_debug_bounds_enabled: 1 in the debug build, 0 otherwise (host only).
 * ---------------------------------------------------------------------- */
sage_status sage_debug_bounds(int32_t *site);
int sage_debug_bounds_enabled(void);

#ifdef __cplusplus
}
#endif
#endif /* SAGE_GB300_H */
