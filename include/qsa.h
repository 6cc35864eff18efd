/*
 * qsa.h - C ABI of the GB300 QSA layer (quantized sparse attention over an int8 KV cache).
 *
 * The layer ("round 6 track b - qsa flash", delivered change; "opus_r9_qsa", what
 * changed) has 2 KV groups with 12 query heads each (query head h reads group h / 12),
 * head dim 256, int8 K/V codes with one fp16 scale per 64 elements, and softmax scale
 * 1/16.  Token t of a call sits at position pos0 + t and attends to the causal cells
 * 0 .. pos0 + t, i.e. n_kv(t) = pos0 + t + 1 cells: all of them while
 * n_kv <= identity_max (2051), otherwise the topk (2048) cells selected by qsa_select
 * ("round 6 track b", delivered change: identity ids per token while n_kv <= 2051).
 *
 * Conventions for every call:
 *  - All array pointers are DEVICE pointers owned by the caller; fp16 values are passed
 *    as IEEE binary16 bit patterns (uint16_t).  Pointers must be 16-byte aligned.
 *  - The library allocates no memory.  Its only state is a per-thread last-error string
 *    and one device status word per device (see qsa_check_device_status).
 *  - Calls are asynchronous on `stream` (a cudaStream_t passed as void*; NULL = the
 *    legacy default stream) and never synchronize, except qsa_check_device_status.
 *    Kernels are launched with programmatic stream serialization: a kernel may be
 *    scheduled while the work before it on the stream finishes, but it waits for that
 *    work to complete before it reads or writes any memory, so ordering against the
 *    caller's earlier and later work on the stream is as with ordinary launches.
 *  - Return value: QSA_OK, or a negative QSA_ERR_* code with qsa_last_error() set.
 *    Argument errors are detected on the host before anything is launched.
 *
 * Layouts (row-major):
 *   q    [T][24][256]      fp16   queries of the call's tokens
 *   kq   [n_cells][2][256] int8   K codes of cache cell c, group g (cells 0 .. n_cells-1)
 *   vq   [n_cells][2][256] int8   V codes
 *   ksc  [n_cells][2][4]   fp16   K scale of elements 64b .. 64b+63
 *   vsc  [n_cells][2][4]   fp16   V scales
 *   ids  [T][2][topk]      int32  selected cells of (token, group), ascending
 *   out  [T][24][256]      fp16   prefill output
 *   part [N][chunk_cap][24][258] fp32  decode partials: o[0..255], m at 256, l at 257
 *   xp   [N][24][256]      fp32   merged decode output
 * Cache contract: the call's own tokens are already in the cache (cells pos0 .. pos0+T-1),
 * so n_cells >= pos0 + T.
 */
#ifndef QSA_H
#define QSA_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define QSA_API __attribute__((visibility("default")))
#else
#define QSA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

#define QSA_OK 0
#define QSA_ERR_INVALID_ARG (-1) /* null / misaligned pointer, bad size, too few cells  */
#define QSA_ERR_UNSUPPORTED (-2) /* parameters outside what the kernels implement       */
#define QSA_ERR_WORKSPACE (-3)   /* workspace missing or smaller than required          */
#define QSA_ERR_CUDA (-4)        /* a CUDA runtime call or launch failed                */
#define QSA_ERR_TIMEOUT (-5)     /* a bounded device-side wait gave up (status word)    */
#define QSA_ERR_DEVICE (-6)      /* another device-side check failed (status word)      */

#define QSA_N_GROUPS 2
#define QSA_HEADS_PER_GROUP 12
#define QSA_N_HEADS 24
#define QSA_HEAD_DIM 256
#define QSA_SCALE_BLOCK 64
#define QSA_CHUNK 64          /* decode split: cells per partial                     */
#define QSA_PART_STRIDE 258   /* floats per (chunk, head) partial: o[256], m, l      */

/* Selection parameters; a NULL pointer means the defaults {2048, 2051, 0.0625}.
 * Constraints: 1 <= topk <= identity_max + 1, 1 <= identity_max, sm_scale > 0 and finite. */
typedef struct qsa_params {
  int topk;          /* cells kept per (token, group) above the identity threshold */
  int identity_max;  /* n_kv <= identity_max: every causal cell, in order          */
  float sm_scale;    /* softmax scale applied to q . k                             */
} qsa_params;

/* Message of the last failing call on this host thread ("" if none). */
QSA_API const char* qsa_last_error(void);

/*
 * qsa_prep_quantize - write fp16 K or V rows into the int8 cache format (the
 * quantisation half of the pages' fused prep kernel, "round 27 track b - qsa prep and
 * merge", correctness: qsa_prep writes kq vq ksc vsc).  The pages do not state the
 * quantiser; this library uses the symmetric absmax rule per 64-element block:
 *   a = max |x|,  scale = fp16_rn(fp32(a / 127)),
 *   code = clamp(round_half_away_from_zero(fp32(x / scale)), -127, 127),
 * with scale = +0 and all codes 0 when the scale is 0.
 *   x   [n_rows][256] fp16 (e.g. n_rows = n_cells * 2 for one cache slice)
 *   xq  [n_rows][256] int8 (written)     xsc [n_rows][4] fp16 (written)
 */
QSA_API int qsa_prep_quantize(const uint16_t* x, int64_t n_rows, int8_t* xq, uint16_t* xsc, void* stream);

/* Position-encoding parameters of qsa_prep; a NULL pointer means {10000, 256, 1e-6, {32, 48, 48}}. */
typedef struct qsa_rope {
  float base;       /* rotary base: theta_i = p * base^(-2 i / rotary_dim)                           */
  int rotary_dim;   /* rotated dims per row, a power of two in [16, 256]; dims >= rotary_dim unrotated */
  float eps;        /* RMS-norm epsilon                                                              */
  int sections[3];  /* mrope: rotation pairs taken by position components 0, 1, 2 (sum rotary_dim/2) */
} qsa_rope;

/*
 * qsa_prep - the fused prep of T new tokens at positions pos0 .. pos0+T-1 (the pages' qsa_prep,
 * "round 27 track b - qsa prep and merge": decision and rejected prep fusion name its raw rows,
 * gains, norm_rope step and mrope variants; correctness lists its outputs qcur kq vq ksc vsc).
 * The pages do not give the formulas; the library's readings:
 *   q and k rows: y = x / sqrt(mean(x^2) + eps) * gamma (per head row of 256), then the rotary
 *     embedding with halves paired: for i < rd/2 (rd = rotary_dim),
 *     (y_i, y_{i+rd/2}) -> (y_i cos th - y_{i+rd/2} sin th, y_{i+rd/2} cos th + y_i sin th),
 *     th = p * base^(-2 i / rd), p = pos0 + t, or for mrope p = pos3[t][c] with c the position
 *     component whose section holds pair i (sections[0], [1], [2] consecutive pairs);
 *   v rows are used as given.
 * Writes qcur [T][24][256] fp16; kcur [T][2][256] fp16 (the k rows before quantisation; may be
 * NULL); and cache cell pos0 + t of kq/ksc and vq/vsc ([n_cells][2][256] int8, [n_cells][2][4]
 * fp16): the qsa_prep_quantize rule applied to kcur's rows and to v_raw's rows.  Other cells are
 * not touched.
 *   q_raw [T][24][256], k_raw, v_raw [T][2][256] fp16; q_gamma, k_gamma [256] fp32;
 *   pos3 [T][3] int32 (DEVICE) or NULL for plain positions.
 */
QSA_API int qsa_prep(const uint16_t* q_raw, const uint16_t* k_raw, const uint16_t* v_raw, const float* q_gamma,
                     const float* k_gamma, const int32_t* pos3, const qsa_rope* rope, int T, int pos0, int n_cells,
                     uint16_t* qcur, uint16_t* kcur, int8_t* kq, uint16_t* ksc, int8_t* vq, uint16_t* vsc,
                     void* stream);

/*
 * Bytes of device workspace qsa_select needs for a call with T tokens at pos0 over a
 * cache of n_cells cells (0 when no token of the call is above the identity threshold, and
 * for caches beyond 65,536 visible cells, whose selection needs no workspace: see qsa_select).
 */
QSA_API size_t qsa_select_workspace_bytes(int T, int pos0, int n_cells, const qsa_params* params);

/*
 * qsa_select - top-k cell selection (the pages' qsa_score + qsa_topk, "round 27 track b",
 * decision; budget boundary 2051/2052 in "round 6 track b", experiment contract).
 * For every token with n_kv(t) > identity_max and each group g:
 *   score(c) = sum over the group's 12 heads h of sm_scale * q[t,h,:] . k^[c,g,:],
 *   k^ = kq * ksc (per 64-element block), over causal cells c < n_kv(t);
 * ids[t][g][0..topk) = the topk cells of largest score, equal scores going to the lower
 * cell index, written in ascending cell order.  The ranking is exact: candidates near the
 * cut are re-scored in exact integer arithmetic, so ids are bit-identical to a ranking by
 * the mathematically exact score.  Rows of tokens at or under the threshold are not
 * written.  Calls whose largest n_kv (pos0 + T) exceeds 65,536 cells are selected by the
 * cluster kernel of qsa_decode_layer (one 16-CTA cluster per (token, group), ids only, the same
 * exact ranking), up to that call's limit of 131,072 cells; they need no workspace and take at
 * most 65535 tokens.  ws should hold qsa_select_workspace_bytes(T, pos0, n_cells, params) bytes;
 * a smaller workspace, down to qsa_select_workspace_bytes(1, pos0 + T - 1, n_cells, params), is
 * taken by selecting the tokens in consecutive chunks, the largest that fit (the same ids, the
 * selection kernels once per chunk), so the memory a caller sets aside need not grow with T.  It
 * is clobbered.  A device-side capacity overflow sets the status word (QSA_ERR_DEVICE).
 */
QSA_API int qsa_select(const uint16_t* q, const int8_t* kq, const uint16_t* ksc, int n_cells, int T, int pos0,
               int32_t* ids, void* ws, size_t ws_bytes, const qsa_params* params, void* stream);

/*
 * Bytes of device workspace qsa_flash_prefill needs for a call with T tokens at pos0: the
 * fp16 dequantised K and V rows of cells 0 .. pos0+T-1, written once per call and read by
 * every tile of the call, 2 * (pos0 + T) * 2 * 256 * 2 bytes.
 */
QSA_API size_t qsa_flash_prefill_workspace_bytes(int T, int pos0, int n_cells, const qsa_params* params);

/*
 * qsa_flash_prefill - prompt attention of T new tokens (the pages' qsa_flash, "opus_r9_qsa",
 * what changed; "round 14 track b: qsa metadata hoist", decision):
 *   out[t,h,:] = sum_{c in set(t,g)} softmax_c(sm_scale * q[t,h,:] . k^[c,g,:]) * v^[c,g,:]
 * with set(t,g) = all causal cells when n_kv(t) <= identity_max (ids rows not read), else
 * ids[t][g][0..topk).  ids may be NULL when every token of the call is at or under the
 * threshold.  ws must hold qsa_flash_prefill_workspace_bytes(...) bytes and is clobbered.
 * k^ = fp16(kq * ksc) and v^ = fp16(vq * vsc) (one rounding), fp16 operands, fp32
 * accumulation and softmax, P rounded to fp16, fp16 out.  Ids outside [0, n_kv(t)) are
 * skipped and flagged in the status word.
 */
QSA_API int qsa_flash_prefill(const uint16_t* q, const int8_t* kq, const int8_t* vq, const uint16_t* ksc,
                              const uint16_t* vsc, int n_cells, int T, int pos0, const int32_t* ids, uint16_t* out,
                              void* ws, size_t ws_bytes, const qsa_params* params, void* stream);

/*
 * qsa_flash_prefill_gated - qsa_flash_prefill with an output gate: every output element is
 * multiplied by the logistic function of the gate input before its fp16 rounding,
 *   out[t,h,d] = fp16( attention[t,h,d] * 1 / (1 + exp(-gate[t,h,d])) ).
 * The pages' evaluator feeds the layer a gate input ("round 6 track b - qsa flash", experiment
 * contract) without stating its formula; this elementwise sigmoid gate is the library's reading.
 *   gate [T][24][256] fp16 (DEVICE, 16-byte aligned); NULL gives qsa_flash_prefill.
 */
QSA_API int qsa_flash_prefill_gated(const uint16_t* q, const int8_t* kq, const int8_t* vq, const uint16_t* ksc,
                                    const uint16_t* vsc, int n_cells, int T, int pos0, const int32_t* ids,
                                    const uint16_t* gate, uint16_t* out, void* ws, size_t ws_bytes,
                                    const qsa_params* params, void* stream);

/*
 * qsa_decode_partial - split-KV partial attention for N decode tokens at positions
 * pos0 .. pos0+N-1 (the pages' qsa_attn / qsa_attn2, "round 27 track b", decision and
 * correctness).  Token t's cell set (identity or ids, ascending) is cut into consecutive
 * chunks of 64; for chunk k and head h:
 *   m = max s,  l = sum exp(s - m),  o = sum exp(s - m) * v^   (natural exp, unnormalised)
 * written to part[t][k][h][0..255], part[...][256] = m, part[...][257] = l (fp32, head
 * stride 258, chunk stride 24*258).  n_chunks[t] receives the chunk count; chunk_cap (the
 * part buffer's second dimension) must be >= ceil(max(identity_max, topk) / 64).
 */
QSA_API int qsa_decode_partial(const uint16_t* q, const int8_t* kq, const int8_t* vq, const uint16_t* ksc,
                       const uint16_t* vsc, int n_cells, int N, int pos0, const int32_t* ids, float* part,
                       int32_t* n_chunks, int chunk_cap, const qsa_params* params, void* stream);

/*
 * qsa_merge - log-sum-exp merge of decode partials (the pages' qsa_merge / qsa_merge2,
 * "round 27 track b", decision: float2 (m,l) loads; correctness: the merge formula):
 *   M = max_k m_k,  L = sum_k l_k exp(m_k - M),  xp = sum_k exp(m_k - M) o_k / L
 * over k < n_chunks[t] (1 <= n_chunks[t] <= chunk_cap; other values are flagged in the
 * status word and produce NaN rows).  chunk_cap <= 1024.  The sums are fp32 reductions in
 * a tree order (not a serial chain over ascending k), so the last bits may differ from a
 * serial sum; results are within the library's float tolerance of the exact merge.
 */
QSA_API int qsa_merge(const float* part, const int32_t* n_chunks, int N, int chunk_cap, float* xp, void* stream);

/*
 * qsa_merge_gated - qsa_merge with the output gate of qsa_flash_prefill_gated applied to the
 * merged output: xp[t,h,d] *= 1 / (1 + exp(-gate[t,h,d])).  gate [N][24][256] fp16 (DEVICE,
 * 16-byte aligned); NULL gives qsa_merge.
 */
QSA_API int qsa_merge_gated(const float* part, const int32_t* n_chunks, int N, int chunk_cap, const uint16_t* gate,
                            float* xp, void* stream);

/*
 * qsa_decode_layer - one whole decode step of the layer in a single launch: the selection of
 * qsa_select, the split attention of qsa_decode_partial and the merge of qsa_merge ("round 27
 * track b - qsa prep and merge", decision: the production decode chain qsa_score, qsa_topk,
 * qsa_attn2, qsa_merge2; "round 6 track b - qsa flash", experiment contract: the 2051/2052
 * budget boundary).  For decode token t (position pos0 + t, n_kv = pos0 + t + 1) and head h:
 *   xp[t,h,:] = sum_{c in set(t,g)} softmax_c(sm_scale * q[t,h,:] . k^[c,g,:]) * v^[c,g,:]
 * with set(t,g) the identity range or the exact top-k of qsa_select, k^ = kq * ksc and
 * v^ = fp16(vq * vsc).  fp32 output; the split into partials is internal (the cluster of CTAs
 * that takes a (token, group) splits its cells, and the merge runs inside the launch), so the
 * result equals the merge of the 64-cell partials up to fp32 rounding.
 *   xp  [N][24][256] fp32 (written)
 *   ids [N][2][topk] int32, or NULL: the selected ids of tokens above the threshold, ascending,
 *       exactly as qsa_select writes them (rows of identity tokens are not written)
 *   gate [N][24][256] fp16, or NULL: the output gate of qsa_flash_prefill_gated, applied to xp
 * Needs no workspace and allocates nothing.  n_kv of every token must not exceed 131072 cells
 * (65536 on a GPU that cannot co-schedule clusters of 16 CTAs; QSA_ERR_UNSUPPORTED otherwise).
 * A (token, group) whose cells hold more than 4096 exactly tied candidates within one of its
 * 16 slices (massive exact ties, only possible above 65536 cells) is flagged in the status
 * word (QSA_ERR_DEVICE) instead of ranked.
 */
QSA_API int qsa_decode_layer(const uint16_t* q, const int8_t* kq, const int8_t* vq, const uint16_t* ksc,
                             const uint16_t* vsc, int n_cells, int N, int pos0, int32_t* ids, const uint16_t* gate,
                             float* xp, const qsa_params* params, void* stream);

/*
 * qsa_decode_layer_batched - qsa_decode_layer for many sequences in one launch (continuous
 * batching: every sequence brings its own tokens and its own cache).  The caches live in one
 * pool of n_pool cells with the layouts above (kq [n_pool][2][256] ...); sequence s owns the
 * pool cells seqs[s][0] .. seqs[s][0] + seqs[s][1] - 1 and its tokens are the consecutive rows
 * seqs[s][3] .. seqs[s+1][3] - 1 of q / xp / ids (the last sequence runs to n_tok), at
 * positions seqs[s][2] + 0, 1, ... within the sequence (ids are cell indices within the
 * sequence).  Every sequence obeys the cache contract: pos0 + its token count <= its cell count.
 *   seqs  DEVICE array [n_seq][4] int32 {first pool cell, n_cells, pos0, first token row},
 *         first token rows increasing from 0; 16-byte aligned
 *   max_n_kv  an upper bound on every token's n_kv (the largest pos0 + token count), at most
 *         131072; it picks the cluster shape
 *   gate  [n_tok][24][256] fp16 output gate, or NULL (as in qsa_decode_layer)
 * A sequence whose entry breaks these rules is skipped (its rows are not written) and flagged
 * in the status word (QSA_ERR_DEVICE); so is a token above max_n_kv's cluster capacity.
 */
QSA_API int qsa_decode_layer_batched(const uint16_t* q, const int8_t* kq, const int8_t* vq, const uint16_t* ksc,
                                     const uint16_t* vsc, int64_t n_pool, const int32_t* seqs, int n_seq, int n_tok,
                                     int max_n_kv, int32_t* ids, const uint16_t* gate, float* xp,
                                     const qsa_params* params, void* stream);

/*
 * Bytes of device workspace qsa_flash_prefill_batched needs: a work list of the identity
 * tokens' tiles (16 bytes per 64 tokens and per sequence, plus 16) rounded up to 256 bytes,
 * then the fp16 dequantised K and V rows of every sequence's identity cells, a fixed
 * R = round_up(min(identity_max, max_n_kv), 128) rows per sequence:
 * 2 * n_seq * R * 2 * 256 * 2 bytes.  0 for invalid arguments.
 */
QSA_API size_t qsa_flash_prefill_batched_workspace_bytes(int n_seq, int n_tok, int max_n_kv,
                                                         const qsa_params* params);

/*
 * qsa_flash_prefill_batched - qsa_flash_prefill_gated for many sequences in one call
 * (continuous batching of prompts: every sequence brings its own new tokens and its own cache),
 * with the selection of qsa_select done inside the call.  Same pool and seqs table as
 * qsa_decode_layer_batched: sequence s owns pool cells seqs[s][0] .. seqs[s][0] + seqs[s][1] - 1,
 * its tokens are rows seqs[s][3] .. seqs[s+1][3] - 1 of q / out / ids (the last runs to n_tok) at
 * positions seqs[s][2] + 0, 1, ..., and its new tokens' K/V are already in its cells.  Token t of
 * sequence s attends to the sequence's cells 0 .. n_kv(t) - 1 (n_kv = pos0 + t + 1), all of them
 * when n_kv <= identity_max ("round 6 track b - qsa flash", delivered change: identity ids under
 * the budget), else the exact top-k of the select score (as qsa_select ranks it):
 *   out[t,h,:] = fp16( sum_{c in set(t,g)} softmax_c(sm_scale * q[t,h,:] . k^[c,g,:]) * v^[c,g,:]
 *                      * (gate ? 1 / (1 + exp(-gate[t,h,:])) : 1) )
 * The pages run one window per call ("round 27 track b - qsa prep and merge", correctness); this
 * batched form is the library's.
 *   seqs  DEVICE [n_seq][4] int32 {first pool cell, n_cells, pos0, first token row}, first token
 *         rows non-decreasing from 0; 16-byte aligned
 *   max_n_kv  an upper bound on every token's n_kv (every sequence's pos0 + token count): at most
 *         131072, and at most qsa_decode_layer's limit when it exceeds identity_max
 *   ids   [n_tok][2][topk] int32, or NULL: the selected ids of tokens above the threshold,
 *         ascending (rows of identity tokens are not written)
 *   gate  [n_tok][24][256] fp16, or NULL
 *   out   [n_tok][24][256] fp16 (written)
 *   ws    qsa_flash_prefill_batched_workspace_bytes(n_seq, n_tok, max_n_kv, params) bytes, 16-byte
 *         aligned, clobbered
 * Identity tokens run on the tensor cores over per-sequence fp16 mirrors (one work list of
 * 64-token tiles, heaviest first); selected tokens take the single-launch decode layer's cluster
 * kernel, whose cost grows with the token count: a sequence with many selected tokens is served
 * better by qsa_select + qsa_flash_prefill.  A sequence whose entry breaks the cache contract or
 * exceeds max_n_kv is skipped (its rows are not written) and flagged in the status word
 * (QSA_ERR_DEVICE).  n_tok and n_seq at most 65535.
 */
QSA_API int qsa_flash_prefill_batched(const uint16_t* q, const int8_t* kq, const int8_t* vq, const uint16_t* ksc,
                                      const uint16_t* vsc, int64_t n_pool, const int32_t* seqs, int n_seq, int n_tok,
                                      int max_n_kv, int32_t* ids, const uint16_t* gate, uint16_t* out, void* ws,
                                      size_t ws_bytes, const qsa_params* params, void* stream);

/*
 * qsa_select_noalloc - qsa_select without a caller workspace.  The paper has no
 * counterpart: this entry point exists for callers that cannot allocate device memory
 * when they call the layer, for example a runtime whose device memory is all reserved up
 * front by its own pool, or a plugin interface that hands the kernel only its input and
 * output buffers.  It computes exactly what qsa_select computes, using a scratch array of
 * 24 MiB that the library keeps in device memory on every GPU that loads it, for as long as
 * the process lives.
 *  - Calls whose qsa_select_workspace_bytes exceeds 24 MiB (roughly more than 16 selected
 *    tokens, or more than 16384 cells) are rejected with QSA_ERR_UNSUPPORTED before any
 *    launch; use qsa_select with a workspace for those.
 *  - It allocates nothing: no cudaMalloc, no cudaFree, no allocating library call.
 *  - The first call on a device looks up the scratch array's device address (once per
 *    device, with that device current); make that first call before any stream capture.
 *  - Every call on a device shares the one scratch array and overwrites it.  Calls that
 *    overlap on the GPU (different streams, or different host threads without ordering)
 *    race on it and give wrong ids; order them on one stream or synchronize between them.
 */
QSA_API int qsa_select_noalloc(const uint16_t* q, const int8_t* kq, const uint16_t* ksc, int n_cells, int T,
                               int pos0, int32_t* ids, const qsa_params* params, void* stream);

/*
 * qsa_debug_wait_probe - a test hook for the failure path of the bounded device waits; the
 * pages have no counterpart.  Launches one CTA whose bounded mbarrier wait (the wait every
 * pipeline of this library uses) is given budget_ns (1 us .. 2 s) on a barrier that nothing
 * arrives on, so the wait gives up and sets the device status word: the next
 * qsa_check_device_status returns QSA_ERR_TIMEOUT and clears it.  Nothing is left in flight,
 * and the context stays usable.
 */
QSA_API int qsa_debug_wait_probe(uint64_t budget_ns, void* stream);

/*
 * qsa_check_device_status - synchronize `stream`, read and clear this device's status
 * word.  Returns QSA_OK, QSA_ERR_TIMEOUT (a bounded wait inside a kernel gave up) or
 * QSA_ERR_DEVICE (an id out of range, a capacity overflow, a bad chunk count).
 */
QSA_API int qsa_check_device_status(void* stream);

#ifdef __cplusplus
}
#endif
#endif /* QSA_H */
