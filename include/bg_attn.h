/*
 * bg_attn.h -- C ABI of the GB300 (sm_103a) attention hot path of a
 * bounded-generation SLM inference engine.
 *
 * The method is described in "SLM 生成式高并发推理引擎：延迟约束下的有效吞吐优化"
 * (163.com):
 *   - abstract: Packed Prefill and a request-internal shared-prefix K/V layout
 *     are two of the custom pieces embedded in the engine;
 *   - section 1.1 (two execution forms): Prefill-Only runs one prefill; Beam
 *     Search runs one prefill plus a fixed number of decode steps at a fixed
 *     beam width, keeping candidates, cumulative scores and a parent index;
 *   - section 1.2 (input/state bounds): only valid tokens of each sequence are
 *     processed (no padding); the beams of one request share one prompt K/V
 *     and each beam keeps its own short suffix K/V; all capacity is planned
 *     and preallocated at load time.
 *
 * Conventions shared by every entry point
 *   - Tensor pointers are DEVICE pointers, owned by the caller, contiguous
 *     row-major, 16-byte aligned.  bf16 tensors are passed as void*.
 *   - The library never allocates or frees memory and never synchronises the
 *     stream: every call only enqueues work on `stream` (0 = legacy default
 *     stream) and returns.
 *   - Host-checkable faults (NULL pointers, bad sizes, unsupported shapes,
 *     misalignment, aliasing) return an error before anything is enqueued.
 *   - Device-data faults (bad cu_seqlens / cu_prompt / parent_idx contents)
 *     cannot be seen by the host without a synchronisation, so the kernels
 *     check them on the device: offending work is skipped (never executed
 *     with bad indices, never trapped) and, when `dev_status` is non-NULL,
 *     the BG_DEVSTAT_* bits below are OR-ed into that device int32.  The
 *     library never clears it; zero it before the calls you want to watch.
 *   - Every internal wait of a kernel is bounded (about one second); if a
 *     wait runs out the kernel gives up, sets BG_DEVSTAT_TIMEOUT and returns.
 *   - Launch failures return BG_ERR_CUDA.
 *   - Query head h uses kv head h / (Hq / Hkv) (contiguous groups).
 */
#ifndef BG_ATTN_H
#define BG_ATTN_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    BG_OK = 0,
    BG_ERR_INVALID_ARG = 1,   /* bad pointer, size, alignment or aliasing      */
    BG_ERR_UNSUPPORTED = 2,   /* valid but outside what the kernels implement  */
    BG_ERR_DEVICE_DATA = 3,   /* reserved: device-data faults go to dev_status */
    BG_ERR_CUDA = 4           /* a CUDA runtime call or launch failed          */
} bg_status_t;

/* Bits OR-ed into *dev_status by the kernels. */
#define BG_DEVSTAT_CU_SEQLENS   0x01  /* cu_seqlens[0]!=0, decreasing, or cu[B]!=T  */
#define BG_DEVSTAT_SEQ_TOO_LONG 0x02  /* a sequence is longer than max_seqlen       */
#define BG_DEVSTAT_PARENT       0x04  /* a parent index is outside [0, W)           */
#define BG_DEVSTAT_CU_PROMPT    0x08  /* cu_prompt invalid or prompt > max_prompt   */
#define BG_DEVSTAT_EMPTY_ROW    0x10  /* prompt length 0 with suffix_len 0          */
#define BG_DEVSTAT_PLAN         0x20  /* planned run: the workspace's work list is
                                         for another packing (nothing written)     */
#define BG_DEVSTAT_TIMEOUT      0x100 /* an internal pipeline wait ran out          */

/* Supported shapes: head_dim in {64, 128}; Hq % Hkv == 0; for decode
 * Hq/Hkv <= 128; suffix_max <= BG_MAX_SUFFIX; max_seqlen <= BG_MAX_SEQLEN. */
#define BG_MAX_SUFFIX 16
#define BG_MAX_SEQLEN 65536
/* Beam width of bg_beam_select: 1 <= W <= BG_MAX_BEAM (the page's configurations
 * keep at most 400 beams); vocabulary: W <= V <= BG_MAX_VOCAB. */
#define BG_MAX_BEAM 512
#define BG_MAX_VOCAB (1 << 22)

/* Human-readable name of a status code (static storage, never NULL). */
const char *bg_status_string(bg_status_t status);

/*
 * Diagnostic of the failure path.  Enqueues one small kernel whose only wait
 * can never complete (an mbarrier that nothing arrives on), made through the
 * same bounded-wait routine as every pipeline wait of the attention kernels.
 * The wait gives up after the library's limit (about one second); the kernel
 * then ORs BG_DEVSTAT_TIMEOUT into *dev_status, stores the nanoseconds it
 * waited (device %globaltimer) in *waited_ns and returns, leaving the stream
 * and the context usable.  Nothing faults, traps or hangs.
 *   dev_status   device int32, 4-byte aligned
 *   waited_ns    device uint64, 8-byte aligned
 * Errors: BG_ERR_INVALID_ARG for NULL or misaligned pointers.
 */
bg_status_t bg_selftest_wait_timeout(int32_t *dev_status, unsigned long long *waited_ns,
                                     cudaStream_t stream);

/*
 * Bytes of device workspace bg_packed_prefill_attn needs for these sizes (an
 * upper bound that depends only on host-known sizes).  The workspace holds
 * the per-call work list the kernels build from cu_seqlens; it may be reused
 * across calls on the same stream but not by calls that overlap in time.
 */
size_t bg_packed_prefill_workspace_size(int32_t num_seqs, int32_t total_tokens,
                                        int32_t max_seqlen, int32_t Hq, int32_t Hkv,
                                        int32_t head_dim);

/*
 * Packed variable-length causal GQA prefill attention.
 * Source: abstract (Packed Prefill) and section 1.2 (valid tokens only, no
 * padding) of the page above.  For every sequence i (packed rows
 * cu_seqlens[i] .. cu_seqlens[i+1]-1), query head h and position p:
 *     out[row p, h] = sum_{j<=p} softmax_j(scale * q[p,h] . k[j,kvh]) v[j,kvh]
 * with kvh = h / (Hq/Hkv).  The softmax runs in fp32; Q.K^T and P.V run on
 * the tensor cores with bf16 operands and fp32 accumulation.
 *
 *   q            bf16 [total_tokens, Hq,  head_dim]
 *   k, v         bf16 [total_tokens, Hkv, head_dim]
 *   cu_seqlens   int32 [num_seqs+1], device; cu[0]=0, non-decreasing,
 *                cu[num_seqs]=total_tokens; zero-length sequences allowed
 *   max_seqlen   host upper bound of every sequence length (checked on device)
 *   scale        softmax scale, finite and > 0 (1/sqrt(head_dim) for standard
 *                attention); anything else gives BG_ERR_INVALID_ARG
 *   out          bf16 [total_tokens, Hq, head_dim]; rows of every valid token
 *                are written, nothing else is touched
 *   lse          fp32 [total_tokens, Hq] natural-log sum-exp of the scaled
 *                logits of each row, or NULL
 *   workspace    device buffer of at least
 *                bg_packed_prefill_workspace_size(...) bytes, 256-B aligned
 *   dev_status   device int32 or NULL (see conventions)
 * Errors: BG_ERR_INVALID_ARG for NULL/misaligned pointers, negative sizes,
 * Hq % Hkv != 0, a too-small workspace, or out aliasing an input;
 * BG_ERR_UNSUPPORTED for head_dim not in {64,128} or max_seqlen > BG_MAX_SEQLEN.
 * total_tokens == 0 or num_seqs == 0 is a valid no-op.
 */
bg_status_t bg_packed_prefill_attn(const void *q, const void *k, const void *v,
                                   const int32_t *cu_seqlens, int32_t num_seqs,
                                   int32_t total_tokens, int32_t max_seqlen,
                                   int32_t Hq, int32_t Hkv, int32_t head_dim, float scale,
                                   void *out, float *lse,
                                   void *workspace, size_t workspace_bytes,
                                   int32_t *dev_status, cudaStream_t stream);

/*
 * The same prefill in two parts, for a batch whose layers share one packing
 * (same cu_seqlens): plan once, then run every layer.  Source: as for
 * bg_packed_prefill_attn; the work list depends on the packing alone.
 *
 * bg_packed_prefill_plan enqueues the work-list pre-pass: it checks
 * cu_seqlens on the device (errors go to dev_status as for the one-call
 * form) and writes the list into the workspace.  Arguments as for
 * bg_packed_prefill_attn; the workspace needs
 * bg_packed_prefill_workspace_size(num_seqs, total_tokens, ...) bytes (the
 * head arguments of that function do not change the size).
 *
 * bg_packed_prefill_attn_planned enqueues only the attention.  Its arguments
 * and result are those of bg_packed_prefill_attn, and it reads the list the
 * last plan left in `workspace`.  That plan must have been enqueued before it,
 * with the same cu_seqlens contents, num_seqs, total_tokens and max_seqlen.
 * No other call may use the workspace in between (a planned run only reads
 * it, so runs on the same stream may follow one plan).  A plan whose
 * cu_seqlens failed the device checks makes every planned run a no-op that
 * writes nothing, as the one-call form does.  The plan records its
 * total_tokens and num_seqs in the workspace; a planned run whose own differ
 * writes nothing and raises BG_DEVSTAT_PLAN (the device cannot tell apart two
 * packings with equal sizes: the caller keeps those matched).
 *
 * Errors: bg_packed_prefill_plan gives BG_ERR_INVALID_ARG for NULL/misaligned
 * pointers, negative sizes, a too-small workspace or a workspace overlapping
 * cu_seqlens, and BG_ERR_UNSUPPORTED for max_seqlen > BG_MAX_SEQLEN;
 * num_seqs == 0 or total_tokens == 0 is a valid no-op.  The planned run gives
 * the errors of bg_packed_prefill_attn.
 */
bg_status_t bg_packed_prefill_plan(const int32_t *cu_seqlens, int32_t num_seqs,
                                   int32_t total_tokens, int32_t max_seqlen,
                                   void *workspace, size_t workspace_bytes,
                                   int32_t *dev_status, cudaStream_t stream);
bg_status_t bg_packed_prefill_attn_planned(const void *q, const void *k, const void *v,
                                           const int32_t *cu_seqlens, int32_t num_seqs,
                                           int32_t total_tokens, int32_t max_seqlen,
                                           int32_t Hq, int32_t Hkv, int32_t head_dim,
                                           float scale, void *out, float *lse,
                                           void *workspace, size_t workspace_bytes,
                                           int32_t *dev_status, cudaStream_t stream);

/*
 * Packed variable-length causal GQA prefill attention with FP8 (E4M3) Q and K.
 * Source: the abstract of the page above counts "selective FP8" among the
 * engine's mixed-precision choices without saying which matmuls use it; the
 * reading taken here is that Q and K arrive as E4M3 codes with one scale per
 * tensor while V, the softmax weights and P.V stay bf16.  The result is the
 * attention of bg_packed_prefill_attn over the dequantised inputs:
 *     q[p,h] = q_scale * e4m3(q_codes[p,h]),  k[j,kvh] = k_scale * e4m3(k_codes[j,kvh])
 *     out[row p, h] = sum_{j<=p} softmax_j(scale * q[p,h] . k[j,kvh]) v[j,kvh]
 * Q.K^T runs on the tensor cores over the codes (kind::f8f6f4, fp32
 * accumulation) and the two scales join the softmax scale.
 *
 *   q_codes      uint8 E4M3 (OCP E4M3FN) codes [total_tokens, Hq, head_dim]
 *   q_scale      finite, > 0 (the reading and its tests use powers of two,
 *                which keep every dequantised value exact in bf16)
 *   k_codes      uint8 E4M3 codes [total_tokens, Hkv, head_dim]
 *   k_scale      finite, > 0
 *   v            bf16 [total_tokens, Hkv, head_dim]
 *   other arguments, the workspace and the outputs as in bg_packed_prefill_attn
 *   (bg_packed_prefill_workspace_size gives the workspace size).
 * NaN codes are not checked: they propagate to the rows they reach.
 * Errors: as bg_packed_prefill_attn; BG_ERR_INVALID_ARG also for a scale
 * that is not finite and > 0 or whose product with the others overflows;
 * BG_ERR_UNSUPPORTED for head_dim != 128.
 */
bg_status_t bg_packed_prefill_attn_fp8(const void *q_codes, float q_scale,
                                       const void *k_codes, float k_scale, const void *v,
                                       const int32_t *cu_seqlens, int32_t num_seqs,
                                       int32_t total_tokens, int32_t max_seqlen,
                                       int32_t Hq, int32_t Hkv, int32_t head_dim, float scale,
                                       void *out, float *lse,
                                       void *workspace, size_t workspace_bytes,
                                       int32_t *dev_status, cudaStream_t stream);

/*
 * Attention of each packed sequence's last valid token only, for the last
 * layer of a Prefill-Only request.  Source: abstract and section 1.1 of the
 * page above (the request is answered from the next-token logits at each
 * sequence's last valid position).  For sequence i of length L >= 1 and
 * query head h (kvh = h / (Hq/Hkv)):
 *     out[i, h] = sum_{j<L} softmax_j(scale * q[i, h] . k[cu[i]+j, kvh]) v[cu[i]+j, kvh]
 * i.e. row L-1 of bg_packed_prefill_attn, at O(L) instead of O(L^2) cost: it
 * reads each sequence's K and V once per kv head (bandwidth-bound).
 *
 *   q            bf16 [num_seqs, Hq, head_dim]: the last valid row of each
 *                sequence (any values for zero-length sequences)
 *   k, v         bf16 [total_tokens, Hkv, head_dim], packed by cu_seqlens
 *   cu_seqlens   int32 [num_seqs+1], device (as for bg_packed_prefill_attn;
 *                checked on device, bad sequences skipped with
 *                BG_DEVSTAT_CU_SEQLENS)
 *   out          bf16 [num_seqs, Hq, head_dim]; rows of zero-length
 *                sequences are not written
 *   lse          fp32 [num_seqs, Hq] natural-log sum-exp, or NULL
 * Errors: as bg_packed_prefill_attn (no workspace);
 * BG_ERR_UNSUPPORTED also for Hq/Hkv > 16.
 */
bg_status_t bg_packed_last_token_attn(const void *q, const void *k, const void *v,
                                      const int32_t *cu_seqlens, int32_t num_seqs,
                                      int32_t total_tokens, int32_t max_seqlen,
                                      int32_t Hq, int32_t Hkv, int32_t head_dim, float scale,
                                      void *out, float *lse,
                                      int32_t *dev_status, cudaStream_t stream);

/*
 * Beam-search decode attention over a shared prompt K/V plus each beam's own
 * suffix K/V.
 * Source: section 1.2 (the beams of a request share one prompt K/V, each
 * beam keeps a short suffix K/V) and section 1.1 (fixed beam width, fixed
 * number of decode steps) of the page above.  For request r, beam b, query
 * head h (kvh = h / (Hq/Hkv)):
 *     keys   = [prompt_k rows of r ; suffix_k[r, b, 0:suffix_len, kvh]]
 *     out[r,b,h] = sum_j softmax_j(scale * q[r,b,h] . key_j) value_j
 * The query is the newest position, so nothing is masked.  The queries of
 * all beams x group heads of a request form dense 128-row tensor-core tiles
 * against the prompt K/V; the suffix slots of runs of consecutive beams
 * follow as extra 64-key tiles in which each row keeps only its own beam's
 * columns, all in one online softmax (fp32).
 *
 *   q                     bf16 [R, W, Hq, head_dim]
 *   prompt_k, prompt_v    bf16 [total_prompt_tokens, Hkv, head_dim], request r
 *                         at rows cu_prompt[r] .. cu_prompt[r+1]-1
 *   cu_prompt             int32 [R+1], device; cu[0]=0, non-decreasing,
 *                         cu[R]=total_prompt_tokens
 *   max_prompt_len        host upper bound of every prompt length
 *   suffix_k, suffix_v    bf16 [R, W, suffix_max, Hkv, head_dim]; slots
 *                         0..suffix_len-1 of each beam are read (already in
 *                         this step's beam order, see bg_beam_suffix_reorder)
 *   suffix_len            0 .. suffix_max (0: prompt only)
 *   out                   bf16 [R, W, Hq, head_dim]
 * A request with prompt length 0 and suffix_len 0 has an empty softmax: its
 * rows are skipped and BG_DEVSTAT_EMPTY_ROW is raised.
 *   scale                 softmax scale, finite and > 0
 * Errors: BG_ERR_INVALID_ARG for NULL/misaligned pointers, bad sizes,
 * suffix_len > suffix_max, Hq % Hkv != 0, scale not finite and > 0, out
 * aliasing an input;
 * BG_ERR_UNSUPPORTED for head_dim not in {64,128}, Hq/Hkv > 128 or
 * suffix_max > BG_MAX_SUFFIX.
 */
bg_status_t bg_beam_decode_attn(const void *q, const void *prompt_k, const void *prompt_v,
                                const int32_t *cu_prompt, int32_t total_prompt_tokens,
                                int32_t max_prompt_len,
                                const void *suffix_k, const void *suffix_v,
                                int32_t suffix_len, int32_t suffix_max,
                                int32_t R, int32_t W, int32_t Hq, int32_t Hkv, int32_t head_dim,
                                float scale, void *out, int32_t *dev_status,
                                cudaStream_t stream);

/*
 * Reorder of the per-beam suffix K/V by the beam parent index, with the
 * optional append of this step's new token.
 * Source: section 1.1 (beam selection yields a parent index per surviving
 * beam) and section 1.2 (each beam keeps its own suffix K/V) of the page
 * above; the page does not spell out the mechanism, the plain reading is
 * that each surviving beam inherits its parent's suffix:
 *     dst[r, b, s] = src[r, parent_idx[r, b], s]   for s < n_tokens
 *     dst[r, b, n_tokens] = new[r, b]              if new_k/new_v non-NULL
 * for K and V.  A pure copy of bf16 bit patterns: bit-exact.
 *
 *   src_k, src_v, dst_k, dst_v   bf16 [R, W, suffix_max, Hkv, head_dim]; dst
 *                                must not overlap src (ping-pong buffers)
 *   parent_idx                   int32 [R, W], device, each in [0, W);
 *                                repeats allowed (one parent, many children)
 *   new_k, new_v                 bf16 [R, W, Hkv, head_dim] or both NULL
 *   n_tokens                     slots moved, 0 .. suffix_max (suffix_max-1
 *                                when appending)
 * Beams whose parent index is out of range are left untouched in dst and
 * raise BG_DEVSTAT_PARENT.
 * Errors: BG_ERR_INVALID_ARG for NULL/misaligned pointers, bad sizes,
 * overlapping src/dst, only one of new_k/new_v given, no room to append;
 * BG_ERR_UNSUPPORTED for head_dim not in {64,128}.
 */
bg_status_t bg_beam_suffix_reorder(const void *src_k, const void *src_v,
                                   void *dst_k, void *dst_v,
                                   const int32_t *parent_idx,
                                   const void *new_k, const void *new_v,
                                   int32_t R, int32_t W, int32_t suffix_max, int32_t n_tokens,
                                   int32_t Hkv, int32_t head_dim,
                                   int32_t *dev_status, cudaStream_t stream);

/*
 * One whole beam-search decode step in one call: the suffix reorder by the
 * parent index with the append of the step's token, then the decode
 * attention over [prompt ; the new suffix].
 * Source: sections 1.1 and 1.2 of the page above, as for
 * bg_beam_suffix_reorder and bg_beam_decode_attn.  With t = suffix_len >= 1
 * the call computes
 *     bg_beam_suffix_reorder(src, dst, parent_idx, new, n_tokens = t - 1)
 *     bg_beam_decode_attn(q, ..., suffix = dst, suffix_len = t)
 * with the arguments of both checked together before anything is enqueued:
 * two launches on `stream`, the second one started by programmatic dependent
 * launch so that its prologue overlaps the first.  dst then holds the
 * reordered suffix, the next step's src.
 *
 *   q, prompt_k, prompt_v, cu_prompt, total_prompt_tokens, max_prompt_len,
 *   R, W, Hq, Hkv, head_dim, scale, out    as in bg_beam_decode_attn
 *   src_suffix_k, src_suffix_v   bf16 [R, W, suffix_max, Hkv, head_dim], the
 *                                previous step's suffix; slots 0..t-2 read;
 *                                may be NULL when suffix_len == 1
 *   parent_idx                   int32 [R, W], device, each in [0, W)
 *   new_k, new_v                 bf16 [R, W, Hkv, head_dim], the step's token
 *   dst_suffix_k, dst_suffix_v   bf16 [R, W, suffix_max, Hkv, head_dim];
 *                                slots 0..t-1 written; must not overlap any
 *                                input, out or each other
 *   suffix_len                   t, 1 .. suffix_max
 * Beams whose parent index is out of range are left untouched in dst and
 * raise BG_DEVSTAT_PARENT (the attention output is then undefined).
 * Errors: those of the two calls it stands for, and BG_ERR_INVALID_ARG for
 * suffix_len < 1 or an overlap of dst or out with an input.
 */
bg_status_t bg_beam_decode_step(const void *q, const void *prompt_k, const void *prompt_v,
                                const int32_t *cu_prompt, int32_t total_prompt_tokens,
                                int32_t max_prompt_len,
                                const void *src_suffix_k, const void *src_suffix_v,
                                const int32_t *parent_idx,
                                const void *new_k, const void *new_v,
                                void *dst_suffix_k, void *dst_suffix_v,
                                int32_t suffix_len, int32_t suffix_max,
                                int32_t R, int32_t W, int32_t Hq, int32_t Hkv, int32_t head_dim,
                                float scale, void *out, int32_t *dev_status,
                                cudaStream_t stream);

/*
 * Beam candidate selection of one decode step.  Source: section 1.1 of the page
 * above: each step selects local candidates from every beam's token
 * distribution, merges them with the accumulated scores and keeps W candidate
 * sequences; candidates, scores and the parent index come out (the parent
 * index is what bg_beam_suffix_reorder consumes next).  For request r, beam b
 * and token v:
 *     score(b, v) = cum[r, b] + logits[r, b, v] - log sum_u exp(logits[r, b, u])
 * and the W candidates (b, v) with the highest scores are kept, best first,
 * equal scores by the smaller b * V + v (all in fp32).  The first step of a
 * search is the same call with only beam 0 alive (cum = 0, -inf, ..., -inf).
 *
 *   logits       fp32 [R, W, V] next-token logits of every beam, 16-byte aligned
 *   cum          fp32 [R, W] accumulated scores (-inf marks a dead beam)
 *   token_out    int32 [R, W]  kept candidate k of request r: its token v
 *   parent_out   int32 [R, W]  ... its parent beam b (in [0, W))
 *   score_out    fp32  [R, W]  ... its score (the new accumulated score)
 *   workspace    device scratch of at least bg_beam_select_workspace_size(R, W, V)
 *                bytes, 256-byte aligned (per-beam candidates and the merge's
 *                intermediate survivors); contents on entry do not matter
 * Outputs must not overlap the inputs or the workspace.  Two or three launches
 * on `stream` (per-beam selection, then a merge: one level when W * W <= 16384,
 * else two); the logits come from HBM
 * once (a second pass over each beam's row reads back from L2 only the 16-byte
 * groups that can hold one of its W best).  NaN logits are
 * not supported (the result is then unspecified).
 * Errors: BG_ERR_INVALID_ARG for NULL/misaligned pointers, R < 0, a too small
 * workspace or overlaps; BG_ERR_UNSUPPORTED unless 1 <= W <= BG_MAX_BEAM and
 * W <= V <= BG_MAX_VOCAB.
 */
size_t bg_beam_select_workspace_size(int32_t R, int32_t W, int32_t V);
bg_status_t bg_beam_select(const float *logits, const float *cum,
                           int32_t R, int32_t W, int32_t V,
                           int32_t *token_out, int32_t *parent_out, float *score_out,
                           void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Allocation-free variant of bg_packed_prefill_attn.  The paper has no
 * counterpart to this entry point; it exists for callers that cannot
 * allocate device memory or hold a workspace of their own -- for example a
 * node inside a runtime that owns every device buffer and passes a kernel
 * call only its inputs and outputs, or a latency-bound serving loop that
 * must not call cudaMalloc.
 *
 * Same arguments, semantics and errors as bg_packed_prefill_attn, minus the
 * workspace: the same argument checks run first.  The work list lives in a
 * fixed array of BG_NOALLOC_SCRATCH_BYTES in the library's own device
 * memory, which every GPU that loads the library keeps until the process
 * exits.  Limits and rules:
 *   - valid problems with bg_packed_prefill_workspace_size(...) larger than
 *     BG_NOALLOC_SCRATCH_BYTES (total_tokens/128 + num_seqs + 1 > 65520)
 *     return BG_ERR_UNSUPPORTED and enqueue nothing;
 *   - all calls in one CUDA context share that array: calls that can overlap
 *     on the GPU (different streams, concurrent graphs) race and must be
 *     serialised by the caller;
 *   - the first call in each CUDA context looks up the array's device
 *     address (cudaGetSymbolAddress, in the context current on the calling
 *     thread) and caches it under the context's unique ID, so a context
 *     created later (after cudaDeviceReset, or another context the caller
 *     makes current) gets its own lookup; make the first call in a context
 *     before any stream capture.
 * It never calls cudaMalloc, cudaFree or any allocating routine.
 */
#define BG_NOALLOC_SCRATCH_BYTES (1u << 20)
bg_status_t bg_packed_prefill_attn_noalloc(const void *q, const void *k, const void *v,
                                           const int32_t *cu_seqlens, int32_t num_seqs,
                                           int32_t total_tokens, int32_t max_seqlen,
                                           int32_t Hq, int32_t Hkv, int32_t head_dim, float scale,
                                           void *out, float *lse,
                                           int32_t *dev_status, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* BG_ATTN_H */
