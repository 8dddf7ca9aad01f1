/*
 * mla_split.h -- C ABI of the GB300 (sm_103a) split-KV sparse-MLA decode library.
 *
 * Scope (every call below cites the passage that defines its operation):
 *
 *   FlashMLA PR #25 (vllm-project/FlashMLA), "Purpose" and "What changes":
 *     decode tokens with h_q = 64 heads attend over a top-k set of rows of one
 *     shared latent KV cache; the job space is (query token, KV split); each
 *     job stores an fp32 partial O normalised by its own l_i plus a log2-space
 *     LSE, and a combine kernel folds the splits, owns the attention sink and
 *     performs the final cast. Without partial buffers the kernel runs the
 *     unsplit path with a direct (fused) epilogue.
 *   "The Split-K Dispatch" (magik.net), "The Reasoning Behind the Design":
 *     the split count is a deterministic function of the batch so the scratch
 *     size and the branch are fixed per CUDA graph; the combine takes the
 *     global max of the per-split maxima and weights splits by exp2(local - global).
 *   cuDNN-frontend PR #768, SM120 FP8 commit: KV ranges cut into near-equal
 *     chunks with the remainder to the leading splits; a chunk past the end is
 *     empty and yields O = 0 / LSE = -inf; the combine owns the amax; the host
 *     requires an LSE under a split and sizes O/LSE as partial workspaces.
 *
 * Conventions for every entry point:
 *   - Every function returns an int status (MLA_OK = 0). Nothing throws.
 *     mla_status_string() maps a status to text. Argument errors are detected
 *     on the host before any launch and leave device memory untouched.
 *   - Pointers named q, kv, idx, workspace, out, lse_out, amax_out, sink are
 *     DEVICE pointers owned by the caller; the library never frees or keeps
 *     them and allocates nothing on any call below.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream). All device work is asynchronous on that stream; no call
 *     synchronises except mla_get_status().
 *   - The calls are capturable into a CUDA graph: no allocation, no host
 *     synchronisation and no data-dependent host branch (the split count comes
 *     from the plan, fixed per s_q_max).
 *   - The calling thread's current CUDA device is the device used. The first call
 *     that touches a device (any call below except the planners with num_sms > 0)
 *     sets that device up once (kernel attributes, status word); make that first
 *     call before capturing a stream into a CUDA graph.
 */
#ifndef MLA_SPLIT_H_
#define MLA_SPLIT_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MLA_API __attribute__((visibility("default")))
#else
#define MLA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define MLA_OK                0
#define MLA_ERR_INVALID_ARG   1   /* null / misaligned pointer, bad size, s_q > plan.s_q_max ... */
#define MLA_ERR_UNSUPPORTED   2   /* shape outside what the kernels implement (e.g. h_q != 64)  */
#define MLA_ERR_WORKSPACE     3   /* workspace missing or smaller than the plan requires       */
#define MLA_ERR_CUDA          4   /* a CUDA runtime/driver call failed (launch, attribute ...) */
#define MLA_ERR_NO_DEVICE     5   /* no usable sm_100-family device is current                 */

/* Bits of the device status word (see mla_get_status). */
#define MLA_STATUS_TIMEOUT    0x1u  /* a bounded wait inside a kernel ran out; that CTA aborted */
#define MLA_STATUS_BAD_SHAPE  0x2u  /* a dense job held more than 64 query rows (s_q_b * h_q/h_kv);
                                       it wrote nothing */
#define MLA_STATUS_BAD_ALIGN  0x4u  /* the dynamic shared memory base was not 1024-byte aligned;
                                       the sparse kernel wrote nothing */
#define MLA_STATUS_BAD_INDEX  0x10u /* with index checks on (mla_set_index_checks), a gathered
                                       index was outside {-1} and [0, n_kv); that row was
                                       masked, as it always is */

/* Output element types of the final cast (FlashMLA PR #25, "What changes":
 * the FP8 cast moves into the combine; the fp32 pass-through exists for parity). */
#define MLA_OUT_F32   0
#define MLA_OUT_BF16  1
#define MLA_OUT_E4M3  2   /* code = e4m3_satfinite_rn(O * out_inv_scale); one per-tensor scale */

/* Largest split count any plan may use. */
#define MLA_MAX_SPLITS 64
#define MLA_FORCE_BALANCED (-1)   /* force_splits value: the balanced schedule wherever it applies */

/* ======================================================================= *
 *  Sparse MLA decode                                                       *
 * ======================================================================= */

/* A plan: every size and offset the split and combine calls need, computed once
 * per s_q bucket on the host ("The Split-K Dispatch", "CUDA Graph Safety").
 * Workspace layout (one caller-owned device buffer, 256-byte aligned):
 *   [0, o_acc_bytes)                       fp32 (or bf16, see partial_bf16) O
 *                                          partials, split-major
 *                                          [num_splits][s_q][h_q][d_v]
 *   [lse_acc_offset, + lse_acc_bytes)      fp32 log2 LSE partials
 *                                          [num_splits][s_q][h_q]
 * where s_q is the s_q of the call (<= s_q_max). For num_splits == 1 no
 * workspace is needed (workspace_bytes == 0) and the direct path runs. */
typedef struct {
  int32_t s_q_max;      /* largest number of decode tokens per call               */
  int32_t h_q;          /* query heads; 64                                         */
  int32_t d_qk;         /* 576 = 512 latent + 64 RoPE dims                         */
  int32_t d_v;          /* 512 = the first 512 dims of each row                    */
  int32_t topk;         /* top-k entries per token (row stride of idx)             */
  int32_t block_rows;   /* 64: top-k entries per KV block, the unit of a split     */
  int32_t num_blocks;   /* ceil(topk / block_rows)                                 */
  int32_t num_splits;   /* S; may exceed num_blocks (those splits are empty)       */
  int32_t num_sms;      /* SM count the split choice was made for                  */
  int32_t balanced_ctas; /* > 0: mla_sparse_decode runs the balanced schedule with at
                            most this many CTAs (see below); 0: the (token, split) jobs */
  int32_t dim_groups;   /* CTAs per (token, split) job: 1, 2 or 4. Each computes the
                           job's scores and softmax and 512/dim_groups of its output
                           dims, so PV and the output stores of one job spread over
                           dim_groups SMs (used when s_q_max * num_splits leaves SMs idle) */
  int32_t partial_bf16; /* 0 (default): O partials in fp32; 1: in bf16 (set with
                           mla_plan_set_partials_bf16; LSE partials stay fp32)     */
  int32_t tail_ctas;    /* > 0: a call whose one-split grid would leave a last wave
                           at most half full cuts that wave's tokens into splits or dims
                           (see "Tail of the grid" below), in at most this many CTAs;
                           the workspace holds their partials                      */
  uint64_t o_acc_bytes;     /* num_splits * s_q_max * h_q * d_v * (4, or 2 with bf16
                               partials)                                           */
  uint64_t lse_acc_offset;  /* o_acc_bytes rounded up to 256                       */
  uint64_t lse_acc_bytes;   /* num_splits * s_q_max * h_q * 4                      */
  uint64_t workspace_bytes; /* what every call on this plan needs; 0 when num_splits == 1
                               and balanced_ctas == 0                              */
} mla_plan_t;

/* Tail of the grid (plan->tail_ctas > 0; automatic plans with num_splits == 1 and
 * s_q_max > num_sms). One split per token runs s_q CTAs in ceil(s_q / num_sms)
 * waves; when the last wave would hold r tokens and S_t = min(num_blocks,
 * floor(num_sms / r)) >= 3, a call cuts each of those r tokens into S_t splits
 * (near-equal block ranges, the first num_blocks mod S_t one block longer), run
 * after the whole tokens, and folds them with the combine over their rows only:
 * the last wave then walks about num_blocks / S_t blocks instead of num_blocks.
 * Measured on GB300 (152 SMs, topk 640, 10 blocks; back-to-back calls, e4m3 out):
 * s_q 153: 59.4 -> 46.1 us, 160: 59.9 -> 49.0, 176: 60.9 -> 49.8, 190: 61.1 ->
 * 53.2, 200: 61.1 -> 55.7, 320: 89.3 -> 84.1; with two splits (s_q 212, 228) no
 * gain, hence the bound S_t >= 3. Otherwise, when 2 r <= num_sms, each of the r
 * tokens runs whole on two CTAs, each with half of the output dims (the full QK
 * and softmax, half the PV, final rows; no partials, no combine), measured s_q
 * 212: 61.5 -> 58.4 us, 220: 61.7 -> 57.9, 228: 61.6 -> 59.1 (where two splits
 * gained nothing). The split form's workspace holds [S_t][r][64][512] O
 * partials (fp32, or bf16 with mla_plan_set_partials_bf16) and [S_t][r][64] LSE
 * partials at the next 256-byte boundary, S_t * r <= num_sms. The pages have no
 * counterpart (their grids are one wave); it reuses their partial / LSE protocol.
 * The no-allocation entry point never cuts a tail; setting tail_ctas to 0 in a
 * plan turns it off. */

/* Balanced schedule of the one-shot call (plan->balanced_ctas > 0). FlashMLA PR #25
 * ("Measured") shows the (token, split) grid losing at s_q >= 96, where s_q * S
 * jobs do not spread evenly over the SMs. Here the s_q * num_blocks 64-row blocks
 * of all tokens, token-major, are cut into P contiguous near-equal ranges, one per
 * CTA, with P the fewest CTAs that reach the smallest per-CTA block count on
 * num_sms SMs: per = ceil(s_q * num_blocks / num_sms), P = ceil(s_q * num_blocks / per).
 * A token inside one range is finished by that CTA (sink, cast, LSE, amax). Each
 * piece of a token cut by range boundaries is a partial with the split definition,
 * written to slot = the piece's place among its token's pieces (0 for the piece
 * that holds the token's first block) in the split layout [slot][s_q][h_q][d_v]
 * (fp32) and [slot][s_q][h_q] (fp32 LSE, at the next 256-byte boundary after the
 * O part sized for s_q_max); the combine, launched as the decode kernel's
 * programmatic dependent, folds each cut token's pieces. So the call is two
 * kernels and the workspace holds one partial slot per piece of the most cut
 * token (over every s_q <= s_q_max the schedule applies to). Nothing in it needs
 * to start at zero. */

/* Choose the split count and size the workspace ("The Split-K Dispatch",
 * "Adaptive NSPLIT"; FlashMLA PR #25, "Measured": partial bytes
 * num_splits * s_q * h_q * d_v * 4).
 *   num_sms      0 = query the current device.
 *   max_splits   0 = MLA_MAX_SPLITS; caps the automatic choice.
 *   force_splits 0 = automatic; > 0 uses exactly that many splits (<= MLA_MAX_SPLITS),
 *                even above num_blocks (the extra splits are empty).
 * Automatic rule: among split counts S with s_q_max * S <= num_sms (at least 1),
 * take the smallest S that reaches the fewest blocks per split, counting
 * max(2, ceil(num_blocks / S)): a split of two 64-row blocks costs about what a
 * split of one does, and fewer splits leave SMs to dim groups and partials to
 * the combine (measured on GB300, topk 640: s_q = 10 takes 5 splits x 2 dim
 * groups, 21.6 us, where 10 splits x 1 took 25.3 us); except that, when that S
 * is above 1, S = num_blocks (one block per split) when num_blocks is within
 * that bound and s_q_max *
 * num_blocks * 4 <= num_sms, i.e. every one-block split still gets 4 dim groups
 * (measured on GB300, topk 640: s_q = 1, 2, 3 take 9.2, 9.4, 9.8 us with 10
 * splits against 10.1, 10.2, 10.5 us with 5).
 * dim_groups is the largest of 4, 2, 1 with s_q_max * S * dim_groups <= num_sms.
 * The balanced schedule is never chosen automatically: measured on GB300 (topk
 * 640, back-to-back calls) the uniform grid beat it at every s_q from 96 to 384,
 * also where the grid leaves a wave half empty (s_q = 200: 61.8 us against 87.9
 * us), because the fp32 partials of the cut tokens, their combine and each CTA's
 * job boundaries cost more than the blocks it saves. force_splits ==
 * MLA_FORCE_BALANCED keeps the automatic S and enables the balanced schedule
 * whenever 2 <= per = ceil(s_q_max * num_blocks / num_sms); enabling it sets
 * balanced_ctas = min(num_sms, s_q_max * num_blocks) and sizes the workspace for
 * both schedules: the larger of the two partial areas. With force_splits > 0 the
 * one-shot call runs the (token, split) jobs.
 * Errors: MLA_ERR_UNSUPPORTED unless h_q == 64, d_qk == 576, d_v == 512;
 *         MLA_ERR_INVALID_ARG for s_q_max < 1, topk < 1, out == NULL, or bad split counts. */
MLA_API int mla_decode_plan(int s_q_max, int h_q, int d_qk, int d_v, int topk,
                    int num_sms, int max_splits, int force_splits, mla_plan_t* out);

/* Switches a plan's O partials to bf16 (enable = 1) or back to fp32 (enable = 0),
 * and recomputes o_acc_bytes, lse_acc_offset, lse_acc_bytes and workspace_bytes
 * for it; every later call on the plan (split pass, combine, one-shot call, also
 * the balanced schedule) stores and reads the partials in that type. The pages
 * name bf16 partials as the way to halve the partial traffic that regressed the
 * 16-token lane ("The Split-K Dispatch", "Numerical Precision Tradeoffs";
 * FlashMLA PR #25, "Measured"). fp32 stays the default because bf16 partials do
 * not keep the identical-code floor of the FP8 output: every e4m3 code stays
 * within one step of the oracle's and O within 2e-3 norm-wise per row, but with
 * non-cancelling V (mean 1.0) fewer than 99 % of the codes equal the oracle's
 * (98.8 % in the oracle's own simulation at s_q = 16, 2 splits). The LSE is
 * unchanged (fp32 partials). Errors: MLA_ERR_INVALID_ARG for plan == NULL,
 * enable not 0 or 1, or a plan not made by mla_decode_plan. This entry point has
 * no counterpart in the pages. */
MLA_API int mla_plan_set_partials_bf16(mla_plan_t* plan, int enable);

/* Zeroes all plan->workspace_bytes of `workspace` on `stream`. No schedule needs
 * its workspace to start at zero (every partial slot a call reads was written by
 * the same call); this is a convenience for callers that want a defined state.
 * Returns MLA_OK at once when the plan needs no
 * workspace; MLA_ERR_WORKSPACE for a NULL or not 256-byte aligned workspace;
 * MLA_ERR_INVALID_ARG for plan == NULL; MLA_ERR_CUDA when the clear cannot be
 * queued. */
MLA_API int mla_workspace_init(const mla_plan_t* plan, void* workspace, void* stream);

/* Split pass: one CTA per (token t, split s) job; the job walks the top-k
 * entries of its own block range (FlashMLA PR #25, "What changes"), gathers the
 * rows idx[t, r] of kv, and writes
 *     O_acc[s][t][h][:] = sum_r exp(s_r) V_r / sum_r exp(s_r)       (fp32)
 *     LSE_acc[s][t][h]  = log2 sum_r exp(s_r)                       (fp32)
 * with s_r = sm_scale * <q[t,h,:], kv[idx[t,r], :]> in natural-log units; an
 * empty split (no blocks, or no valid index) writes O = 0 and LSE = -inf
 * (cuDNN-frontend PR #768, SM120 FP8 commit). No sink is applied here.
 *   q    bf16 [s_q][h_q][576], contiguous, 16-byte aligned.
 *   kv   bf16 [n_kv][576], contiguous rows, 16-byte aligned; 1 <= n_kv < 2^31.
 *   idx  int32 [s_q][topk]; an entry outside [0, n_kv) (e.g. -1 padding) is masked.
 *   workspace >= plan->workspace_bytes, 256-byte aligned (layout in mla_plan_t).
 * Requires plan->num_splits > 1 (MLA_ERR_INVALID_ARG otherwise: use
 * mla_sparse_decode_direct) and 1 <= s_q <= plan->s_q_max. */
MLA_API int mla_sparse_decode_split(const mla_plan_t* plan, int s_q,
                            const void* q, const void* kv, int64_t n_kv,
                            const int32_t* idx, float sm_scale,
                            void* workspace, void* stream);

/* Combine: for every (t, h), with M = max_s LSE_acc[s][t][h],
 *     w_s = 2^(LSE_acc[s] - M)               (0 for an empty split)
 *     O   = sum_s w_s O_acc[s] / (sum_s w_s + 2^(sink_h * log2(e) - M))
 *     LSE = M + log2 sum_s w_s               (the sink is NOT included)
 * then casts O to out_dtype ("The Split-K Dispatch", "The LSE Combine Strategy";
 * FlashMLA PR #25, "What changes": the combine owns the sink and the cast). A
 * (t, h) whose splits are all empty gives O = 0, LSE = -inf.
 *   sink      fp32 [h_q] natural-log logits, or NULL for no sink.
 *   out       [s_q][h_q][d_v] of out_dtype (fp32 / bf16 / e4m3 bytes), 16-byte aligned.
 *   out_inv_scale  multiplies O before the e4m3 cast (ignored otherwise).
 *   lse_out   fp32 [s_q][h_q] or NULL.
 *   amax_out  fp32 scalar or NULL: overwritten with max |O| of the recombined,
 *             pre-cast O (cuDNN-frontend PR #768: the combine owns the amax). */
MLA_API int mla_split_combine(const mla_plan_t* plan, int s_q, const void* workspace,
                      const float* sink, int out_dtype, float out_inv_scale,
                      void* out, float* lse_out, float* amax_out, void* stream);

/* Unsplit path with the fused epilogue (FlashMLA PR #25, "What changes":
 * "Unsplit behaviour is unchanged"): one CTA per token over all top-k entries,
 * sink and cast applied in the epilogue; the same O / LSE / amax definitions as
 * mla_split_combine. Needs no plan and no workspace. Arguments as above;
 * topk >= 1, s_q >= 1. */
MLA_API int mla_sparse_decode_direct(int s_q, int topk, const void* q, const void* kv, int64_t n_kv,
                             const int32_t* idx, float sm_scale, const float* sink,
                             int out_dtype, float out_inv_scale,
                             void* out, float* lse_out, float* amax_out, void* stream);

/* One call for the whole decode step. With plan->balanced_ctas > 0: the balanced
 * schedule (described above mla_decode_plan) unless this call's s_q leaves fewer
 * than 2 blocks per CTA (per rule above with s_q for s_q_max). Otherwise the direct path when
 * plan->num_splits == 1, else mla_sparse_decode_split followed by
 * mla_split_combine on the same stream. Same O / LSE / amax definitions either way. */
MLA_API int mla_sparse_decode(const mla_plan_t* plan, int s_q,
                      const void* q, const void* kv, int64_t n_kv,
                      const int32_t* idx, float sm_scale, const float* sink,
                      int out_dtype, float out_inv_scale,
                      void* out, float* lse_out, float* amax_out,
                      void* workspace, void* stream);

/* The same decode step with the step's inputs and results in host memory, for a
 * caller whose queries and indices arrive from the host and whose output is read
 * there. In order on `stream`: q and idx are copied from host memory into the
 * caller's device buffers, mla_sparse_decode runs on those, and out (and lse)
 * are copied back into host memory; one cudaMemcpyAsync per buffer. With
 * page-locked host buffers every copy is asynchronous and the call returns at
 * once; with pageable ones the runtime may finish a copy before returning. The
 * host results are complete once the stream has passed the call. The KV cache,
 * sink, workspace and amax stay on the device (decode state).
 *   q_host   bf16 [s_q][h_q][576]            copied into q_dev (device, same size, 16-byte aligned)
 *   idx_host int32 [s_q][plan->topk]         copied into idx_dev (device, same size)
 *   out_dev  [s_q][h_q][512] of out_dtype    copied into out_host
 *   lse_dev, lse_host  fp32 [s_q][h_q], both NULL or both set
 * Other arguments as mla_sparse_decode. A NULL buffer (other than the lse pair,
 * sink, amax_out and workspace as mla_sparse_decode allows) or a lone lse
 * pointer gives MLA_ERR_INVALID_ARG before anything is queued; a failed copy
 * gives MLA_ERR_CUDA. This entry point has no counterpart in the pages: it is a
 * packaging of mla_sparse_decode for host-resident inputs and outputs. */
MLA_API int mla_sparse_decode_host(const mla_plan_t* plan, int s_q,
                           const void* q_host, void* q_dev, const void* kv, int64_t n_kv,
                           const int32_t* idx_host, int32_t* idx_dev, float sm_scale, const float* sink,
                           int out_dtype, float out_inv_scale,
                           void* out_dev, void* out_host, float* lse_dev, float* lse_host,
                           float* amax_out, void* workspace, void* stream);

/* ======================================================================= *
 *  Dense FP8 GQA split-KV SDPA decode (cuDNN-frontend PR #768 form)        *
 * ======================================================================= */

/* Workspace layout as for MLA with rows = total_q * h_q and d = head dim:
 *   [0, o_acc_bytes)                    fp32 [num_splits][total_q][h_q][d]
 *   [lse_acc_offset, + lse_acc_bytes)   fp32 [num_splits][total_q][h_q]          */
typedef struct {
  int32_t batch;          /* sequences                                           */
  int32_t h_q;            /* query heads (32)                                     */
  int32_t h_kv;           /* KV heads (8); h_q % h_kv == 0, group <= 16           */
  int32_t d;              /* head dim; 128                                        */
  int32_t max_q_per_seq;  /* new tokens per sequence, <= 64 / (h_q / h_kv)        */
  int32_t total_q_max;    /* bound on sum of new tokens over the batch            */
  int32_t max_kv;         /* bound on keys per sequence                           */
  int32_t key_tile;       /* 128: keys per tile, the unit of a split              */
  int32_t num_splits;     /* splits per sequence; with adaptive_splits, the most any sequence gets */
  int32_t num_sms;
  int32_t adaptive_splits; /* 1: each sequence's split count is chosen on the GPU from the KV
                              lengths (see sdpa_fp8_decode_plan); its unused slots get LSE = -inf */
  uint64_t o_acc_bytes;
  uint64_t lse_acc_offset;
  uint64_t lse_acc_bytes;
  uint64_t workspace_bytes;
} sdpa_plan_t;

/* Split counts for the dense path. force_splits > 0: every sequence is cut into
 * exactly that many near-equal runs of 128-key tiles (remainder to the leading
 * splits). Automatic (force_splits == 0): adaptive_splits = 1 and num_splits =
 * min(max_splits or 64, 16, tiles of max_kv); each call then gives sequence b
 * clamp(ceil(tiles_b / T), 1, num_splits) splits, with T the smallest tile count
 * from ceil(sum_b tiles_b * h_kv / num_sms) up for which the jobs (splits x
 * h_kv) fit num_sms CTAs, computed on the GPU from cu_seqlens_kv, so the batch's
 * work fills one wave of SMs whatever its length mix (measured, config 5 on
 * GB300: 94.7 us, against 116.5 us for 4 splits of every sequence); the same
 * near-equal rule cuts each sequence. Split slots a sequence does not use hold LSE = -inf (and O that the
 * combine never reads). Errors as for mla_decode_plan (d must be 128). */
MLA_API int sdpa_fp8_decode_plan(int batch, int h_q, int h_kv, int d, int max_q_per_seq,
                         int total_q_max, int max_kv, int num_sms, int max_splits,
                         int force_splits, sdpa_plan_t* out);

/* Split pass over jobs (sequence b, KV head g, split s). Sequence b has
 * s_q_b = cu_seqlens_q[b+1] - cu_seqlens_q[b] new tokens and kv_b keys
 * (cu_seqlens_kv); query i sits at position kv_b - s_q_b + i and sees keys
 * 0..that position (bottom-right causal); query head j reads KV head j / (h_q/h_kv).
 * The key range [0, kv_b) is cut into num_splits near-equal runs of 128-key
 * tiles, remainder to the leading splits; an empty run writes O = 0 / LSE = -inf
 * (cuDNN-frontend PR #768, SM120 FP8 commit). Values are code * descale.
 *   q  e4m3 codes [total_q][h_q][d]; k, v e4m3 codes [total_kv][h_kv][d] (16-byte aligned).
 *   total_q, total_kv  row counts of q and k/v (= cu_seqlens_q[batch], cu_seqlens_kv[batch]);
 *      the kernels never read outside them.
 *   cu_seqlens_q, cu_seqlens_kv  int32 [batch + 1] device arrays, starting at 0, with
 *      s_q_b * (h_q / h_kv) <= 64 for every sequence (a sequence beyond that is not
 *      computed and sets MLA_STATUS_BAD_SHAPE).
 *   descale_q/k/v  fp32 device scalars (NULL = 1.0).
 * Requires plan->num_splits > 1 and total_q <= plan->total_q_max. */
MLA_API int sdpa_fp8_decode_split(const sdpa_plan_t* plan, int total_q, int64_t total_kv,
                          const void* q, const void* k, const void* v,
                          const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv,
                          const float* descale_q, const float* descale_k, const float* descale_v,
                          float sm_scale, void* workspace, void* stream);

/* Combine for the dense path: the mla_split_combine fold with no sink; writes O
 * (bf16 by default), the log2 LSE and, if amax_out != NULL, max |O| of the
 * recombined O (cuDNN-frontend PR #768: the in-kernel amax stands down under a split). */
MLA_API int sdpa_split_combine(const sdpa_plan_t* plan, int total_q, const void* workspace,
                       int out_dtype, float out_inv_scale,
                       void* out, float* lse_out, float* amax_out, void* stream);

/* Unsplit dense path with the direct epilogue (bf16/fp32/e4m3 O, LSE, amax). */
MLA_API int sdpa_fp8_decode_direct(int batch, int h_q, int h_kv, int d, int total_q, int64_t total_kv,
                           const void* q, const void* k, const void* v,
                           const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv,
                           const float* descale_q, const float* descale_k, const float* descale_v,
                           float sm_scale, int out_dtype, float out_inv_scale,
                           void* out, float* lse_out, float* amax_out, void* stream);

/* One call: direct when plan->num_splits == 1, else split + combine. */
MLA_API int sdpa_fp8_decode(const sdpa_plan_t* plan, int total_q, int64_t total_kv,
                    const void* q, const void* k, const void* v,
                    const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv,
                    const float* descale_q, const float* descale_k, const float* descale_v,
                    float sm_scale, int out_dtype, float out_inv_scale,
                    void* out, float* lse_out, float* amax_out,
                    void* workspace, void* stream);

/* ======================================================================= *
 *  Status and diagnostics                                                  *
 * ======================================================================= */

/* Synchronises the current device, then reads and clears its status word
 * (MLA_STATUS_* bits set by kernels whose bounded waits ran out). *site_out,
 * if not NULL, receives the code of the first wait that ran out (0 = none). */
MLA_API int mla_get_status(uint32_t* status_out, uint32_t* site_out);

/* Launches a one-CTA kernel that waits on an mbarrier nothing ever arrives on,
 * with the given limit in nanoseconds; the wait gives up, sets
 * MLA_STATUS_TIMEOUT and the kernel returns normally. Exercises the abort path
 * of the bounded waits without hanging or faulting the GPU. */
MLA_API int mla_selftest_wait_timeout(uint64_t limit_ns, void* stream);

/* Sets the time limit of the decode kernels' pipeline waits (every mbarrier
 * wait of the sparse-MLA and the dense kernels' roles) for the calls launched
 * after it, process wide. limit_ns = 0 restores the default of 2 s; otherwise
 * 100 ns .. 10 s, else MLA_ERR_INVALID_ARG. A wait that runs out records
 * MLA_STATUS_TIMEOUT and the wait's site in the status word (mla_get_status) and
 * aborts its CTA: the other roles stop at their next wait, the CTA waits (up to
 * 2 s, whatever this limit) for its own copies and MMAs in flight, frees its
 * tensor memory and exits; the call's outputs are then undefined. For tests of
 * that abort path: a limit far below a step's latency makes real waits run out.
 * The pages have no counterpart (failure handling of this library). */
MLA_API int mla_set_wait_limit_ns(uint64_t limit_ns);

/* Index checks for the sparse-MLA calls launched after it, process wide (a debug
 * mode switched at run time; off by default). Every index is masked the same way
 * with or without it: -1 (padding) and any value outside [0, n_kv) contribute no
 * row. With enable = 1 a value outside {-1} and [0, n_kv) also sets
 * MLA_STATUS_BAD_INDEX in the status word (mla_get_status), so a caller can tell
 * padding from a corrupt index list. enable must be 0 or 1, else
 * MLA_ERR_INVALID_ARG. No counterpart in the pages (the library's own checking). */
MLA_API int mla_set_index_checks(int enable);

/* ======================================================================= *
 *  Decode without allocation                                               *
 * ======================================================================= */

/* Size of the library-owned scratch array used by mla_sparse_decode_noalloc. */
#define MLA_NOALLOC_SCRATCH_BYTES (16u << 20)

/* The whole decode step (as mla_sparse_decode) for callers that cannot call
 * cudaMalloc: for example a plugin whose host hands it only its input and output
 * buffers and owns all device memory through a fixed memory plan, or code on a
 * path where an allocation could block on device synchronisation. The fp32
 * partial workspace of the split pass is a 16 MiB array inside the library's own
 * device image (MLA_NOALLOC_SCRATCH_BYTES); every GPU that loads the library
 * holds that array until the process exits. The caller still passes q, kv, idx,
 * sink and the outputs, as for mla_sparse_decode; the plan is made internally
 * for this s_q (num_splits: 0 = the automatic choice among the split counts
 * whose workspace fits the array, so it is never refused; > 0 forces that many).
 * This entry point has no counterpart in the pages: it is a packaging of the
 * same split + combine for that kind of caller.
 *   - Nothing is allocated: no cudaMalloc, cudaFree or allocating library call.
 *   - A forced num_splits whose workspace would exceed MLA_NOALLOC_SCRATCH_BYTES
 *     (num_splits * s_q * 64 * (512 + 1) * 4 bytes, rounded up) returns
 *     MLA_ERR_WORKSPACE and launches nothing; use fewer splits, the automatic
 *     choice, or mla_sparse_decode with a caller workspace.
 *   - Every call on a device shares the one array and leaves its contents
 *     behind; the split pass overwrites every slot it needs before the combine
 *     reads it, so no clearing is needed. Calls that overlap on the GPU (on
 *     different streams, or from several threads) race on the array: order them.
 *   - The first call on a device resolves the array's device address for that
 *     device (cudaGetSymbolAddress) and keeps it for the life of the process;
 *     make that first call before capturing a stream into a CUDA graph. As with
 *     the rest of this library's per-device state (the status word, the kernel
 *     attributes), a device reset (cudaDeviceReset) is not supported: the
 *     process must not call into the library after one. */
MLA_API int mla_sparse_decode_noalloc(int s_q, int topk, const void* q, const void* kv, int64_t n_kv,
                                      const int32_t* idx, float sm_scale, const float* sink,
                                      int num_splits, int out_dtype, float out_inv_scale,
                                      void* out, float* lse_out, float* amax_out, void* stream);

/* Text for a status code. */
MLA_API const char* mla_status_string(int status);

/* ABI version of this header (bumped on any signature or layout change). */
MLA_API int mla_abi_version(void);
#define MLA_ABI_VERSION 2

#ifdef __cplusplus
}
#endif
#endif /* MLA_SPLIT_H_ */
