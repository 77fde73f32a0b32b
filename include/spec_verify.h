/*
 * spec_verify.h — C ABI of libspecverify: the verify-and-accept step of
 * speculative decoding on one NVIDIA GB300 (sm_103a).
 *
 * After the target model's single forward pass over the gamma+1 verify
 * positions of a sequence (prefix + draft tokens d_1..d_gamma), row j of the
 * target logits is its next-token distribution after prefix + d_1..d_j
 * ("第 8 章 投机解码：一次前向，验证好几个字", section 为什么一次前向能验证多个 token).
 * This library turns those logits (and, when sampling, the drafter's logits)
 * into the tokens the round emits.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Every tensor argument is a DEVICE pointer owned by the caller, row-major
 *   and contiguous.  Logit tensors must be 16-byte aligned and V must be a
 *   multiple of 8 (rows are moved as 16-byte vectors by bulk copies).
 * - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *   All work is enqueued on it; calls return before the GPU finishes.
 * - The library allocates nothing per call.  Scratch state lives in a
 *   caller-owned device workspace of spec_verify_workspace_bytes() bytes,
 *   256-byte aligned, ZEROED ONCE before its first use (cudaMemset or
 *   spec_verify_workspace_init).  A workspace serves one call at a time; calls
 *   on different workspaces are independent.
 * - Host-side argument checks run before anything is enqueued and return a
 *   negative code.  Errors found on the device (a wait that ran out, a draft
 *   token outside [0, V)) are recorded in the workspace and reported by
 *   spec_verify_status().  No C++ exception crosses this boundary.
 * - Temperatures: T <= 0 (or NaN) marks a greedy sequence.  Logits must be
 *   finite or -inf; NaN/+inf logits give unspecified tokens.
 * - out_tokens [B, gamma+1] int32: for sequence b the first n+1 entries are
 *   the emitted tokens (n accepted drafts, then the replacement / resampled /
 *   bonus token); the remaining entries are -1.  out_num_accepted [B] = n.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { SPEC_F32 = 0, SPEC_BF16 = 1 } spec_dtype;

enum {
  SPEC_OK = 0,
  SPEC_ERR_INVALID_ARG = -1,  /* null pointer, B < 1, gamma outside 1..31, V bad */
  SPEC_ERR_UNSUPPORTED = -2,  /* dtype / shape not supported by this build      */
  SPEC_ERR_ALIGNMENT = -3,    /* a logit pointer is not 16-byte aligned         */
  SPEC_ERR_WORKSPACE = -4,    /* workspace null, misaligned or too small        */
  SPEC_ERR_CUDA = -5,         /* a CUDA runtime call or kernel launch failed    */
  SPEC_ERR_TIMEOUT = -6,      /* device side: a bounded wait ran out            */
  SPEC_ERR_DEVICE_INPUT = -7, /* device side: a draft token outside [0, V)      */
  SPEC_ERR_STATE = -8,        /* host round driver: inconsistent bookkeeping   */
  SPEC_ERR_DEVICE_BOUNDS = -9 /* device side, bounds-checked build only: an
                                 index outside its extent (access skipped)    */
};

#define SPEC_MAX_GAMMA 31
#define SPEC_MAX_VOCAB (1 << 26)

/*
 * Bytes of workspace needed for batches up to B sequences, draft length up to
 * gamma and vocabulary up to V.  H = 0 sizes it for the logit entry points;
 * H > 0 (the lm_head hidden size) for spec_verify_lmhead_sample, and that
 * workspace serves the logit entry points too.  The lm_head size includes the
 * stored fp32 target logits of rows j < gamma, B*gamma*V*4 bytes (268 MB at
 * B=64, gamma=4, V=262144).  Writes *bytes; returns SPEC_OK,
 * SPEC_ERR_INVALID_ARG, or SPEC_ERR_UNSUPPORTED for lm_head shapes beyond
 * its limits (see spec_verify_lmhead_sample).
 */
int spec_verify_workspace_bytes(int B, int gamma, int V, int H, size_t *bytes);

/* Zero a workspace on `stream` (equivalent to cudaMemsetAsync(ws, 0, bytes)). */
int spec_verify_workspace_init(void *workspace, size_t workspace_bytes, void *stream);

/*
 * Greedy verification ("Accelerating Gemma 4: faster inference with
 * multi-token prediction drafters", §3.2 验证与接受机制; "自投机解码：层跳过与拒绝采样
 * 实现大模型推理加速", §3.1 贪心解码).
 *
 *   target_logits [B, gamma+1, V] (dtype dt)   row j scores position j
 *   draft_tokens  [B, gamma] int32              d_{j+1} is checked against row j
 *
 * Draft d_{j+1} is accepted iff it equals the argmax of the raw logits of row
 * j (lowest index on ties).  At the first mismatch n the target's argmax of
 * row n replaces the draft and the rest is discarded; when all gamma drafts
 * match, the argmax of row gamma is emitted as the bonus token ("第 8 章 …",
 * section 多出来的那一个 token 从哪来).  The draft logits are never read.
 */
int spec_verify_greedy(const void *target_logits, spec_dtype dt,
                       const int32_t *draft_tokens, int B, int gamma, int V,
                       int32_t *out_tokens, int32_t *out_num_accepted,
                       void *workspace, size_t workspace_bytes, void *stream);

/*
 * Greedy verification of several draft candidates per sequence ("Accelerating
 * Gemma 4: faster inference with multi-token prediction drafters", §6 进阶优化
 * 与扩展思路, item 2 多候选草稿): the target verifies n candidate drafts in one
 * pass and the candidate with the longest accepted prefix is kept.
 *
 *   target_logits [B, n_cand, gamma+1, V] (dtype dt)  rows of candidate c of
 *                                                     sequence b: its path's
 *                                                     verify positions
 *   draft_tokens  [B, n_cand, gamma] int32
 *   out_tokens [B, gamma+1], out_num_accepted [B]     as spec_verify_greedy,
 *                                                     for the kept candidate
 *   out_choice    optional [B] int32 (NULL to skip)   the kept candidate's index
 *
 * Each candidate is verified as in spec_verify_greedy; the kept one has the
 * most accepted drafts, the lowest candidate index on ties.  The workspace
 * must come from spec_verify_workspace_bytes(B * n_cand, gamma, V, 0);
 * B * n_cand must not exceed 65535.
 */
int spec_verify_greedy_multi(const void *target_logits, spec_dtype dt,
                             const int32_t *draft_tokens, int B, int n_cand, int gamma,
                             int V, int32_t *out_tokens, int32_t *out_num_accepted,
                             int32_t *out_choice, void *workspace, size_t workspace_bytes,
                             void *stream);

/*
 * Rejection-sampling verification ("Gemma 4 Multi-Token Prediction (MTP)
 * 深度解析", §2.2 推测解码的数学保证; "第 8 章 …", section 为什么输出不会变;
 * "自投机解码 …", §3.2 采样解码 and §3.3 随机数与 batch 内对齐).
 *
 *   target_logits [B, gamma+1, V], draft_logits [B, gamma, V] (both dtype dt)
 *   draft_tokens  [B, gamma] int32
 *   temperature   [B] float32; T_b <= 0 makes sequence b greedy (as above)
 *   u_accept      [B, gamma] float32 in [0, 1): one uniform per draft position
 *   u_resample    [B] float32 in [0, 1): one uniform per sequence
 *   out_debug     optional [B, gamma+1, 4] float32 (NULL to skip): for j < gamma
 *                 {p_j(d_{j+1}), q_j(d_{j+1}), L_p[j], L_q[j]}, for j = gamma
 *                 {0, 0, L_p[gamma], 0}; L = ln sum exp(l/T).  NaN for greedy.
 *
 * With p_j = softmax(l_p[j]/T_b) and q_j = softmax(l_q[j]/T_b), draft d_{j+1}
 * is accepted iff u_accept[b,j] < p_j(d)/q_j(d) (probability min(1, p/q)).
 * The first rejection n stops the walk; position n is drawn from
 * max(0, p_n - q_n)/Z by inverse CDF: the smallest token k with
 * sum_{x<=k} w(x) > u_resample[b]*Z.  If every draft passes, the bonus token
 * is drawn from p_gamma the same way.
 */
int spec_verify_sample(const void *target_logits, const void *draft_logits,
                       spec_dtype dt, const int32_t *draft_tokens,
                       const float *temperature, const float *u_accept,
                       const float *u_resample, int B, int gamma, int V,
                       int32_t *out_tokens, int32_t *out_num_accepted,
                       float *out_debug, void *workspace,
                       size_t workspace_bytes, void *stream);

/*
 * Rejection-sampling verification with top-k / top-p truncation applied
 * identically to the target and the draft distributions ("Gemma 4
 * Multi-Token Prediction (MTP) 深度解析" §5.1 samples with top_k=64,
 * top_p=0.95 next to the drafter; "第 8 章 …", 为什么输出不会变: whatever
 * transforms the target distribution must transform the draft the same way).
 *
 * Per row, at the sequence's temperature T:
 *   K  = tokens with fewer than top_k strictly larger logits (ties at the
 *        top_k-th value stay in);
 *   K' = tokens of K whose strictly more likely tokens hold less than top_p of
 *        softmax(l/T) over K (tie groups stay together);
 *   p' = softmax(l/T) over K', 0 elsewhere; q' likewise.
 * Then the rule of spec_verify_sample with p', q': accept iff
 * u_accept < p'(d)/q'(d) (q'(d) = 0: accepted); draw position n from
 * max(0, p'_n - q'_n) or the bonus from p'_gamma by inverse CDF in ascending
 * vocabulary order.  out_debug's normalisers are those of the truncated rows.
 *
 * Same arguments as spec_verify_sample plus 1 <= top_k <= 1024 and
 * 0 < top_p <= 1 (else SPEC_ERR_INVALID_ARG).  A row whose K holds more than
 * 2048 entries (massive ties) makes spec_verify_status return
 * SPEC_ERR_UNSUPPORTED.  The workspace comes from
 * spec_verify_topkp_workspace_bytes.
 */
int spec_verify_topkp_workspace_bytes(int B, int gamma, int V, size_t *bytes);

int spec_verify_sample_topkp(const void *target_logits, const void *draft_logits,
                             spec_dtype dt, const int32_t *draft_tokens,
                             const float *temperature, const float *u_accept,
                             const float *u_resample, int B, int gamma, int V,
                             int top_k, float top_p, int32_t *out_tokens,
                             int32_t *out_num_accepted, float *out_debug,
                             void *workspace, size_t workspace_bytes, void *stream);

/*
 * Centroid-masked sparse draft head ("Gemma 4 Multi-Token Prediction (MTP)
 * 深度解析" §3.4 Centroids Masking; "Gemma 4 - Drafter 解析", 高效 Embedder).
 * The token embeddings are stored cluster by cluster: cluster c owns the
 * ordered rows cluster_off[c] .. cluster_off[c+1]-1 of W_ord, and ordered row
 * i is token ord2tok[i].  For each of the R hidden rows h (the drafter's
 * hidden state at one draft position):
 *   z[c]  = h . centroids[c]                 (fp32 sums of bf16 products)
 *   S     = the top_k clusters by z, the lowest cluster index first among
 *           equal scores;
 *   out   = (token, h . W_ord[i]) for every ordered row i of the clusters in
 *           S, ascending token id; out_count[r] candidates.
 * Tokens outside S get no logit: the draft distribution is the softmax over
 * the candidates (spec_verify_sample_sparse consumes exactly this layout).
 *
 * Layouts (device, row-major): hidden [R, H], centroids [n_clusters, H],
 * W_ord [V, H] bf16, 16-byte aligned, 256 <= H <= 2048, H % 256 == 0;
 * cluster_off int32 [n_clusters+1] (non-decreasing, 0 .. V); ord2tok int32
 * [V] (a permutation of 0..V-1); out_tok int32 and out_logit f32
 * [R, max_cand]; out_count int32 [R].  1 <= n_clusters <= 8192,
 * 1 <= top_k <= min(n_clusters, 256), 1 <= max_cand <= 8192.  A row whose
 * clusters hold more than max_cand tokens keeps the first max_cand (in
 * cluster-score order) and makes spec_verify_status return
 * SPEC_ERR_UNSUPPORTED.  The workspace (spec_centroid_head_workspace_bytes,
 * zeroed once by spec_verify_workspace_init) holds the scores (up to 8
 * partial sums per score while R x n_clusters is small: the score GEMM's K
 * parts), the selection and the status word.  Asynchronous; host checks return negative codes.
 */
int spec_centroid_head_workspace_bytes(int R, int n_clusters, int top_k, size_t *bytes);

int spec_centroid_head(const void *hidden, const void *centroids, const void *W_ord,
                       const int32_t *cluster_off, const int32_t *ord2tok, int R, int H, int V,
                       int n_clusters, int top_k, int max_cand, int32_t *out_tok,
                       float *out_logit, int32_t *out_count, void *workspace,
                       size_t workspace_bytes, void *stream);

/*
 * Rejection-sampling verification against sparse draft rows.  Draft row j of
 * sequence b (row b*gamma + j of the candidate arrays) is cand_count[row]
 * candidates: tokens cand_tok[row*cand_stride + i] in ascending order, with
 * logits cand_logit[row*cand_stride + i] (the layout spec_centroid_head
 * writes).  q_j = softmax(logits / T) over the candidates and 0 elsewhere; the
 * rule is spec_verify_sample's ("Gemma 4 Multi-Token Prediction (MTP) 深度解析"
 * §2.2): accept iff u_accept < p(d)/q(d), a draft that is not a candidate
 * (q(d) = 0) is accepted; after a rejection at n the token is drawn from
 * max(0, p_n - q_n), which is p_n itself on every non-candidate token; after
 * a full acceptance the bonus is drawn from p_gamma.  Only the target rows are
 * streamed.  out_debug's L_q is the normaliser over the candidates.
 *
 * target_logits [B, gamma+1, V] f32 or bf16 (16-byte aligned, V % 8 == 0);
 * cand_stride >= 1; counts outside [0, cand_stride] are clamped.  Other
 * arguments, ownership and errors as spec_verify_sample; the workspace comes
 * from spec_verify_sparse_workspace_bytes.
 */
int spec_verify_sparse_workspace_bytes(int B, int gamma, int V, size_t *bytes);

int spec_verify_sample_sparse(const void *target_logits, spec_dtype dt, const int32_t *cand_tok,
                              const float *cand_logit, const int32_t *cand_count,
                              int cand_stride, const int32_t *draft_tokens,
                              const float *temperature, const float *u_accept,
                              const float *u_resample, int B, int gamma, int V,
                              int32_t *out_tokens, int32_t *out_num_accepted,
                              float *out_debug, void *workspace, size_t workspace_bytes,
                              void *stream);

/*
 * Timing / profiling aid: the same arguments and checks as
 * spec_verify_sample, but only the first kernel of its launch chain (the
 * vocab-row reducer, which streams every logit the call reads) is enqueued,
 * in the launch configuration spec_verify_sample uses.  Outputs are not
 * written.  A later spec_verify_sample call is unaffected.
 */
int spec_verify_sample_reduce_only(const void *target_logits, const void *draft_logits,
                                   spec_dtype dt, const int32_t *draft_tokens,
                                   const float *temperature, const float *u_accept,
                                   const float *u_resample, int B, int gamma, int V,
                                   int32_t *out_tokens, int32_t *out_num_accepted,
                                   float *out_debug, void *workspace,
                                   size_t workspace_bytes, void *stream);

/*
 * spec_verify_sample without a workspace, for callers that cannot allocate
 * device memory (the pages have no counterpart: this is an integration aid).
 * Such callers include plugins or custom ops inside an inference engine that
 * owns all device memory through its own pool, and decode loops where a
 * cudaMalloc could synchronise the device and stall other streams.
 *
 * Same arguments and results as spec_verify_sample, minus the workspace.  The
 * scratch is a fixed 16 MiB array built into the library; every GPU that
 * loads the library holds it until the process exits.  Problems whose
 * workspace (spec_verify_workspace_bytes) exceeds 16 MiB are rejected with
 * SPEC_ERR_WORKSPACE (B=128, gamma=8, V=262144 needs about 9 MB).
 *
 * - The first call on a device, with that device current, looks up the
 *   array's address (cudaGetSymbolAddress; no memory is touched).  Every
 *   call then clears the array's header and counters with cudaMemsetAsync on
 *   the caller's stream, ahead of its kernel, so calls on any stream (a
 *   non-blocking one included) start from a clean scratch.  Nothing is ever
 *   allocated or freed.
 * - All calls share the one array: calls that overlap on the GPU (other
 *   streams, other host threads) race and give wrong tokens.  Serialise them.
 * - Device-side errors are recorded in the built-in scratch but cannot be
 *   read back through this entry point; host-side checks return codes as
 *   usual.  A draft token outside [0, V) is treated as rejected at its
 *   position (greedy: replaced by the target argmax; sampling: the residual
 *   draw runs there), so the outputs are well formed but meaningless for
 *   that sequence; other sequences of the call are unaffected.  Callers that
 *   cannot rule such tokens out should use spec_verify_sample and
 *   spec_verify_status.
 */
int spec_verify_sample_noalloc(const void *target_logits, const void *draft_logits,
                               spec_dtype dt, const int32_t *draft_tokens,
                               const float *temperature, const float *u_accept,
                               const float *u_resample, int B, int gamma, int V,
                               int32_t *out_tokens, int32_t *out_num_accepted,
                               float *out_debug, void *stream);

/*
 * Rejection-sampling verification with the target logits computed in the
 * call: l[b, j, x] = sum_k hidden[b*(gamma+1)+j, k] * W[x, k], the target's
 * final hidden states times its output embedding (tied to the input
 * embedding: "Gemma 4 Multi-Token Prediction (MTP) 深度解析" §3.1; "Gemma 4 -
 * Drafter 解析", 高效 Embedder).  The GEMM runs on the tcgen05 tensor cores
 * (bf16 operands, fp32 accumulation) and the target logits are reduced to
 * the verify statistics as they leave the accumulator; only rows j < gamma of
 * sampling sequences are stored (fp32, in the workspace) because the residual
 * max(0, p_n - q_n) needs them after the decision.  The rule, the uniforms and
 * the outputs are those of spec_verify_sample.
 *
 *   hidden        [B*(gamma+1), H] bf16: rows b*(gamma+1) .. b*(gamma+1)+gamma
 *                 are sequence b's verify positions 0..gamma
 *   W             [V, H] bf16
 *   draft_logits  [B, gamma, V] bf16
 *   draft_tokens, temperature, u_accept, u_resample, out_*: as spec_verify_sample
 *
 * Limits: B*(gamma+1) <= 384 rows, H a multiple of 64 in [64, 65536], V a
 * multiple of 8; hidden, W and draft_logits 16-byte aligned.  Beyond the row
 * limit the call returns SPEC_ERR_UNSUPPORTED.  The workspace must come from
 * spec_verify_workspace_bytes(B, gamma, V, H, ...).
 */
int spec_verify_lmhead_sample(const void *hidden, const void *W, const void *draft_logits,
                              const int32_t *draft_tokens, const float *temperature,
                              const float *u_accept, const float *u_resample, int B,
                              int gamma, int V, int H, int32_t *out_tokens,
                              int32_t *out_num_accepted, float *out_debug,
                              void *workspace, size_t workspace_bytes, void *stream);

/*
 * Timing / profiling aid: the same arguments and checks as
 * spec_verify_lmhead_sample, but only its lm_head GEMM kernel is enqueued, in
 * the launch configuration that call uses, and without the draft rows' chunk
 * statistics that kernel also computes in a whole call.  Outputs are not
 * written.
 */
int spec_verify_lmhead_gemm_only(const void *hidden, const void *W, const void *draft_logits,
                                 const int32_t *draft_tokens, const float *temperature,
                                 const float *u_accept, const float *u_resample, int B,
                                 int gamma, int V, int H, int32_t *out_tokens,
                                 int32_t *out_num_accepted, float *out_debug,
                                 void *workspace, size_t workspace_bytes, void *stream);

/*
 * Host bookkeeping after a verify round (HOST pointers; no GPU work).
 *
 * Per sequence the caller keeps seq_len (prompt + emitted tokens), kv_len
 * (entries in the target's KV cache) and gamma (the next round's draft
 * length).  Between rounds the newest token has no KV entry yet, so
 * kv_len == seq_len - 1.  Given num_accepted[b] = n from the verify call
 * (0 <= n <= gamma), spec_round_update sets, for every sequence:
 *   seq_len += n + 1   (accepted drafts + the replacement / resampled / bonus
 *                       token: "第 8 章 …", 多出来的那一个 token 从哪来)
 *   kv_len  += n + 1   and kv_keep[b] = the new kv_len: the verify pass
 *                       appended gamma + 1 entries; the caller keeps the first
 *                       kv_keep[b] and drops the rest ("自投机解码 …" §3.3:
 *                       trim to the accepted length; cache and sequence
 *                       lengths must agree after every round)
 *   gamma   += 2 if n == gamma, else gamma -= 1, clamped to
 *                       [gamma_min, gamma_max] ("Gemma 4 Multi-Token
 *                       Prediction (MTP) 深度解析" §5.1, the heuristic
 *                       schedule; the page finds drafts beyond about 10
 *                       tokens rarely pay)
 * All sequences are checked first (kv_len == seq_len - 1, 0 <= n <= gamma,
 * gamma >= 1): if one fails, nothing is changed, *first_bad (optional) gets
 * its index and SPEC_ERR_STATE is returned.  Bad arguments (NULL states or
 * counts, B < 0, gamma_min < 1, gamma_max > SPEC_MAX_GAMMA, gamma_min >
 * gamma_max) return SPEC_ERR_INVALID_ARG.  kv_keep [B] may be NULL.
 */
typedef struct {
  int32_t gamma;
  int32_t reserved;
  int64_t seq_len;
  int64_t kv_len;
} spec_round_state;

int spec_round_update(spec_round_state *states, const int32_t *num_accepted, int B,
                      int gamma_min, int gamma_max, int64_t *kv_keep, int *first_bad);

/*
 * Synchronise `stream`, then return the device-side status recorded in
 * `workspace` since the last call (SPEC_OK, SPEC_ERR_TIMEOUT or
 * SPEC_ERR_DEVICE_INPUT) and clear it.  Returns SPEC_ERR_CUDA if the
 * synchronisation itself fails.
 */
int spec_verify_status(void *workspace, void *stream);

/*
 * Self-test of the bounded waits: enqueue one tiny kernel whose only wait can
 * never be satisfied; it gives up after about a millisecond, records
 * SPEC_ERR_TIMEOUT in `workspace` and returns, leaving the context usable.
 * spec_verify_status() then reports SPEC_ERR_TIMEOUT.  No data is read.
 */
int spec_verify_selftest_timeout(void *workspace, size_t workspace_bytes, void *stream);

/* Static description of an error code. */
const char *spec_verify_error_string(int code);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
int spec_verify_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */
