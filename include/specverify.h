/*
 * specverify.h - C ABI of the GB300 speculative-sampling verification library
 * (libspecverify.so, CUDA for sm_103a).
 *
 * What is computed (citations name the page and its section):
 *   - Acceptance: draft token x is accepted iff u < min(1, p(x)/q(x)) with u an
 *     independent uniform in [0,1).  whoami-wesleyyou.top "Speculative
 *     Decoding" notes, section "Acceptance 与 correction"; wineandchord.com
 *     "推测解码：接受规则、状态与收益边界", section "单位置接受 reference".
 *   - Correction: at the first rejection the replacement token is drawn from
 *     norm([p - q]+); if all drafts are accepted a bonus token is drawn from
 *     the next target row.  Same notes, section "从单个 token 接到一段 draft";
 *     tannlonggtaoo.github.io "Speculative Decoding", section "算法".
 *   - Policy: p and q come from logits through each side's temperature,
 *     top-k and softmax; temperature 0 is greedy (accept iff the draft equals
 *     the argmax, correction = argmax).  Notes section "从 LM head 到 sampling
 *     distribution"; "Speculative Decoding" (tannlonggtaoo), section "Greedy
 *     Sampling".
 *   - Tree: recursive rejection over siblings (after a rejection p becomes
 *     norm([p - q]+) and the next sibling is tested).  Notes section "Token
 *     Tree Verifier"; zzszmyf.github.io "LLM 推测解码精读笔记 · 04 EAGLE",
 *     section 6.2.
 *   - Tree mask: each node sees itself and its ancestors; position = depth.
 *     Notes section "Token Tree Verifier: topology-aware causal mask";
 *     jennyma11.github.io "11.3 Self-Draft", section 11.3.4 Tree Attention.
 *   - Overlap (spec_overlap): beta_i = sum_v min(p_i(v), q_i(v)), the
 *     acceptance rate of draft position i.  Notes section "Correction 为什么
 *     用正残差".
 *   - Typical acceptance (spec_typical_accept): an approximate rule, not
 *     distribution-exact; p(x_i) > min(epsilon, delta exp(-H(p_i))), longest
 *     passing prefix, then the target's greedy token.  Notes section
 *     "Medusa-1 与 typical acceptance".
 *   - EAGLE-2 rerank (spec_tree_rerank): the m nodes of highest product of
 *     confidences along the path, shallow nodes first on ties.
 *     zzszmyf.github.io "LLM 推测解码精读笔记 · 04 EAGLE", section 10.3.
 *
 * Readings where the pages are silent (fixed here, identical in the tests):
 *   greedy/argmax ties -> lowest index; top-k keeps every logit >= the k-th
 *   largest raw logit (k <= 0 or k >= V: no filter); draws use the inverse CDF
 *   in index order (smallest v whose running sum exceeds u * total; if
 *   rounding leaves none, the largest v with positive weight); uniforms are
 *   Philox4x32-10 with key (seed lo, seed hi), counter (seq, pos, draw, 0),
 *   u = (word0 >> 8) * 2^-24; draw 0 = acceptance uniform, draw 1 = draw
 *   uniform.
 *
 * Conventions for every entry point:
 *   - All array pointers are DEVICE pointers owned by the caller; the library
 *     allocates nothing.  Work is enqueued on `stream` and the call returns
 *     without synchronising.
 *   - Host-checkable problems (a NULL required pointer, a negative size, a
 *     stride shorter than the row, a size above the limits below, a workspace
 *     that is too small) return SPEC_ERR_INVALID_ARG before anything is
 *     launched.  SPEC_ERR_UNSUPPORTED means the call cannot be run by this
 *     build: a vocabulary beyond the limits below (the verifiers), or a
 *     top-k, top-p or min-p policy passed to spec_overlap or
 *     spec_typical_accept.
 *     SPEC_ERR_CUDA reports a failed launch (cudaGetLastError).
 *   - Data-dependent problems never trap the GPU: they set per-sequence flag
 *     bits (SPEC_FLAG_*) and the sequence takes the defined fallback.
 *   - Logit rows must start on 16-byte boundaries for the vectorised path;
 *     other strides are accepted and take a scalar-load path.
 *   - The workspace needs no initialisation: each call first clears, with
 *     one cudaMemsetAsync on `stream`, the part of it that must start at zero
 *     (arrival counters and the weight-task queue).  Calls that share one
 *     workspace must not overlap on the GPU.
 *
 * Limits: 0 <= gamma <= 4095; 1 <= N <= 4096; V >= 1, and for the verifiers
 * a V that the call's kernel path takes (SPEC_ERR_UNSUPPORTED otherwise):
 *   - chains of gamma <= 31 with 16-byte-aligned rows (with or without a
 *     row filter: top-k, top-p, min-p) stream their rows: V <= 2,097,152;
 *   - trees of at most 256 nodes with aligned rows and no row filter stream
 *     their rows and walk the accepted path: V <= 2,097,152;
 *   - larger trees and longer chains with aligned rows and no row filter
 *     stream slices of at most 32 KB, 64 per row: V <= 1,048,576 bf16 /
 *     524,288 fp32;
 *   - rows with a filter, or unaligned rows, hold a target+draft row pair in
 *     16 thread blocks' shared memory: about 800k bf16 or 400k fp32 entries.
 * spec_overlap and spec_typical_accept read rows from global memory and take
 * any V >= 1.
 */
#ifndef SPECVERIFY_H
#define SPECVERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *spec_stream_t;

typedef enum {
  SPEC_OK = 0,
  SPEC_ERR_INVALID_ARG = 1,
  SPEC_ERR_CUDA = 2,
  SPEC_ERR_UNSUPPORTED = 3
} spec_status;

typedef enum { SPEC_F32 = 0, SPEC_BF16 = 1 } spec_dtype;

/* Per-sequence (or per-tree) policy arrays, device memory.
 *   temperature [B]: 0 -> greedy; > 0 -> softmax(z / T); NaN, < 0 or inf ->
 *                    the row is flagged SPEC_FLAG_NONFINITE.  Required.
 *   top_k [B]:       k-th largest raw logit filter; <= 0 or >= V: off.
 *                    May be NULL (no filtering).
 *   top_p [B]:       nucleus filter on the distribution after temperature and
 *                    top-k: keep the most probable values until their mass
 *                    reaches top_p (every entry tied with the boundary value
 *                    is kept); >= 1 or NaN: off; <= 0: the most probable
 *                    value only.  May be NULL.
 *   min_p [B]:       after top-p, keep p(x) >= min_p * max p; <= 0 or NaN:
 *                    off; > 1 is taken as 1.  May be NULL.
 *   Both sides of a verification must apply the policies they sampled with
 *   (wineandchord.com "推测解码：接受规则、状态与收益边界", section
 *   "与 Logit Processor 的组合" lists top-k, top-p and min-p among the
 *   processors p and q must both reflect); each filter renormalises.  A call
 *   with any top-k, top-p or min-p array runs on the cluster kernel that holds
 *   each row pair in shared memory; greedy rows ignore the filters.  The
 *   floating-point top-p boundary is decided on single-precision masses summed
 *   exactly in fixed point, so a boundary whose cumulative mass lies within
 *   about 1e-6 of top_p may fall on either side. */
typedef struct {
  const float *temperature;
  const int32_t *top_k;
  const float *top_p;
  const float *min_p;
} spec_policy;

/* Per-sequence flag bits (uint32). */
#define SPEC_FLAG_BAD_TOKEN 1u           /* draft token outside [0, V): rejected there */
#define SPEC_FLAG_ZERO_Q 2u              /* q(x) == 0 for a draft token: rejected there */
#define SPEC_FLAG_NONFINITE 4u           /* NaN/+inf logit, no finite logit, or bad T:
                                            the row becomes one-hot at its finite argmax
                                            (index 0 if none) */
#define SPEC_FLAG_DEGENERATE_RESIDUAL 8u /* sum [p - q]+ <= 0 at a rejection: the chain
                                            draws from p; the tree keeps its current p */
#define SPEC_FLAG_DEPTH 16u              /* a tree node deeper than max_depth */
#define SPEC_FLAG_TIMEOUT 32u            /* a bounded on-device wait gave up; on the
                                            streaming chain path the sequence then
                                            gets the fallback outputs: 0 accepted
                                            drafts, every token -1; on the tree walk
                                            path the tree: 0 accepted nodes, every
                                            path entry and token -1 */
#define SPEC_FLAG_BAD_TREE 64u           /* parent[0] != -1 or parent[n] not in [0, n) */

/* Bytes of workspace spec_verify_chain needs for B sequences of gamma drafts
 * (0 for a negative size, V < 1 or an unknown dtype). */
size_t spec_verify_chain_workspace_size(int B, int gamma, int V, spec_dtype dtype);

/* Chain verification of B sequences with gamma drafts each.
 *
 * target_logits [B, gamma+1, V]: row (b, i) at target_logits + (b*(gamma+1)+i)*ld_target
 *                                elements; rows i < gamma score draft i, row gamma is
 *                                the bonus position.
 * draft_logits  [B, gamma, V]:   row (b, i) at draft_logits + (b*gamma+i)*ld_draft; the
 *                                distribution draft token i was drawn from.  Never read
 *                                for sequences whose target temperature is 0.
 * draft_tokens  [B, gamma] int32.
 * uniform_override: NULL -> Philox keyed (seed, b, i, draw); else float [B, gamma+1, 2]
 *                   in [0,1): [b,i,0] acceptance uniform of draft i, [b,i,1] draw
 *                   uniform when position i samples (correction or bonus).
 * Outputs (device):
 *   out_num_accepted [B]: number of accepted drafts j (0..gamma).
 *   out_tokens [B, gamma+1]: the j accepted drafts, then the correction (j < gamma)
 *                            or bonus (j == gamma) token, then -1.
 *   out_flags [B] (nullable): OR of the SPEC_FLAG_* raised on positions 0..j.
 *   out_residual [B, V] float (nullable): the distribution the correction token was
 *                            drawn from (norm([p_j - q_j]+), p_j on a degenerate
 *                            residual, one-hot for greedy rows); zeros when all
 *                            drafts were accepted.
 */
spec_status spec_verify_chain(
    const void *target_logits, int64_t ld_target,
    const void *draft_logits, int64_t ld_draft,
    spec_dtype dtype, int B, int gamma, int V,
    const int32_t *draft_tokens,
    spec_policy target_policy, spec_policy draft_policy,
    uint64_t seed, const float *uniform_override,
    int32_t *out_num_accepted, int32_t *out_tokens,
    uint32_t *out_flags, float *out_residual,
    void *workspace, size_t workspace_bytes, spec_stream_t stream);

/* Size of the scratch array spec_verify_chain_static works in (16 MiB). */
#define SPEC_STATIC_SCRATCH_BYTES (16u * 1024u * 1024u)

/* spec_verify_chain without a caller workspace: the call allocates nothing.
 *
 * The pages have no counterpart of this entry point; it exists for callers
 * that cannot allocate device memory at the call site: a decode loop whose
 * device memory is reserved up front by its own pool (the KV cache takes the
 * rest, so a per-shape workspace has nowhere to come from), or a plain C host
 * without a device allocator of its own.  Arguments, outputs, limits and
 * results are those of spec_verify_chain (it forwards to it).
 *
 * Workspace: a file-scope device array of SPEC_STATIC_SCRATCH_BYTES inside
 *   this library, one per device.  The call uses no cudaMalloc, cudaFree or
 *   any other allocating routine.
 * Size limit: shapes with spec_verify_chain_workspace_size(B, gamma, V, dtype)
 *   > SPEC_STATIC_SCRATCH_BYTES return SPEC_ERR_UNSUPPORTED before any CUDA
 *   call; use spec_verify_chain there.  For V = 128256 bf16 and gamma = 7,
 *   B = 512 fits (9.6 MiB) and B = 1024 does not (19.1 MiB).
 * Address: every call looks the array's address up with cudaGetSymbolAddress
 *   in the device context current on the calling thread, so a call made after
 *   a device reset works in the new context.  The first call on each device
 *   may load this library's device code for that device: make it outside any
 *   stream capture.  A failed lookup returns SPEC_ERR_CUDA.
 * Errors: the arguments are checked exactly as spec_verify_chain checks them
 *   (SPEC_ERR_INVALID_ARG) before the size limit below is applied.
 * Zero state: none is needed; like spec_verify_chain, every call clears the
 *   counters and task queue it uses (one cudaMemsetAsync on `stream`).
 * Concurrency: all calls on one device share the one array, so calls whose
 *   GPU work could overlap (different streams without ordering between them)
 *   race on it and give undefined results; order them on one stream.
 */
spec_status spec_verify_chain_static(
    const void *target_logits, int64_t ld_target,
    const void *draft_logits, int64_t ld_draft,
    spec_dtype dtype, int B, int gamma, int V,
    const int32_t *draft_tokens,
    spec_policy target_policy, spec_policy draft_policy,
    uint64_t seed, const float *uniform_override,
    int32_t *out_num_accepted, int32_t *out_tokens,
    uint32_t *out_flags, float *out_residual, spec_stream_t stream);

/* Bytes of workspace spec_verify_tree needs for T trees of N nodes (0 as above). */
size_t spec_verify_tree_workspace_size(int T, int N, int V, spec_dtype dtype);

/* Tree verification of T candidate trees of N nodes each (recursive rejection).
 *
 * target_logits [T, N, V]: row (t, n) = target next-token logits after the path
 *                          root..n, at target_logits + (t*N+n)*ld_target.
 * draft_logits  [T, N, V]: row (t, n) = the draft logits the children of n were
 *                          drawn from (rows of leaves are never read).
 * node_tokens [T, N], parent [T, N] int32: node 0 is the root (token ignored,
 *                          parent -1); parent[n] < n.  Children of a node are
 *                          tested in ascending node id.
 * max_depth >= 0: the deepest allowed node; outputs hold max_depth+1 entries.
 * uniform_override: NULL or float [T, N, 2]: [t,c,0] acceptance uniform of child
 *                   c, [t,n,1] draw uniform at node n.  Philox keys: (seed, t, c, 0)
 *                   and (seed, t, n, 1).
 * Outputs:
 *   out_num_accepted [T]: accepted draft nodes on the path; -1 when the tree is
 *                          invalid (SPEC_FLAG_BAD_TREE) or too deep (SPEC_FLAG_DEPTH).
 *   out_path [T, max_depth+1]: accepted node ids, root first, then -1.
 *   out_tokens [T, max_depth+1]: accepted node tokens, then the final (correction
 *                          or bonus) token, then -1.
 *   out_flags [T] (nullable), out_residual [T, V] (nullable): the distribution the
 *                          final token was drawn from when every child of the last
 *                          node was rejected; zeros for a bonus draw at a leaf.
 * Launches (trees of at most 256 nodes, aligned rows, no row filter): one
 * cudaMemsetAsync, then the first-child, rows, walk and refine kernels; the
 * rows kernel reads every target row and the draft rows of internal nodes once,
 * the walk re-reads the row pair of each node where a sibling is rejected.
 */
spec_status spec_verify_tree(
    const void *target_logits, int64_t ld_target,
    const void *draft_logits, int64_t ld_draft,
    spec_dtype dtype, int T, int N, int V, int max_depth,
    const int32_t *node_tokens, const int32_t *parent,
    spec_policy target_policy, spec_policy draft_policy,
    uint64_t seed, const float *uniform_override,
    int32_t *out_num_accepted, int32_t *out_path, int32_t *out_tokens,
    uint32_t *out_flags, float *out_residual,
    void *workspace, size_t workspace_bytes, spec_stream_t stream);

/* Ancestor-or-self masks and depth position ids for T trees of N nodes.
 *
 * out_mask [T, N, (N+63)/64] uint64: bit m of word m/64 of node n is set iff m == n
 *          or m is an ancestor of n.
 * out_position [T, N] int32: depth of n (root 0); -1 when n's parent chain hits an
 *          invalid link before the root (the mask then holds the part reached).
 * out_flags [T] (nullable): SPEC_FLAG_BAD_TREE, SPEC_FLAG_DEPTH (depth > max_depth).
 */
spec_status spec_tree_mask(const int32_t *parent, int T, int N, int max_depth,
                           uint64_t *out_mask, int32_t *out_position,
                           uint32_t *out_flags, spec_stream_t stream);

/* Per-position overlap of a draft chain: beta_i = sum_v min(p_i(v), q_i(v)),
 * the acceptance rate of draft position i (1 - beta_i is the mass of the
 * residual [p_i - q_i]_+).  whoami-wesleyyou.top "Speculative Decoding"
 * notes, section "Correction 为什么用正残差" (beta := sum_x min{p(x), q(x)}).
 *
 * Inputs as for spec_verify_chain (target rows [B, gamma+1, V], draft rows
 * [B, gamma, V]; target row i and draft row i are compared for i < gamma).
 * Policies: temperature per sequence (0: greedy, the one-hot at the argmax);
 * the top_k pointers must be NULL (SPEC_ERR_UNSUPPORTED otherwise).  A row
 * whose temperature or logits are not finite is the one-hot at its finite
 * argmax and sets SPEC_FLAG_NONFINITE in out_flags.
 *
 * out_beta [B, gamma] float: beta_i of sequence b at b * gamma + i.
 * out_flags [B] (nullable): cleared by the call, then SPEC_FLAG_NONFINITE.
 * No workspace.  B = 0 or gamma = 0 is a no-op; B * gamma above 2^28 - 1 is
 * SPEC_ERR_INVALID_ARG (one cluster of up to 4 CTAs per position).  Arguments are
 * checked on the host before any launch; a CUDA launch error is
 * SPEC_ERR_CUDA and leaves out_beta undefined.
 */
spec_status spec_overlap(
    const void *target_logits, int64_t ld_target,
    const void *draft_logits, int64_t ld_draft,
    spec_dtype dtype, int B, int gamma, int V,
    spec_policy target_policy, spec_policy draft_policy,
    float *out_beta, uint32_t *out_flags, spec_stream_t stream);

/* Static description of a status code. */
const char *spec_status_string(spec_status status);

/* Profiling hook (the pages have no counterpart; it exists so that a benchmark
 * can time the dominant kernel of a chain verification live, on the stream the
 * kernel runs on).
 *
 * start_event, stop_event: cudaEvent_t handles (as void *) created by the
 *   caller, or both NULL to switch the hook off.  While set, every
 *   spec_verify_chain / spec_verify_chain_static call that takes the streaming
 *   path (16-byte aligned rows, no top-k, gamma <= 31) records start_event
 *   immediately before and stop_event immediately after its rows kernel (the
 *   pass that reads every logit row once) on the call's stream.  Other calls
 *   record nothing.
 * The setting is process-wide, not per thread; the library does not own or
 * destroy the events.  Returns SPEC_ERR_INVALID_ARG when exactly one of the
 * two is NULL (the previous setting is kept), SPEC_OK otherwise.
 */
spec_status spec_set_profile_events(void *start_event, void *stop_event);

/* Bound on one on-device wait (diagnostics and tests; the pages have no
 * counterpart).  Every wait inside the kernels gives up after a bound (about two
 * seconds by default) and sets SPEC_FLAG_TIMEOUT instead of hanging.  This
 * shortens the first wait the streaming chain path's rows kernel makes for each
 * chunk to `cycles` SM clock cycles (0: a single non-blocking test); negative
 * restores the default.  When that wait gives up the kernel flags the call and
 * then waits again with the full bound, so no copy is left in flight and the
 * call completes; every sequence of the call gets SPEC_FLAG_TIMEOUT and the
 * fallback outputs.  Process-wide, read at each call's launch.  Returns SPEC_OK.
 */
spec_status spec_set_wait_limit(int64_t cycles);

/* Bytes of workspace spec_typical_accept needs for B sequences of gamma
 * drafts over a vocabulary of V entries of type dtype: 256 bytes, 8 per target
 * row (B (gamma + 1) rows), and 128 per 32 KB of each target row (the streaming
 * form's records).  0 for a negative size, V < 1 or an unknown dtype. */
size_t spec_typical_workspace_size(int B, int gamma, int V, spec_dtype dtype);

/* Typical acceptance of a draft chain (an approximate rule: the output is not
 * distributed as the target's).  whoami-wesleyyou.top "Speculative Decoding"
 * notes, section "Medusa-1 与 typical acceptance": draft token x_i passes when
 * p_i(x_i) > min(epsilon, delta * exp(-H(p_i))), H the entropy (natural log)
 * of the target's distribution at position i; the longest passing prefix is
 * kept and the target's greedy token follows it.
 *
 * target_logits [B, gamma+1, V]: as for spec_verify_chain; every row is read
 *                                once (rows past the first failure too).
 * draft_tokens  [B, gamma] int32 (may be NULL when gamma == 0).
 * target_policy: temperature per sequence (0: greedy, the one-hot at the
 *                argmax, H = 0); top_k must be NULL (SPEC_ERR_UNSUPPORTED).
 * epsilon, delta: finite, >= 0.
 * Outputs (device):
 *   out_num_accepted [B]: length n of the passing prefix (0..gamma).
 *   out_tokens [B, gamma+1]: the n passing drafts, then the greedy token of row
 *                            n (the lowest index of the largest logit), then -1.
 *   out_flags [B] (nullable): OR over rows 0..n of SPEC_FLAG_NONFINITE (a NaN or
 *                            +inf logit, no finite logit, or a bad temperature:
 *                            the row is the one-hot at its finite argmax) and
 *                            SPEC_FLAG_BAD_TOKEN (x_n outside [0, V): it fails).
 * workspace: device, >= spec_typical_workspace_size(B, gamma, V, dtype)
 *            bytes, 8-byte aligned; no contents carried between calls (each
 *            call first clears its first 256 bytes).
 * Errors: SPEC_ERR_INVALID_ARG (bad sizes, NULL pointers, ld_target < V, a
 * short or misaligned workspace, epsilon or delta negative or not finite),
 * before any launch; SPEC_ERR_CUDA for a failed launch.  16-byte-aligned rows
 * take the streaming form: one cudaMemsetAsync and three launches (the rows
 * stream, a merge, the walk); other rows two launches.  A bounded wait of the
 * stream that gives up sets SPEC_FLAG_TIMEOUT, 0 accepted drafts and every
 * token -1.
 */
spec_status spec_typical_accept(
    const void *target_logits, int64_t ld_target, spec_dtype dtype,
    int B, int gamma, int V, spec_policy target_policy,
    const int32_t *draft_tokens, float epsilon, float delta,
    int32_t *out_num_accepted, int32_t *out_tokens, uint32_t *out_flags,
    void *workspace, size_t workspace_bytes, spec_stream_t stream);

/* EAGLE-2 rerank of T draft trees of N nodes: keep the m nodes of highest
 * value.  zzszmyf.github.io "LLM 推测解码精读笔记 · 04 EAGLE：特征空间草稿",
 * section 10.3: value(t_i) is the product of the confidences c_j on the path
 * from the root to t_i; the m nodes of highest value over the whole tree are
 * kept, ties to the shallower node (then to the lower index).  Since c <= 1
 * the kept set is a connected tree; it is returned in ascending node order
 * with re-indexed parents, ready for spec_tree_mask.
 *
 * parent [T, N] int32: node 0 is the root (parent -1), 0 <= parent[n] < n.
 * confidence [T, N] float: c_n in [0, 1]; values outside (or NaN) are
 *                clamped into [0, 1] (NaN -> 0) and flag SPEC_FLAG_NONFINITE.
 *                value[n] = value[parent[n]] * c[n] in float32, value[0] = c[0].
 * 1 <= N <= 4096, m >= 1.
 * Outputs (device):
 *   out_nodes [T, m] int32: the kept node ids, ascending, then -1.
 *   out_parent [T, m] int32: each kept node's parent as a position in
 *                            out_nodes (-1 for the root), then -1.
 *   out_value [T, m] float (nullable): their values, then 0.
 *   out_count [T] int32: min(m, N), or 0 for an invalid tree.
 *   out_flags [T] (nullable): SPEC_FLAG_BAD_TREE (invalid parent array:
 *                             nothing kept), SPEC_FLAG_NONFINITE (clamped).
 * Errors: SPEC_ERR_INVALID_ARG (bad sizes or NULL pointers) before any launch;
 * SPEC_ERR_CUDA for a failed launch.  T = 0 is a no-op.  One launch.
 */
spec_status spec_tree_rerank(const int32_t *parent, const float *confidence, int T, int N, int m,
                             int32_t *out_nodes, int32_t *out_parent, float *out_value,
                             int32_t *out_count, uint32_t *out_flags, spec_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SPECVERIFY_H */
