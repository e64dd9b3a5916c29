/*
 * spec_tree.h — C ABI of the GB300 token-tree verification library
 * (libspec_tree.so, hand-written CUDA for sm_103a).
 *
 * The library computes the data-parallel hot path of tree-based speculative
 * decoding: the tree mask, tree attention over a contiguous KV cache, and
 * verification of the speculated tree against the target model's logits.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - All array pointers are DEVICE pointers owned by the caller.  The library
 *    never allocates device memory and keeps no state between calls, except
 *    for the fixed scratch array that spec_tree_verify_static uses.
 *  - Every call is asynchronous on `stream` (a cudaStream_t passed as void*;
 *    NULL means the legacy default stream).  No call synchronises the host.
 *  - A call launches on the calling thread's current CUDA device; its
 *    pointers and stream must belong to that device.  Calls may come from
 *    several threads and go to several devices in one process: what the
 *    library caches about a device (kernel shared-memory limits, the SM
 *    count) is kept per device.  Calls whose work overlaps must not share a
 *    workspace; spec_tree_verify_static shares one array per device among
 *    all its calls (see there).
 *  - Host-detectable errors (null pointers, bad sizes, workspace too small)
 *    return a negative spec_status synchronously and launch nothing.
 *  - Data-dependent errors found on the device (a malformed parent array, a
 *    tree larger than SPEC_MAX_TREE_NODES, a token outside [0, V), a prefix
 *    that does not fit the cache, a bounded wait that ran out) are written to
 *    the caller's `status[b]` for request b with an atomic compare-and-swap
 *    from 0, so the first error sticks.  The kernels never write 0: the caller
 *    zero-fills `status` before a step and reads it after synchronising.  A
 *    call leaves the outputs of a request untouched when it finds an error
 *    for that request itself; codes that other calls wrote into `status`
 *    (which may run concurrently on other streams) do not affect it.  After
 *    SPEC_ERR_TIMEOUT (never expected) the request's outputs are unspecified,
 *    and a verification workspace used by that call must be zero-filled
 *    again before its next use (a node whose CTAs disagree on the timeout
 *    may leave its request's arrival counter off zero).
 *  - A batch is packed ragged: request b owns global nodes
 *    [tree_offsets[b], tree_offsets[b+1]) with tree_offsets[0] = 0 and
 *    tree_offsets[B] = T.  Node indices inside a request (parents, path
 *    nodes) are request-local; node 0 of each request is its root.
 *  - A parent array satisfies parent[0] = -1 and 0 <= parent[i] < i, so node
 *    order is topological and siblings are ordered by index.
 *  - A return value of SPEC_OK means the work was enqueued.
 *  - Bounds-checked build (libspec_tree_checked.so, compiled with
 *    -DSPEC_CHECKED): every global access whose index is computed from the
 *    inputs (a tree offset, a parent, a token, a path node, a prefix length)
 *    is first tested against the extent of its buffer as the call's size
 *    arguments define it.  A failed test writes SPEC_ERR_INDEX to the
 *    request's status word (request 0's when the request is not known) and
 *    skips the access: a load yields 0, a store is dropped.  It never traps
 *    or asserts.  The host-side checks and the results are those of the
 *    normal build; only speed differs.  spec_build_checked() says which
 *    build is loaded.
 */
#ifndef SPEC_TREE_H
#define SPEC_TREE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SPEC_OK = 0,
  SPEC_ERR_NULL = -1,            /* a required pointer is NULL */
  SPEC_ERR_SHAPE = -2,           /* a size argument is out of range or unsupported */
  SPEC_ERR_DTYPE = -3,           /* unknown spec_dtype */
  SPEC_ERR_TREE_TOO_LARGE = -4,  /* N_b < 1, N_b > SPEC_MAX_TREE_NODES, bad offsets, or a path
                                    longer than the output rows */
  SPEC_ERR_BAD_PARENT = -5,      /* parent[0] != -1 or parent[i] not in [0, i) */
  SPEC_ERR_TOKEN_RANGE = -6,     /* a speculated token outside [0, V) */
  SPEC_ERR_WORKSPACE = -7,       /* workspace NULL or smaller than the _workspace_size value */
  SPEC_ERR_CUDA = -8,            /* a CUDA runtime call or launch failed */
  SPEC_ERR_TIMEOUT = -9,         /* a bounded device-side wait ran out (never expected) */
  SPEC_ERR_PREFIX_RANGE = -10,   /* prefix_lens[b] < 0 or L_b + N_b > S_cap */
  SPEC_ERR_ALIGNMENT = -11,      /* a pointer is not 16-byte aligned */
  SPEC_ERR_INDEX = -12           /* bounds-checked build only: a computed global index fell
                                    outside its buffer; the access was skipped */
} spec_status;

typedef enum { SPEC_F32 = 0, SPEC_BF16 = 1 } spec_dtype;

/* Largest tree (root included) one request may carry. */
#define SPEC_MAX_TREE_NODES 128

/*
 * spec_build_tree_mask — step A1, the tree-attention mask.
 *
 * Source: SpecInfer news write-up (sunluscious.com.cn), section
 * "Token 樹驗證器": verification uses a mask matrix built from the token tree;
 * SpecInfer developer article "SpecInfer：基于树结构的LLM推测性推理加速技术",
 * §2.1 (tree nodes keep a parent pointer; tree_attention snippet: a mask entry
 * of 0 hides the key).
 *
 * For every node i of request b: bit a of mask[i] is set iff a == i or a is
 * an ancestor of i (a node sees itself and its ancestors), and
 * depth[i] = number of edges from the root.
 *
 *   parents      [T]    int32, request-local parent indices (see conventions)
 *   tree_offsets [B+1]  int32
 *   mask         [T][4] uint32 out: 128-bit ancestor-or-self set, bit a of node
 *                       i is word a/32, bit a%32
 *   depth        [T]    int32 out
 *   status       [B]    int32 in/out (see conventions)
 * Errors on the device: SPEC_ERR_TREE_TOO_LARGE, SPEC_ERR_BAD_PARENT.
 */
int spec_build_tree_mask(const int32_t *parents, const int32_t *tree_offsets, int B, int T,
                         uint32_t *mask, int32_t *depth, int32_t *status, void *stream);

/*
 * Bytes of scratch spec_tree_attn needs for these sizes.  The kernels merge
 * their key splits on chip (the splits of a query block form one thread-block
 * cluster), so this is 0; the argument stays part of the ABI so a future
 * split layout needs no signature change.
 */
size_t spec_tree_attn_workspace_size(int B, int T, int Hq, int Hkv, int D, int max_prefix);

/*
 * spec_tree_attn — steps A2 and A3, tree attention with a split-KV merge.
 *
 * Source: SpecInfer developer article §2.1, tree_attention snippet (scores of
 * the queries against the keys, masked entries removed, softmax, times V);
 * SpecInfer news write-up "Token 樹驗證器" (the tree's K/V are appended to the
 * KV cache depth-first, so all paths decode in one pass).
 *
 * For node i of request b and query head h, with KV head g = h / (Hq/Hkv)
 * and scale s (softmax_scale, or 1/sqrt(D) when softmax_scale <= 0):
 *   o[i][h] = sum_{j in K(i)} softmax_j(s * q[i][h] . k[b][g][j]) * v[b][g][j]
 * where K(i) = {0 .. L_b-1} (the prefix) u {L_b + a : bit a of mask[i]}.
 * The tree's own K/V must already sit at cache slots [L_b, L_b + N_b) in node
 * order.  Slots >= L_b + N_b are never read into the result (they may hold
 * anything, NaN included).
 *
 *   q            [T][Hq][D]           dtype (bf16 or f32)
 *   k_cache,
 *   v_cache      [B][Hkv][S_cap][D]   dtype; 16-byte aligned
 *   o            [T][Hq][D]           dtype out
 *   dtype        SPEC_BF16 (tensor-core path) or SPEC_F32 (plain fp32 path)
 *   D            64 or 128;  Hq % Hkv == 0 and Hq / Hkv in {1, 2, 4, 8}
 *   max_prefix   host-side upper bound on every prefix_lens[b]; sizes the
 *                key splits (a larger value is safe, only slower)
 *   prefix_lens  [B] int32 (L_b)
 *   mask         [T][4] uint32 from spec_build_tree_mask (bits >= N_b ignored)
 *   workspace    may be NULL while spec_tree_attn_workspace_size() is 0
 * Accumulation is fp32; the bf16 path splits every softmax weight into a bf16
 * high part and a bf16 remainder for the P·V product (about 16 significant
 * bits per weight) and rounds o to bf16.
 * Errors on the device: SPEC_ERR_TREE_TOO_LARGE, SPEC_ERR_PREFIX_RANGE,
 * SPEC_ERR_TIMEOUT.
 */
int spec_tree_attn(const void *q, const void *k_cache, const void *v_cache, void *o, int dtype,
                   int B, int T, int Hq, int Hkv, int D, int S_cap, int max_prefix,
                   const int32_t *prefix_lens, const int32_t *tree_offsets, const uint32_t *mask,
                   float softmax_scale, void *workspace, size_t workspace_bytes, int32_t *status,
                   void *stream);

/*
 * spec_tree_attn_ex — spec_tree_attn with two options for a caller that runs
 * other kernels beside it (another stream, another graph branch).
 *
 *   max_ctas  the bf16 path plans its key splits (the CTAs of one query
 *             block) for at most max_ctas CTAs resident at once instead of
 *             the whole GPU, so that the other work keeps the SMs it needs.
 *             0 means the device's SM count (spec_tree_attn); negative is
 *             SPEC_ERR_SHAPE.  The result is the same; only the launch shape
 *             changes.  The fp32 path ignores it.
 *   parents   [T] int32, the request-local parent array of spec_build_tree_mask
 *             (device).  Read only when mask is NULL: then every row's
 *             ancestor set is built inside the kernel from the parents (the
 *             SpecInfer developer article's topology mask, §2.1), so the mask
 *             kernel need not run before this one.  The result equals the
 *             call with the mask spec_build_tree_mask writes for the same
 *             parents.  A parent that is not below its node, or a root whose
 *             parent is not -1, reports SPEC_ERR_BAD_PARENT for its request
 *             (the walk stops there; the request's outputs are then
 *             unspecified).  mask and parents both NULL is SPEC_ERR_NULL.
 */
int spec_tree_attn_ex(const void *q, const void *k_cache, const void *v_cache, void *o, int dtype,
                      int B, int T, int Hq, int Hkv, int D, int S_cap, int max_prefix,
                      const int32_t *prefix_lens, const int32_t *tree_offsets,
                      const uint32_t *mask, const int32_t *parents, float softmax_scale,
                      void *workspace, size_t workspace_bytes, int max_ctas, int32_t *status,
                      void *stream);

/*
 * Bytes of scratch spec_tree_verify needs: per-node acceptance flags and
 * fallback tokens plus one arrival counter per request.  The workspace must
 * be zero-filled before its FIRST use; every call leaves the counters at zero
 * again, so one buffer can be reused by later calls on the same stream.  Two
 * calls that run at the same time need two workspaces.
 */
size_t spec_tree_verify_workspace_size(int B, int T, int V);

/*
 * spec_tree_verify — steps V1-V4 and R, verification of the token tree.
 *
 * Sources: SpecInfer developer article §2.1 (the accept stage keeps the
 * longest verified prefix); speculative-decoding explainer
 * (intelliparadigm.com) §2.2 三阶段工作流程详解: stage 2 computes the accept
 * probability alpha = min(1, p_target / p_draft); stage 3 checks left to right,
 * stops at the first rejection and replaces it with a new target prediction,
 * keeping the output distribution equal to the target model's.
 *
 * Greedy (temperature == 0): at node u (starting at the root) accept the
 * first child, in index order, whose token equals argmax of u's target logits
 * (lowest index on ties); when none matches, emit that argmax and stop.
 * Stochastic (temperature > 0): p = softmax(target/temperature),
 * q = softmax(draft/temperature) of node u; with r = p, test u's children c in
 * index order: accept iff U(c) < min(1, r(x_c) / q(x_c)); after a rejection
 * r becomes max(0, r - q) renormalised (unchanged if that is all zero).  When
 * every child is rejected, or u is a leaf, emit a draw from r by inverse CDF
 * and stop.  The emitted tokens are the accepted path's tokens followed by
 * that one extra (bonus) token.
 * Uniforms: Philox4x64-10 with key (seed, 0) and counter (node, b, kind, 0),
 * node request-local, kind 0 for the accept test of child `node`, kind 1 for
 * the draw at `node`; U = (first output word >> 40) * 2^-24.
 *
 *   target_logits [T][V] f32
 *   draft_logits  [T][V] f32 (row u is the draft distribution u's children
 *                 were drawn from); may be NULL when temperature == 0
 *   tokens        [T] int32, the token node i proposes (the root's is ignored)
 *   parents       [T] int32
 *   accept_len    [B] int32 out: accepted speculated tokens (path length)
 *   path_nodes    [B][max_depth_plus1] int32 out: root (0), then the accepted
 *                 nodes; unused entries -1
 *   out_tokens    [B][max_depth_plus1] int32 out: accepted tokens then the
 *                 bonus token (accept_len + 1 entries); unused entries -1
 *   near_ties     [B] int32 out: decisions on the walked path whose uniform
 *                 lay within 1e-6 of its threshold (fp32 rounding could have
 *                 flipped them)
 *   max_depth_plus1  row stride of path_nodes / out_tokens; must exceed the
 *                 depth of every tree
 * Errors on the device: SPEC_ERR_TREE_TOO_LARGE, SPEC_ERR_BAD_PARENT,
 * SPEC_ERR_TOKEN_RANGE, SPEC_ERR_TIMEOUT.
 */
int spec_tree_verify(const float *target_logits, const float *draft_logits,
                     const int32_t *tokens, const int32_t *parents,
                     const int32_t *tree_offsets, int B, int T, int V, float temperature,
                     uint64_t seed, int32_t *accept_len, int32_t *path_nodes,
                     int32_t *out_tokens, int32_t *near_ties, int max_depth_plus1,
                     void *workspace, size_t workspace_bytes, int32_t *status, void *stream);

/*
 * spec_tree_verify_top_p — spec_tree_verify with the target and draft
 * distributions of every node filtered to their top_p nucleus first.
 *
 * Source: SpecInfer developer article, deployment configuration (top_p as
 * a sampling parameter of the serving system); the walk itself is the one
 * of spec_tree_verify.  Reading: tau is the largest probability whose upper
 * tail {x : p(x) >= tau} holds at least top_p of the mass; every entry of
 * that tail is kept (entries tied at tau included), the rest drop to 0, and
 * the tail is renormalised; q is filtered the same way with its own tau.
 * Verification of the filtered pair is lossless for the filtered target.
 *
 * Arguments, layouts, workspace and errors are those of spec_tree_verify,
 * plus top_p in (0, 1]; top_p >= 1 is spec_tree_verify; temperature 0
 * (greedy) ignores top_p (the argmax is in every nucleus).  The nucleus is
 * found by a radix search over the float bits of the probabilities with
 * their mass summed in 2^-40 fixed point; its membership follows each
 * entry's float value.  Near-ties (in near_ties) are counted, besides those
 * of spec_tree_verify, for a child whose probability is within 128 ulps of
 * tau, or a drawn token whose is, at a node where another entry lies that
 * close to tau (their exact order may differ).  Host errors: SPEC_ERR_SHAPE
 * for top_p <= 0 or NaN,
 * and for top_p < 1 with V > 131072 (the nucleus search runs in the
 * register-resident kernel only).
 */
int spec_tree_verify_top_p(const float *target_logits, const float *draft_logits,
                           const int32_t *tokens, const int32_t *parents,
                           const int32_t *tree_offsets, int B, int T, int V, float temperature,
                           float top_p, uint64_t seed, int32_t *accept_len, int32_t *path_nodes,
                           int32_t *out_tokens, int32_t *near_ties, int max_depth_plus1,
                           void *workspace, size_t workspace_bytes, int32_t *status, void *stream);

/*
 * spec_kv_compact — the depth-first KV-cache update after verification.
 *
 * Source: SpecInfer news write-up, section "Token 樹驗證器": the verifier
 * updates the KV cache depth-first, so the accepted path's keys and values
 * become the next step's prefix without extra storage.
 *
 * For request b with prefix L_b, tree nodes at cache slots [L_b, L_b + N_b)
 * and an accepted path (path_nodes / accept_len from spec_tree_verify): slot
 * L_b + j receives the old slot L_b + path_nodes[b][j] for j = 1 .. acc_b in
 * both caches, for every KV head; the root (slot L_b) and every other slot
 * are unchanged; new_prefix_lens[b] = L_b + 1 + acc_b (prefix, root and the
 * accepted tokens; the bonus token's keys and values come from the next
 * step).  The copy reads the old slots, so a slot that is both a destination
 * and a later source is handled.
 *
 *   k_cache, v_cache [B][Hkv][S_cap][D]   dtype, modified in place, 16-byte aligned
 *   prefix_lens      [B] int32 (L_b, before the update)
 *   tree_offsets     [B+1] int32
 *   path_nodes       [B][max_depth_plus1] int32, accept_len [B] int32
 *   new_prefix_lens  [B] int32 out (L_b for a skipped request)
 *   status           [B] int32 in/out: requests whose status is already
 *                    non-zero are skipped (caches untouched)
 * Errors on the device: SPEC_ERR_PREFIX_RANGE (L_b + N_b > S_cap),
 * SPEC_ERR_TREE_TOO_LARGE (acc_b + 1 > max_depth_plus1), SPEC_ERR_BAD_PARENT
 * (the path does not start at 0 or is not increasing inside the tree).
 */
int spec_kv_compact(void *k_cache, void *v_cache, int dtype, int B, int Hkv, int D, int S_cap,
                    const int32_t *prefix_lens, const int32_t *tree_offsets,
                    const int32_t *path_nodes, const int32_t *accept_len, int max_depth_plus1,
                    int32_t *new_prefix_lens, int32_t *status, void *stream);

/*
 * spec_tree_expand — one level of draft token-tree construction.
 *
 * Source: SpecInfer developer article §2.1 (the speculator proposes, from
 * each node's draft distribution, the candidate tokens of the next level of
 * the token tree; each node keeps its parent pointer) and its deployment
 * configuration (tree width).
 *
 * For frontier row f (node node_ids[f] of request requests[f]; draft logits
 * draft_logits[f][V]; cumulative score parent_scores[f]):
 *   temperature > 0: q = softmax(draft / temperature); child j < width is the
 *     inverse-CDF draw of q at the Philox4x64-10 uniform of counter
 *     (node, request, 2, j), key (seed, 0) (the uniform convention of
 *     spec_tree_verify);
 *   temperature == 0: q = softmax(draft); the children are the width most
 *     likely tokens in order, ties to the lower index.
 * child_scores[f][j] = parent_scores[f] + log q(child_tokens[f][j]);
 * near_ties[f][j] = 1 when a draw lay within 1e-6 of an inverse-CDF boundary,
 *   -1 when an exchange between the CTAs that share row f timed out (the
 *   row's outputs are then unreliable; not expected in normal operation).
 *   width <= 16.  All arrays are device memory.  A row is split over
 *   ceil(V / 8192) CTAs (at most 8) of one thread-block cluster.
 */
int spec_tree_expand(const float *draft_logits, const float *parent_scores,
                     const int32_t *node_ids, const int32_t *requests, int F, int V, int width,
                     float temperature, uint64_t seed, int32_t *child_tokens, float *child_scores,
                     int32_t *near_ties, void *stream);

/*
 * spec_tree_prune — pruning of a candidate token tree to its best subtree.
 *
 * Source: SpecInfer developer article §2.1 (the token tree organises the
 * speculated candidates; parent pointers).  For request b with candidates
 * [cand_offsets[b], cand_offsets[b+1]) (request-local parents, parent < index,
 * root first) keep the root and the keep - 1 other candidates of highest
 * score, ties to the lower index.  Scores never increase along a path (each
 * adds a log-probability <= 0), so the kept set is closed under ancestors.
 * Scores from elsewhere must keep that property.  When a kept candidate's
 * parent is not kept, its out_parent is -1: the output is then no tree, and
 * spec_build_tree_mask rejects it with SPEC_ERR_BAD_PARENT.
 * Outputs at stride `keep`, kept candidates in their original order:
 *   out_parents [B][keep] renumbered parents (-2 past n_out[b])
 *   out_tokens  [B][keep], kept_index [B][keep] (candidate index, -1 past n_out)
 *   n_out       [B] = min(keep, candidate count)
 *   keep <= SPEC_MAX_TREE_NODES; at most 1024 candidates per request.
 * Errors on the device: SPEC_ERR_TREE_TOO_LARGE (no candidate, or more than
 * 1024), SPEC_ERR_BAD_PARENT.
 */
int spec_tree_prune(const int32_t *parents, const int32_t *tokens, const float *scores,
                    const int32_t *cand_offsets, int B, int keep, int32_t *out_parents,
                    int32_t *out_tokens, int32_t *kept_index, int32_t *n_out, int32_t *status,
                    void *stream);

/*
 * spec_tree_merge — merging two speculators' token trees into one tree.
 *
 * Source: SpecInfer developer article, §7.2 混合推测策略 (mixed speculation:
 * an LLM speculator's token tree merged with an n-gram speculator's,
 * tree.merge(other), to widen coverage); the merged tree is then verified
 * in one pass like any token tree.
 *
 * For request b, trees A (nodes [offsets_a[b], offsets_a[b+1])) and B share
 * the root (the last committed token; root tokens are ignored).  The merged
 * tree keeps A's nodes at indices 0 .. n_a - 1 unchanged; every node of B
 * whose token path from the root is already present maps to the present
 * node of lowest merged index, and the others are appended in B's order
 * (so parent < index holds).  Outputs per request at stride
 * SPEC_MAX_TREE_NODES:
 *   out_parents [B][128]  merged parents (-2 past n_out[b])
 *   out_tokens  [B][128]  merged tokens (-1 past n_out[b])
 *   map_b       [B][128]  merged index of B's node i (-1 past n_b), e.g. to
 *                         gather a speculator's draft rows for the merged tree
 *   n_out       [B]
 *   Ta, Tb: total nodes of A and of B (offsets_a[B], offsets_b[B]).
 * Errors on the device (outputs untouched): SPEC_ERR_TREE_TOO_LARGE (a tree
 * with no node or more than SPEC_MAX_TREE_NODES, or a merged tree larger
 * than that), SPEC_ERR_BAD_PARENT.
 */
int spec_tree_merge(const int32_t *parents_a, const int32_t *tokens_a, const int32_t *offsets_a,
                    const int32_t *parents_b, const int32_t *tokens_b, const int32_t *offsets_b,
                    int B, int Ta, int Tb, int32_t *out_parents, int32_t *out_tokens,
                    int32_t *map_b, int32_t *n_out, int32_t *status, void *stream);

/*
 * spec_tree_verify_static — spec_tree_verify without a caller workspace.
 *
 * No counterpart in the paper: this is a library convenience.  It serves
 * callers that cannot allocate device memory, such as a plugin inside an
 * inference engine that owns all device memory and passes the library only
 * a step's inputs and outputs, or a binding from a runtime without a CUDA
 * allocator.  The scratch spec_tree_verify takes as `workspace` lives
 * instead in a fixed array of SPEC_VERIFY_STATIC_SCRATCH_BYTES inside the
 * library, held on every GPU that loads the library until the process exits.
 *
 * Arguments, outputs and device-side errors are those of spec_tree_verify.
 * The call allocates nothing and frees nothing; once every host-side check
 * has passed it clears the part of the array it uses (an asynchronous memset
 * on `stream`) and then runs the same kernels as spec_tree_verify.  A call
 * that fails a host-side check enqueues nothing.
 *  - Returns SPEC_ERR_WORKSPACE, before touching the device, when
 *    spec_tree_verify_workspace_size(B, T, V) exceeds
 *    SPEC_VERIFY_STATIC_SCRATCH_BYTES (for example more than about 32000
 *    tree nodes in one batch); use spec_tree_verify with a workspace then.
 *  - The first call made with a device current looks up the array's device
 *    address on that device (cudaGetSymbolAddress), and so does the first
 *    call after that device's context was destroyed and created again (a
 *    device reset).  Make such a call before any stream capture.
 *  - Every call on a device shares the one array, and it keeps the last
 *    call's contents: calls whose work overlaps on the GPU (different
 *    streams, or different host threads) race and give wrong results.
 *    Serialise them, for example on one stream.
 */
#define SPEC_VERIFY_STATIC_SCRATCH_BYTES (256u * 1024u)

int spec_tree_verify_static(const float *target_logits, const float *draft_logits,
                            const int32_t *tokens, const int32_t *parents,
                            const int32_t *tree_offsets, int B, int T, int V, float temperature,
                            uint64_t seed, int32_t *accept_len, int32_t *path_nodes,
                            int32_t *out_tokens, int32_t *near_ties, int max_depth_plus1,
                            int32_t *status, void *stream);

/*
 * spec_test_verify_timeout — a test of verification's failure path, for the
 * test-suite; no counterpart in the pages.
 *
 * Runs spec_tree_verify (stochastic, V <= 131072: the register-resident
 * kernel) with every bounded device wait limited to wait_ns nanoseconds
 * (0 < wait_ns <= 2 s) instead of the normal 2 s, and with one CTA of every
 * node of request drop_request withholding its share of the first
 * statistics exchange.  Nothing else completes those waits, so they run out:
 * the kernel returns, status[drop_request] becomes SPEC_ERR_TIMEOUT, that
 * request's outputs are left as they were (its walk is not run), and every
 * other request is verified exactly as by spec_tree_verify.  The workspace
 * is left reusable.  Arguments are those of spec_tree_verify plus the two
 * above; SPEC_ERR_SHAPE for greedy, wider vocabularies, or out-of-range
 * wait_ns / drop_request.
 */
int spec_test_verify_timeout(const float *target_logits, const float *draft_logits,
                             const int32_t *tokens, const int32_t *parents,
                             const int32_t *tree_offsets, int B, int T, int V, float temperature,
                             uint64_t seed, int32_t *accept_len, int32_t *path_nodes,
                             int32_t *out_tokens, int32_t *near_ties, int max_depth_plus1,
                             void *workspace, size_t workspace_bytes, int32_t *status,
                             void *stream, uint64_t wait_ns, int drop_request);

/*
 * spec_philox_uniforms — step R on its own: the uniform the kernels draw for
 * each of n counters.
 *
 * Source: the counter-based generator the method's stochastic decisions use
 * (a generator shared with any independent check of the decisions).
 * Philox4x64-10 (Salmon et al., SC'11) with key (seed, 0); for counter
 * (c0, c1, c2, c3): u = (first output word >> 40) * 2^-24, exact in float.
 * spec_tree_verify draws with counters (node, request, 0, 0) for the accept
 * test of child `node` and (node, request, 1, 0) for the draw at `node`;
 * spec_tree_expand with (node, request, 2, j) for child slot j.
 *
 *   counters [n][4] int64 (each word taken as its uint64 bit pattern), device
 *   u        [n] float out, device
 * n == 0 launches nothing.
 */
int spec_philox_uniforms(uint64_t seed, const int64_t *counters, int n, float *u, void *stream);

/* Human-readable name of a spec_status value (static storage). */
const char *spec_status_string(int code);

/* 1 in the bounds-checked build (-DSPEC_CHECKED), 0 otherwise. */
int spec_build_checked(void);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_TREE_H */
