/*
 * Plain, slow, single-threaded CPU oracle for token-tree verification.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code, header, table or helper with the
 * CUDA library; the two are compared on the same seeded inputs.
 *
 * Everything is computed in IEEE double.  fp32 and bf16 inputs widen to
 * double exactly, so the oracle sees the same numbers the GPU sees.
 *
 * Sources (pages the method is written from):
 *   [news]  SpecInfer news write-up (sunluscious.com.cn), section
 *           "Token 樹驗證器" (token tree verifier): the speculated tokens form a
 *           tree, verified in one pass with a tree-attention mask and a
 *           depth-first KV-cache update.
 *   [dev]   "SpecInfer：基于树结构的LLM推测性推理加速技术" (bjdmk.com.cn),
 *           §2.1 整体工作流程: node = (distribution, parent pointer, children),
 *           the tree_attention snippet (masked scores, softmax, times V), and
 *           the accept stage (longest verified prefix).
 *   [expl]  speculative-decoding explainer (intelliparadigm.com), §2.2
 *           三阶段工作流程详解: stage 2 (accept probability min(1, p/q)),
 *           stage 3 (left-to-right check, stop at the first rejection and
 *           replace it with a new target prediction; output distribution equal
 *           to the target's).
 *
 * Readings where the pages are silent (each one is listed with its reason in
 * the design notes): node 0 is the root (last committed token) and is not
 * verified; children are tested in ascending index order against a running
 * residual; the bonus token after a fully accepted path is drawn from the
 * leaf's target distribution; temperature divides both target and draft
 * logits; a node sees itself; the softmax scale defaults to 1/sqrt(D).
 *
 * Parity pins: every function here is checked by the CPU test-suite against
 * something other than itself (networkx ancestor sets, torch SDPA, numpy's
 * Philox, closed-form acceptance rates, brute-force path enumeration, a
 * chi-square test of the lossless claim, a hand-worked example).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Status codes.  Same numeric values as the library's public header so the
 * tests can compare them, but defined here independently. */
#define OR_OK 0
#define OR_ERR_SHAPE (-2)
#define OR_ERR_TREE (-4)
#define OR_ERR_PARENT (-5)
#define OR_ERR_TOKEN (-6)
#define OR_ERR_PREFIX (-10)

#define OR_MAX_NODES 128

/* ------------------------------------------------------------------------ */
/* Philox4x64-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As   */
/* Easy as 1, 2, 3", SC'11).  Ten rounds of: two 64x64->128 multiplies, the  */
/* high halves XOR-ed with the other counter words and the round key, a word */
/* permutation; the key is bumped by the Weyl constants between rounds.      */
/* ------------------------------------------------------------------------ */
static void mul_hi_lo_64(uint64_t a, uint64_t b, uint64_t *hi, uint64_t *lo) {
  /* schoolbook 32-bit limbs, no compiler extensions */
  uint64_t a_lo = a & 0xffffffffu, a_hi = a >> 32;
  uint64_t b_lo = b & 0xffffffffu, b_hi = b >> 32;
  uint64_t ll = a_lo * b_lo;
  uint64_t lh = a_lo * b_hi;
  uint64_t hl = a_hi * b_lo;
  uint64_t hh = a_hi * b_hi;
  uint64_t mid = (ll >> 32) + (lh & 0xffffffffu) + (hl & 0xffffffffu);
  *lo = (ll & 0xffffffffu) | (mid << 32);
  *hi = hh + (lh >> 32) + (hl >> 32) + (mid >> 32);
}

void oracle_philox4x64_10(const uint64_t ctr_in[4], const uint64_t key_in[2],
                          uint64_t out[4]) {
  const uint64_t mult0 = 0xD2E7470EE14C6C93ull, mult1 = 0xCA5A826395121157ull;
  const uint64_t weyl0 = 0x9E3779B97F4A7C15ull, weyl1 = 0xBB67AE8584CAA73Bull;
  uint64_t x0 = ctr_in[0], x1 = ctr_in[1], x2 = ctr_in[2], x3 = ctr_in[3];
  uint64_t k0 = key_in[0], k1 = key_in[1];
  for (int round = 0; round < 10; ++round) {
    uint64_t hi0, lo0, hi1, lo1;
    mul_hi_lo_64(mult0, x0, &hi0, &lo0);
    mul_hi_lo_64(mult1, x2, &hi1, &lo1);
    uint64_t y0 = hi1 ^ x1 ^ k0;
    uint64_t y1 = lo1;
    uint64_t y2 = hi0 ^ x3 ^ k1;
    uint64_t y3 = lo0;
    x0 = y0; x1 = y1; x2 = y2; x3 = y3;
    k0 += weyl0;
    k1 += weyl1;
  }
  out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

/* The uniform the method draws for (request, node, kind): counter =
 * (node, request, kind, 0), key = (seed, 0); u = top 24 bits of the first
 * output word times 2^-24, so u is in [0, 1) and exact in float and double.
 * kind 0 = accept test of child `node`; kind 1 = fallback sample at `node`. */
double oracle_uniform(uint64_t seed, int64_t node, int64_t request, int64_t kind) {
  uint64_t ctr[4] = {(uint64_t)node, (uint64_t)request, (uint64_t)kind, 0};
  uint64_t key[2] = {seed, 0};
  uint64_t out[4];
  oracle_philox4x64_10(ctr, key, out);
  return (double)(out[0] >> 40) * (1.0 / 16777216.0);
}

/* ------------------------------------------------------------------------ */
/* Tree validation: parent[0] = -1 and 0 <= parent[i] < i for i > 0 ([dev]  */
/* §2.1: each node keeps a parent pointer; index order is topological).      */
/* ------------------------------------------------------------------------ */
static int check_request(const int32_t *offsets, int B, int T, int b, int *n_out) {
  int32_t lo = offsets[b], hi = offsets[b + 1];
  if (lo < 0 || hi > T || hi <= lo) return OR_ERR_TREE;
  if (hi - lo > OR_MAX_NODES) return OR_ERR_TREE;
  (void)B;
  *n_out = hi - lo;
  return OR_OK;
}

static int check_parents(const int32_t *par, int n) {
  if (par[0] != -1) return OR_ERR_PARENT;
  for (int i = 1; i < n; ++i)
    if (par[i] < 0 || par[i] >= i) return OR_ERR_PARENT;
  return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* Step A1: ancestor-or-self bitmask and depth per node ([news] mask matrix;  */
/* [dev] tree_mask, 0 = masked).  Walk the parent pointers to the root and   */
/* set one bit per node visited.                                             */
/* mask: [T][4] uint32, bit a of node i set iff a is i or an ancestor of i.  */
/* ------------------------------------------------------------------------ */
int oracle_build_mask(const int32_t *parents, const int32_t *offsets, int B, int T,
                      uint32_t *mask, int32_t *depth, int32_t *status) {
  if (B < 1 || T < 1) return OR_ERR_SHAPE;
  for (int b = 0; b < B; ++b) {
    int n = 0;
    int st = check_request(offsets, B, T, b, &n);
    if (st == OR_OK) st = check_parents(parents + offsets[b], n);
    status[b] = st;
    if (st != OR_OK) continue;
    const int32_t *par = parents + offsets[b];
    for (int i = 0; i < n; ++i) {
      uint32_t *m = mask + 4 * (size_t)(offsets[b] + i);
      m[0] = m[1] = m[2] = m[3] = 0;
      int steps = 0;
      for (int a = i; a != -1; a = par[a]) {
        m[a >> 5] |= 1u << (a & 31);
        ++steps;
      }
      depth[offsets[b] + i] = steps - 1;
    }
  }
  return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* Step A2: tree attention, the [dev] §2.1 tree_attention snippet written    */
/* out per (node, query head): scores of the query against the request's     */
/* whole key sequence [prefix slots 0..L-1 | tree slots L..L+N-1], masked    */
/* keys set to -inf, softmax, weighted sum of the values in ascending key    */
/* order.  The tree's K/V sit after the prefix in node order (the [news]     */
/* depth-first KV-cache update).  A key is visible to node i iff it is a     */
/* prefix slot or the slot of i itself or of one of i's ancestors.           */
/*                                                                           */
/* q: [T][Hq][D]; k, v: [B][Hkv][S_cap][D]; o: [nrows][D] in double.         */
/* rows: list of (node * Hq + head) to compute, or NULL for all T*Hq rows.   */
/* Query head h reads KV head h / (Hq / Hkv) (grouped-query attention).      */
/* ------------------------------------------------------------------------ */
int oracle_tree_attn(const float *q, const float *k, const float *v, double *o,
                     int B, int T, int Hq, int Hkv, int D, int S_cap,
                     const int32_t *prefix_lens, const int32_t *offsets,
                     const int32_t *parents, double scale,
                     const int64_t *rows, int64_t nrows) {
  if (B < 1 || T < 1 || Hq < 1 || Hkv < 1 || D < 1 || Hq % Hkv) return OR_ERR_SHAPE;
  const int G = Hq / Hkv;
  if (!(scale > 0.0)) scale = 1.0 / sqrt((double)D);
  if (rows == NULL) nrows = (int64_t)T * Hq;
  double *scores = (double *)malloc(sizeof(double) * (size_t)(S_cap + 1));
  double *acc = (double *)malloc(sizeof(double) * (size_t)D);
  unsigned char *visible = (unsigned char *)malloc((size_t)S_cap + 1);
  if (!scores || !acc || !visible) { free(scores); free(acc); free(visible); return OR_ERR_SHAPE; }
  int rc = OR_OK;
  for (int64_t r = 0; r < nrows; ++r) {
    int64_t row = rows ? rows[r] : r;
    int t = (int)(row / Hq), h = (int)(row % Hq);
    int b = 0;
    while (b < B && !(offsets[b] <= t && t < offsets[b + 1])) ++b;
    if (b == B) { rc = OR_ERR_TREE; break; }
    int n = offsets[b + 1] - offsets[b];
    int i = t - offsets[b];
    int L = prefix_lens[b];
    if (L < 0 || L + n > S_cap) { rc = OR_ERR_PREFIX; break; }
    const int32_t *par = parents + offsets[b];
    if (check_parents(par, n) != OR_OK) { rc = OR_ERR_PARENT; break; }
    int g = h / G;
    const float *qv = q + ((size_t)t * Hq + h) * D;
    const float *kb = k + ((size_t)b * Hkv + g) * (size_t)S_cap * D;
    const float *vb = v + ((size_t)b * Hkv + g) * (size_t)S_cap * D;
    const int nkeys = L + n;
    /* visibility: prefix, then ancestor-or-self slots of node i */
    for (int j = 0; j < nkeys; ++j) visible[j] = (unsigned char)(j < L);
    for (int a = i; a != -1; a = par[a]) visible[L + a] = 1;
    /* masked scores */
    double mx = -INFINITY;
    for (int j = 0; j < nkeys; ++j) {
      if (!visible[j]) { scores[j] = -INFINITY; continue; }
      double dot = 0.0;
      const float *kj = kb + (size_t)j * D;
      for (int d = 0; d < D; ++d) dot += (double)qv[d] * (double)kj[d];
      scores[j] = scale * dot;
      if (scores[j] > mx) mx = scores[j];
    }
    /* softmax by max subtraction */
    double sum = 0.0;
    for (int j = 0; j < nkeys; ++j) {
      scores[j] = exp(scores[j] - mx);
      sum += scores[j];
    }
    for (int d = 0; d < D; ++d) acc[d] = 0.0;
    for (int j = 0; j < nkeys; ++j) {
      double p = scores[j] / sum;
      const float *vj = vb + (size_t)j * D;
      for (int d = 0; d < D; ++d) acc[d] += p * (double)vj[d];
    }
    memcpy(o + (size_t)r * D, acc, sizeof(double) * (size_t)D);
  }
  free(scores); free(acc); free(visible);
  return rc;
}

/* ------------------------------------------------------------------------ */
/* Steps V1-V4: verification, walked root to leaf one request at a time.    */
/* ------------------------------------------------------------------------ */

/* softmax of row / temperature into out[V] (double); returns nothing. */
static void softmax_t(const float *row, int V, double temperature, double *out) {
  double mx = -INFINITY;
  for (int x = 0; x < V; ++x) {
    double z = (double)row[x] / temperature;
    out[x] = z;
    if (z > mx) mx = z;
  }
  double s = 0.0;
  for (int x = 0; x < V; ++x) {
    out[x] = exp(out[x] - mx);
    s += out[x];
  }
  for (int x = 0; x < V; ++x) out[x] /= s;
}

/* argmax with the lowest index winning ties. */
static int argmax_f(const float *row, int V) {
  int best = 0;
  for (int x = 1; x < V; ++x)
    if (row[x] > row[best]) best = x;
  return best;
}

/* Inverse-CDF draw from unnormalised weights w[V] >= 0 with uniform u:
 * the first x whose running sum (ascending x) exceeds u * sum(w); if rounding
 * never lets the running sum pass it, the last x with w[x] > 0.  Sets *tie
 * when u*sum lies within 1e-6*sum of the chosen interval's ends. */
static int sample_inverse_cdf(const double *w, int V, double u, int *tie) {
  double total = 0.0;
  for (int x = 0; x < V; ++x) total += w[x];
  double target = u * total;
  double run = 0.0, prev = 0.0;
  int pick = -1;
  for (int x = 0; x < V; ++x) {
    prev = run;
    run += w[x];
    if (run > target) { pick = x; break; }
  }
  if (pick < 0) {
    for (int x = V - 1; x >= 0; --x)
      if (w[x] > 0.0) { pick = x; break; }
    if (pick < 0) pick = 0;
    prev = run; /* boundary is the end of the cumulative sum */
  }
  if (fabs(target - prev) < 1e-6 * total || fabs(target - run) < 1e-6 * total) *tie = 1;
  return pick;
}

/* target_logits, draft_logits: [T][V] fp32 (draft may be NULL when
 * temperature == 0).  tokens[T]: the token each node proposes (the root's is
 * ignored).  Outputs per request b (W = max_depth_plus1 entries per row):
 *   accept_len[b]          number of speculated tokens accepted
 *   path_nodes[b][0..a]    request-local node ids: root, then accepted nodes
 *   out_tokens[b][0..a]    tokens of the accepted nodes, then the bonus token
 *   near_ties[b]           decisions on the walk within 1e-6 of flipping
 * unused row entries are set to -1.
 *
 * Greedy (temperature == 0): at node u accept the first child whose token is
 * argmax of u's target logits; if none, emit that argmax and stop ([dev]
 * §2.1 accept stage: longest verified prefix; [expl] §2.2 stage 1 drafts
 * greedily).
 *
 * Stochastic: p = softmax(target/T), q = softmax(draft/T) of node u.  With
 * r = p, test u's children c in ascending index order: alpha = min(1,
 * r(x_c)/q(x_c)) ([expl] §2.2 stage 2), accept iff uniform < alpha; on
 * rejection r <- max(0, r - q) renormalised ([expl] §2.2 stage 3: the
 * rejected token is replaced by a new target prediction; the residual keeps
 * the output distribution equal to the target's).  If every child is
 * rejected (or u is a leaf), draw the emitted token from r and stop. */
/* Nucleus (top-p) of a distribution d[V] (developer article, deployment
 * configuration: top_p).  tau is the largest value whose upper tail
 * {d >= tau} holds at least top_p of the mass; every entry of that tail is
 * kept (entries tied at tau included), the rest set to 0, and the tail
 * renormalised.
 *
 * Which nucleus a finite-precision implementation finds can differ from the
 * exact one where the running mass crosses top_p within its rounding: every
 * cut {d >= t} whose tail holds at least top_p - eps while the tail above t
 * holds less than top_p + eps is one it may find.  nucleus_cuts lists those
 * thresholds t (the exact tau first); the walk counts a near-tie at a node
 * only when two of them lead to different decisions there. */
static int cmp_desc(const void *a, const void *b) {
  const double x = *(const double *)a, y = *(const double *)b;
  return (x < y) - (x > y);
}

#define NUCLEUS_EPS 5e-6
#define NUCLEUS_MAX_CUTS 64

/* Returns the number of plausible thresholds written to cuts[] (cuts[0] is
 * the exact tau), or -1 when there are more than NUCLEUS_MAX_CUTS. */
static int nucleus_cuts(const double *d, int V, double top_p, double *sorted, double *cuts) {
  memcpy(sorted, d, sizeof(double) * (size_t)V);
  qsort(sorted, (size_t)V, sizeof(double), cmp_desc);
  /* distinct values in descending order with the tail mass above each */
  double above = 0.0, tau = sorted[V - 1];
  int n = 0, found = 0;
  for (int i = 0; i < V;) {
    const double t = sorted[i];
    double group = 0.0;
    int k = i;
    while (k < V && sorted[k] == t) group += sorted[k++];
    const double ge = above + group;  /* tail {d >= t} */
    if (!found && ge >= top_p) { tau = t; found = 1; }
    i = k;
    above = ge;
  }
  if (!found) tau = sorted[V - 1];
  cuts[n++] = tau;
  above = 0.0;
  for (int i = 0; i < V;) {
    const double t = sorted[i];
    double group = 0.0;
    int k = i;
    while (k < V && sorted[k] == t) group += sorted[k++];
    const double ge = above + group;
    if (t != tau && ge >= top_p - NUCLEUS_EPS && above < top_p + NUCLEUS_EPS) {
      if (n == NUCLEUS_MAX_CUTS) return -1;
      cuts[n++] = t;
    }
    if (above >= top_p + NUCLEUS_EPS) break;
    i = k;
    above = ge;
  }
  return n;
}

/* out = d restricted to {d >= t}, renormalised */
static void nucleus_apply(const double *d, int V, double t, double *out) {
  double mass = 0.0;
  for (int v = 0; v < V; ++v)
    if (d[v] >= t) mass += d[v];
  for (int v = 0; v < V; ++v) out[v] = d[v] >= t ? d[v] / mass : 0.0;
}

/* The stochastic decisions at node u of request b for target p and draft qd:
 * u's children in ascending index order against the residual r (scratch,
 * V entries), then, when every child is rejected, the inverse-CDF draw from
 * r.  Returns the accepted child, or -1 with *token the drawn token;
 * *ties counts decisions within 1e-6 of flipping. */
static int node_decide(const double *p, const double *qd, double *r, int V,
                       const int32_t *par, const int32_t *tok, int n, int u, int b,
                       uint64_t seed, int *token, int *ties) {
  memcpy(r, p, sizeof(double) * (size_t)V);
  for (int c = u + 1; c < n; ++c) {
    if (par[c] != u) continue;
    int x = tok[c];
    double alpha = qd[x] > 0.0 ? fmin(1.0, r[x] / qd[x]) : 1.0;
    double uu = oracle_uniform(seed, c, b, 0);
    if (fabs(uu - alpha) < 1e-6) ++*ties;
    if (uu < alpha) return c;
    /* rejected: residual r <- norm(max(0, r - q)); a zero residual
     * (r == q up to rounding) leaves r unchanged */
    double s = 0.0;
    for (int y = 0; y < V; ++y) s += fmax(0.0, r[y] - qd[y]);
    if (s > 0.0)
      for (int y = 0; y < V; ++y) r[y] = fmax(0.0, r[y] - qd[y]) / s;
  }
  int tie = 0;
  *token = sample_inverse_cdf(r, V, oracle_uniform(seed, u, b, 1), &tie);
  *ties += tie;
  return -1;
}

static int tree_verify_impl(const float *target_logits, const float *draft_logits,
                            const int32_t *tokens, const int32_t *parents,
                            const int32_t *offsets, int B, int T, int V, float temperature,
                            double top_p, uint64_t seed, int32_t *accept_len,
                            int32_t *path_nodes, int32_t *out_tokens, int32_t *near_ties,
                            int max_depth_plus1, int32_t *status);

int oracle_tree_verify(const float *target_logits, const float *draft_logits,
                       const int32_t *tokens, const int32_t *parents,
                       const int32_t *offsets, int B, int T, int V, float temperature,
                       uint64_t seed, int32_t *accept_len, int32_t *path_nodes,
                       int32_t *out_tokens, int32_t *near_ties, int max_depth_plus1,
                       int32_t *status) {
  return tree_verify_impl(target_logits, draft_logits, tokens, parents, offsets, B, T, V,
                          temperature, 1.0, seed, accept_len, path_nodes, out_tokens, near_ties,
                          max_depth_plus1, status);
}

/* The same walk with the target and draft distributions each filtered to
 * their top_p nucleus first (top_p >= 1: no filter; greedy is unaffected).
 * A node whose nucleus boundary is a near-tie counts one near-tie when the
 * walk visits it. */
int oracle_tree_verify_top_p(const float *target_logits, const float *draft_logits,
                             const int32_t *tokens, const int32_t *parents,
                             const int32_t *offsets, int B, int T, int V, float temperature,
                             double top_p, uint64_t seed, int32_t *accept_len,
                             int32_t *path_nodes, int32_t *out_tokens, int32_t *near_ties,
                             int max_depth_plus1, int32_t *status) {
  if (!(top_p > 0.0)) return OR_ERR_SHAPE;
  return tree_verify_impl(target_logits, draft_logits, tokens, parents, offsets, B, T, V,
                          temperature, top_p, seed, accept_len, path_nodes, out_tokens, near_ties,
                          max_depth_plus1, status);
}

static int tree_verify_impl(const float *target_logits, const float *draft_logits,
                            const int32_t *tokens, const int32_t *parents,
                            const int32_t *offsets, int B, int T, int V, float temperature,
                            double top_p, uint64_t seed, int32_t *accept_len,
                            int32_t *path_nodes, int32_t *out_tokens, int32_t *near_ties,
                            int max_depth_plus1, int32_t *status) {
  if (B < 1 || T < 1 || V < 1 || max_depth_plus1 < 1) return OR_ERR_SHAPE;
  const int greedy = !(temperature > 0.0f);
  if (!greedy && draft_logits == NULL) return OR_ERR_SHAPE;
  const double temp = (double)temperature;
  const int W = max_depth_plus1;
  const size_t vb = sizeof(double) * (size_t)V;
  double *p = (double *)malloc(vb), *qd = (double *)malloc(vb), *r = (double *)malloc(vb);
  /* top-p: filtered rows, one alternative pair, sort scratch, thresholds */
  double *fp = (double *)malloc(vb), *fq = (double *)malloc(vb);
  double *vp = (double *)malloc(vb), *vq = (double *)malloc(vb), *sorted = (double *)malloc(vb);
  double cuts_p[NUCLEUS_MAX_CUTS], cuts_q[NUCLEUS_MAX_CUTS];
  if (!p || !qd || !r || !fp || !fq || !vp || !vq || !sorted) {
    free(p); free(qd); free(r); free(fp); free(fq); free(vp); free(vq); free(sorted);
    return OR_ERR_SHAPE;
  }

  for (int b = 0; b < B; ++b) {
    int n = 0;
    int st = check_request(offsets, B, T, b, &n);
    const int32_t *par = parents + (st == OR_OK ? offsets[b] : 0);
    const int32_t *tok = tokens + (st == OR_OK ? offsets[b] : 0);
    if (st == OR_OK) st = check_parents(par, n);
    if (st == OR_OK) {
      for (int i = 1; i < n; ++i)
        if (tok[i] < 0 || tok[i] >= V) st = OR_ERR_TOKEN;
    }
    if (st == OR_OK) {
      /* the output rows must hold the deepest possible path */
      int maxd = 0;
      for (int i = 0; i < n; ++i) {
        int d = 0;
        for (int a = i; par[a] != -1; a = par[a]) ++d;
        if (d > maxd) maxd = d;
      }
      if (maxd + 1 > W) st = OR_ERR_TREE;
    }
    status[b] = st;
    if (st != OR_OK) continue;

    int32_t *pn = path_nodes + (size_t)b * W;
    int32_t *ot = out_tokens + (size_t)b * W;
    for (int j = 0; j < W; ++j) pn[j] = ot[j] = -1;
    int ties = 0, acc = 0;
    int u = 0;
    pn[0] = 0;
    for (;;) {
      const float *lrow = target_logits + (size_t)(offsets[b] + u) * V;
      int next = -1;
      if (greedy) {
        int a = argmax_f(lrow, V);
        for (int c = u + 1; c < n; ++c)
          if (par[c] == u && tok[c] == a) { next = c; break; }
        if (next < 0) { ot[acc] = a; break; }
      } else {
        const float *drow = draft_logits + (size_t)(offsets[b] + u) * V;
        softmax_t(lrow, V, temp, p);
        softmax_t(drow, V, temp, qd);
        int token = -1;
        if (top_p < 1.0) {
          int has_child = 0;
          for (int c = u + 1; c < n; ++c) has_child |= par[c] == u;
          const int np = nucleus_cuts(p, V, top_p, sorted, cuts_p);
          const int nq = has_child ? nucleus_cuts(qd, V, top_p, sorted, cuts_q) : 1;
          if (!has_child) cuts_q[0] = 0.0;   /* a leaf never reads q */
          nucleus_apply(p, V, cuts_p[0], fp);
          if (has_child) nucleus_apply(qd, V, cuts_q[0], fq);
          next = node_decide(fp, fq, r, V, par, tok, n, u, b, seed, &token, &ties);
          if (np < 0 || nq < 0 || np * nq > NUCLEUS_MAX_CUTS * 4) {
            ++ties;   /* too many plausible nuclei to compare */
          } else {
            int differs = 0;
            for (int i = 0; i < np && !differs; ++i)
              for (int j = 0; j < nq && !differs; ++j) {
                if (i == 0 && j == 0) continue;
                int tk = -1, scratch_ties = 0;
                nucleus_apply(p, V, cuts_p[i], vp);
                if (has_child) nucleus_apply(qd, V, cuts_q[j], vq);
                const int nx = node_decide(vp, has_child ? vq : fq, r, V, par, tok, n, u, b, seed,
                                           &tk, &scratch_ties);
                differs = nx != next || (nx < 0 && tk != token);
              }
            ties += differs;
          }
        } else {
          next = node_decide(p, qd, r, V, par, tok, n, u, b, seed, &token, &ties);
        }
        if (next < 0) {
          ot[acc] = token;
          break;
        }
      }
      ot[acc] = tok[next];
      ++acc;
      pn[acc] = next;
      u = next;
    }
    accept_len[b] = acc;
    near_ties[b] = ties;
  }
  free(p); free(qd); free(r); free(fp); free(fq); free(vp); free(vq); free(sorted);
  return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* Depth-first KV-cache update [news]: after verification request b commits  */
/* its root (slot L_b) and the accepted path's nodes, so their keys/values   */
/* must sit contiguously after the prefix for the next step.  Slot L_b + j   */
/* receives the old slot L_b + path[j] for j = 1 .. acc_b (path[0] is the    */
/* root); every other slot is unchanged, and the committed prefix becomes    */
/* L_b + 1 + acc_b.  The copy reads the old cache: a destination slot may    */
/* also be the source of a later path entry (path 0 -> 2 -> 3).              */
/* cache: [B][H][S_cap][D] elements of elem_bytes bytes.  Requests whose     */
/* status is already non-zero are skipped (new prefix = L_b).                */
/* ------------------------------------------------------------------------ */
int oracle_kv_compact(uint8_t *cache, int elem_bytes, int B, int H, int S_cap, int D,
                      const int32_t *prefix_lens, const int32_t *offsets,
                      const int32_t *path_nodes, const int32_t *accept_len, int W,
                      int32_t *new_prefix, int32_t *status) {
  if (B < 1 || H < 1 || S_cap < 1 || D < 1 || W < 1 || elem_bytes < 1) return OR_ERR_SHAPE;
  const size_t row = (size_t)D * (size_t)elem_bytes;
  uint8_t *old = (uint8_t *)malloc(row * (size_t)S_cap);
  if (!old) return OR_ERR_SHAPE;
  for (int b = 0; b < B; ++b) {
    const int L = prefix_lens[b];
    new_prefix[b] = L;
    if (status[b] != 0) continue;
    const int n = offsets[b + 1] - offsets[b];
    const int acc = accept_len[b];
    const int32_t *pn = path_nodes + (size_t)b * W;
    if (L < 0 || L + n > S_cap) { status[b] = OR_ERR_PREFIX; continue; }
    if (acc < 0 || acc + 1 > W) { status[b] = OR_ERR_TREE; continue; }
    int bad = pn[0] != 0;
    for (int j = 1; j <= acc; ++j)
      if (pn[j] <= pn[j - 1] || pn[j] >= n) bad = 1;
    if (bad) { status[b] = OR_ERR_PARENT; continue; }
    for (int h = 0; h < H; ++h) {
      uint8_t *base = cache + (((size_t)b * H + h) * (size_t)S_cap) * row;
      memcpy(old, base, row * (size_t)S_cap);
      for (int j = 1; j <= acc; ++j)
        memcpy(base + (size_t)(L + j) * row, old + (size_t)(L + pn[j]) * row, row);
    }
    new_prefix[b] = L + 1 + acc;
  }
  free(old);
  return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* Draft token-tree construction ([dev] §2.1: the speculator proposes, from  */
/* each node's draft distribution, several candidate tokens that form the    */
/* next level of the token tree, and each node keeps its parent pointer;     */
/* the article's deployment configuration sets the tree width).              */
/*                                                                           */
/* Level expansion, per frontier row f (node u = node_ids[f] of request      */
/* reqs[f], draft logits draft[f][V], cumulative score parent_scores[f]):    */
/*   T > 0:  q = softmax(draft / T); child j (j < width) is the inverse-CDF  */
/*           draw of q at the uniform of counter (u, request, 2, j);          */
/*   T == 0: q = softmax(draft); the children are the `width` most likely    */
/*           tokens in order (ties to the lower index).                      */
/* score of child j = parent score + log q(token).  ties[f][j] = 1 when a    */
/* draw lay within 1e-6 of an inverse-CDF boundary.                          */
/* ------------------------------------------------------------------------ */
static double oracle_uniform4(uint64_t seed, int64_t c0, int64_t c1, int64_t c2, int64_t c3) {
  uint64_t ctr[4] = {(uint64_t)c0, (uint64_t)c1, (uint64_t)c2, (uint64_t)c3};
  uint64_t key[2] = {seed, 0};
  uint64_t out[4];
  oracle_philox4x64_10(ctr, key, out);
  return (double)(out[0] >> 40) * (1.0 / 16777216.0);
}

int oracle_tree_expand(const float *draft, const double *parent_scores, const int32_t *node_ids,
                       const int32_t *reqs, int F, int V, int width, double temperature,
                       uint64_t seed, int32_t *tokens, double *scores, int32_t *ties) {
  if (F < 1 || V < 1 || width < 1 || width > V || !(temperature >= 0.0)) return OR_ERR_SHAPE;
  const double t = temperature > 0.0 ? temperature : 1.0;
  double *w = (double *)malloc(sizeof(double) * (size_t)V);
  if (!w) return OR_ERR_SHAPE;
  for (int f = 0; f < F; ++f) {
    const float *row = draft + (size_t)f * V;
    double m = -INFINITY;
    for (int x = 0; x < V; ++x) m = row[x] > m ? row[x] : m;
    double s = 0.0;
    for (int x = 0; x < V; ++x) {
      w[x] = exp(((double)row[x] - m) / t);
      s += w[x];
    }
    const double log_s = log(s);
    for (int j = 0; j < width; ++j) {
      int tok, tie = 0;
      if (temperature > 0.0) {
        tok = sample_inverse_cdf(w, V, oracle_uniform4(seed, node_ids[f], reqs[f], 2, j), &tie);
      } else {
        /* the j-th most likely token: the best one not yet taken */
        tok = -1;
        for (int x = 0; x < V; ++x) {
          int taken = 0;
          for (int i = 0; i < j; ++i) taken |= tokens[(size_t)f * width + i] == x;
          if (!taken && (tok < 0 || row[x] > row[tok])) tok = x;
        }
      }
      tokens[(size_t)f * width + j] = tok;
      scores[(size_t)f * width + j] = parent_scores[f] + ((double)row[tok] - m) / t - log_s;
      ties[(size_t)f * width + j] = tie;
    }
  }
  free(w);
  return OR_OK;
}

/* Pruning of a candidate tree (request b's candidates at [cand_off[b],    */
/* cand_off[b+1]), request-local parents, breadth-first order so parent <   */
/* index): keep the root and the keep - 1 other candidates of highest score */
/* (ties to the lower index).  A child's score never exceeds its parent's   */
/* (log q <= 0) and ties go to the lower index, so the kept set is closed   */
/* under ancestors.  The kept nodes keep their relative order; outputs per  */
/* request at stride `keep`: parents (renumbered), tokens, the kept          */
/* candidates' indices, and n_out[b] = min(keep, n_b).                      */
int oracle_tree_prune(const int32_t *parents, const int32_t *tokens, const double *scores,
                      const int32_t *cand_off, int B, int keep, int32_t *out_parents,
                      int32_t *out_tokens, int32_t *kept_index, int32_t *n_out, int32_t *status) {
  if (B < 1 || keep < 1) return OR_ERR_SHAPE;
  for (int b = 0; b < B; ++b) {
    const int lo = cand_off[b], n = cand_off[b + 1] - lo;
    n_out[b] = 0;
    for (int i = 0; i < keep; ++i) {
      out_parents[(size_t)b * keep + i] = -2;
      out_tokens[(size_t)b * keep + i] = -1;
      kept_index[(size_t)b * keep + i] = -1;
    }
    if (n < 1) { status[b] = OR_ERR_TREE; continue; }
    if (check_parents(parents + lo, n) != OR_OK) { status[b] = OR_ERR_PARENT; continue; }
    int *keepf = (int *)calloc((size_t)n, sizeof(int));
    int *newid = (int *)malloc(sizeof(int) * (size_t)n);
    if (!keepf || !newid) { free(keepf); free(newid); return OR_ERR_SHAPE; }
    keepf[0] = 1;
    for (int i = 1; i < n; ++i) {
      int better = 0; /* non-root candidates ranked before i */
      for (int j = 1; j < n; ++j)
        if (scores[lo + j] > scores[lo + i] || (scores[lo + j] == scores[lo + i] && j < i)) ++better;
      keepf[i] = better < keep - 1;
    }
    int c = 0;
    for (int i = 0; i < n; ++i) newid[i] = keepf[i] ? c++ : -1;
    for (int i = 0; i < n; ++i) {
      if (!keepf[i]) continue;
      const int k = newid[i];
      out_parents[(size_t)b * keep + k] = i == 0 ? -1 : newid[parents[lo + i]];
      out_tokens[(size_t)b * keep + k] = tokens[lo + i];
      kept_index[(size_t)b * keep + k] = i;
    }
    n_out[b] = c;
    free(keepf);
    free(newid);
  }
  return OR_OK;
}
