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

/* The uniforms of n counters (c0, c1, c2, c3) [n][4], key (seed, 0), the
 * same conversion: for checking a device implementation of the generator. */
void oracle_uniforms(uint64_t seed, const uint64_t *ctr, int64_t n, double *u) {
  const uint64_t key[2] = {seed, 0};
  for (int64_t i = 0; i < n; ++i) {
    uint64_t out[4];
    oracle_philox4x64_10(ctr + 4 * i, key, out);
    u[i] = (double)(out[0] >> 40) * (1.0 / 16777216.0);
  }
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

/* Two decisions the walk takes are compared against a threshold: the accept
 * test (uniform against alpha) and the inverse-CDF draw (u * total against
 * the running sums).  A decision whose distance from its threshold is below
 * TIE_BAND is a near-tie: a float32 implementation may take it the other
 * way, so it is counted ([expl] §2.2 fixes the rule, not its rounding). */
#define TIE_BAND 1e-6

/* Inverse-CDF draw from unnormalised weights w[V] >= 0 with uniform u:
 * the first x whose running sum (ascending x) exceeds u * sum(w); if rounding
 * never lets the running sum pass it, the last x with w[x] > 0.  *gap is the
 * distance of u * sum(w) from the nearer end of the chosen interval, relative
 * to sum(w) (infinite for an all-zero w). */
static int sample_inverse_cdf(const double *w, int V, double u, double *gap) {
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
  *gap = total > 0.0 ? fmin(fabs(target - prev), fabs(target - run)) / total : INFINITY;
  return pick;
}

/* target_logits, draft_logits: [T][V] fp32 (draft may be NULL when
 * temperature == 0).  tokens[T]: the token each node proposes (the root's is
 * ignored).  Outputs per request b (W = max_depth_plus1 entries per row):
 *   accept_len[b]          number of speculated tokens accepted
 *   path_nodes[b][0..a]    request-local node ids: root, then accepted nodes
 *   out_tokens[b][0..a]    tokens of the accepted nodes, then the bonus token
 *   near_ties[b]           decisions on the walk within TIE_BAND of flipping
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

/* What happens at one node if the walk reaches it. */
typedef struct {
  int next;       /* the accepted child (request-local index), or -1: stop at the node */
  int token;      /* the emitted token when next == -1 */
  int ties;       /* decisions within TIE_BAND of flipping */
  double margin;  /* the smallest distance of any decision from its threshold */
  int n_close;    /* decisions within the caller's band (and, for top-p, decisions
                     that involve an entry near the nucleus threshold; see below) */
} node_outcome;

static void note_decision(node_outcome *o, double dist, double band) {
  if (dist < TIE_BAND) ++o->ties;
  if (dist < band) ++o->n_close;
  if (dist < o->margin) o->margin = dist;
}

/* The stochastic decisions at node u of request b for target p and draft qd
 * (r: V entries of scratch for the running residual): u's children in
 * ascending index order, each against r, then, when every child is
 * rejected, the inverse-CDF draw from r.  Distances: |uniform - alpha| for a
 * test, the draw's relative gap for the draw. */
static node_outcome node_decide(const double *p, const double *qd, double *r, int V,
                                const int32_t *par, const int32_t *tok, int n, int u, int b,
                                uint64_t seed, double band) {
  node_outcome o = {-1, -1, 0, INFINITY, 0};
  memcpy(r, p, sizeof(double) * (size_t)V);
  for (int c = u + 1; c < n; ++c) {
    if (par[c] != u) continue;
    int x = tok[c];
    double alpha = qd[x] > 0.0 ? fmin(1.0, r[x] / qd[x]) : 1.0;
    double uu = oracle_uniform(seed, c, b, 0);
    note_decision(&o, fabs(uu - alpha), band);
    if (uu < alpha) { o.next = c; return o; }
    /* rejected: residual r <- norm(max(0, r - q)); a zero residual
     * (r == q up to rounding) leaves r unchanged */
    double s = 0.0;
    for (int y = 0; y < V; ++y) s += fmax(0.0, r[y] - qd[y]);
    if (s > 0.0)
      for (int y = 0; y < V; ++y) r[y] = fmax(0.0, r[y] - qd[y]) / s;
  }
  double gap;
  o.token = sample_inverse_cdf(r, V, oracle_uniform(seed, u, b, 1), &gap);
  note_decision(&o, gap, band);
  return o;
}

/* ---- top-p (developer article, deployment configuration: top_p) -------
 * The nucleus of a distribution d[V]: tau is the largest value whose upper
 * tail {d >= tau} holds at least top_p of the mass (the smallest value when
 * rounding leaves every tail below it); every entry of that tail is kept
 * (entries tied at tau included), the rest drop to 0, and the tail is
 * renormalised.
 *
 * Which nucleus a float32 implementation finds can differ from the exact one
 * in two ways, and each has one band:
 *  - mass: a cut {d >= t} whose tail mass lies within NUCLEUS_MASS_BAND of
 *    top_p on the right side (tail >= top_p - band, mass above t < top_p +
 *    band) may be the one it finds;
 *  - value: entries within NUCLEUS_VALUE_BAND * tau of tau (2^-16 relative,
 *    128 float32 ulps at the bottom of a binade) may sit on either side of
 *    tau in float32, so any subset of their distinct values may be kept.
 * The plausible nuclei are the exact one, the mass-band cuts and the
 * value-band subsets; a node is fragile when two plausible pairs (p's
 * nucleus, q's nucleus) lead to different decisions there. */
#define NUCLEUS_MASS_BAND 5e-6
#define NUCLEUS_VALUE_BAND (1.0 / 65536.0)
#define NUCLEUS_MAX_CUTS 16
#define NUCLEUS_MAX_NEAR 4
#define NUCLEUS_MAX_ALT (1 + NUCLEUS_MAX_CUTS + (1 << NUCLEUS_MAX_NEAR))

static int cmp_desc(const void *a, const void *b) {
  const double x = *(const double *)a, y = *(const double *)b;
  return (x < y) - (x > y);
}

/* d's values sorted in descending order into sorted[V]; returns tau. */
static double nucleus_tau(const double *d, int V, double top_p, double *sorted) {
  memcpy(sorted, d, sizeof(double) * (size_t)V);
  qsort(sorted, (size_t)V, sizeof(double), cmp_desc);
  double above = 0.0;
  for (int i = 0; i < V;) {
    const double t = sorted[i];
    double group = 0.0;
    int k = i;
    while (k < V && sorted[k] == t) group += sorted[k++];
    if (above + group >= top_p) return t;
    above += group;
    i = k;
  }
  return sorted[V - 1];
}

/* The plausible nuclei of d as keep-flags keeps[a][V] (a = 0: the exact
 * nucleus).  Returns their number, or -1 when there are more cuts or
 * near-tau values than this enumeration takes (the node is then fragile).
 * *tau_out receives the exact tau. */
static int nucleus_alternatives(const double *d, int V, double top_p, double *sorted,
                                unsigned char *keeps, double *tau_out) {
  const double tau = nucleus_tau(d, V, top_p, sorted);
  *tau_out = tau;
  int n = 0;
  for (int x = 0; x < V; ++x) keeps[x] = d[x] >= tau;
  ++n;
  /* mass band: cuts at the other distinct values t (sorted[] descending) */
  double above = 0.0;
  for (int i = 0; i < V;) {
    const double t = sorted[i];
    double group = 0.0;
    int k = i;
    while (k < V && sorted[k] == t) group += sorted[k++];
    if (t != tau && above + group >= top_p - NUCLEUS_MASS_BAND &&
        above < top_p + NUCLEUS_MASS_BAND) {
      if (n == 1 + NUCLEUS_MAX_CUTS) return -1;
      unsigned char *kp = keeps + (size_t)n * V;
      for (int x = 0; x < V; ++x) kp[x] = d[x] >= t;
      ++n;
    }
    if (above >= top_p + NUCLEUS_MASS_BAND) break;
    above += group;
    i = k;
  }
  /* value band: the distinct values within NUCLEUS_VALUE_BAND * tau of tau */
  const double lo = tau * (1.0 - NUCLEUS_VALUE_BAND), hi = tau * (1.0 + NUCLEUS_VALUE_BAND);
  double near[NUCLEUS_MAX_NEAR];
  int nn = 0;
  for (int i = 0; i < V; ++i) {
    const double t = sorted[i];
    if (t < lo || t > hi || (nn > 0 && near[nn - 1] == t)) continue;
    if (nn == NUCLEUS_MAX_NEAR) return -1;
    near[nn++] = t;
  }
  if (nn > 1) {
    for (int s = 0; s < (1 << nn); ++s) {
      unsigned char *kp = keeps + (size_t)n * V;
      for (int x = 0; x < V; ++x) {
        int keep = d[x] > hi;
        for (int j = 0; j < nn; ++j)
          if (((s >> j) & 1) && d[x] == near[j]) keep = 1;
        kp[x] = (unsigned char)keep;
      }
      ++n;
    }
  }
  return n;
}

/* out = d restricted to keep[], renormalised */
static void nucleus_apply(const double *d, int V, const unsigned char *keep, double *out) {
  double mass = 0.0;
  for (int v = 0; v < V; ++v)
    if (keep[v]) mass += d[v];
  for (int v = 0; v < V; ++v) out[v] = keep[v] ? d[v] / mass : 0.0;
}

/* Scratch for node_eval: softmax rows, residual, top-p rows and nuclei. */
typedef struct {
  double *p, *qd, *r, *fp, *fq, *vp, *vq, *sorted;
  unsigned char *keeps_p, *keeps_q;
} verify_scratch;

static void scratch_free(verify_scratch *s) {
  free(s->p); free(s->qd); free(s->r); free(s->fp); free(s->fq); free(s->vp); free(s->vq);
  free(s->sorted); free(s->keeps_p); free(s->keeps_q);
}

static int scratch_alloc(verify_scratch *s, int V) {
  const size_t vb = sizeof(double) * (size_t)V;
  const size_t kb = (size_t)NUCLEUS_MAX_ALT * (size_t)V;
  s->p = (double *)malloc(vb); s->qd = (double *)malloc(vb); s->r = (double *)malloc(vb);
  s->fp = (double *)malloc(vb); s->fq = (double *)malloc(vb);
  s->vp = (double *)malloc(vb); s->vq = (double *)malloc(vb); s->sorted = (double *)malloc(vb);
  s->keeps_p = (unsigned char *)malloc(kb); s->keeps_q = (unsigned char *)malloc(kb);
  if (!s->p || !s->qd || !s->r || !s->fp || !s->fq || !s->vp || !s->vq || !s->sorted ||
      !s->keeps_p || !s->keeps_q) {
    scratch_free(s);
    return 0;
  }
  return 1;
}

/* An entry within twice the value band of tau, at a node where d has a value
 * other than tau that close: a float32 implementation that decides
 * membership by the entry's own float value may see the two in either order,
 * so a decision that involves the entry is close. */
static int near_tau(const double *d, int V, double tau, int x) {
  const double w = 2.0 * NUCLEUS_VALUE_BAND * tau;
  if (fabs(d[x] - tau) > w) return 0;
  for (int y = 0; y < V; ++y)
    if (d[y] != tau && fabs(d[y] - tau) <= w) return 1;
  return 0;
}

/* The decisions at node u (request-local) of request b: greedy, stochastic,
 * or stochastic on the top_p nuclei (top_p < 1). */
static node_outcome node_eval(const float *lrow, const float *drow, int V, int greedy,
                              double temp, double top_p, const int32_t *par, const int32_t *tok,
                              int n, int u, int b, uint64_t seed, double band,
                              verify_scratch *s) {
  if (greedy) {
    node_outcome o = {-1, argmax_f(lrow, V), 0, INFINITY, 0};
    for (int c = u + 1; c < n; ++c)
      if (par[c] == u && tok[c] == o.token) { o.next = c; break; }
    return o;
  }
  softmax_t(lrow, V, temp, s->p);
  softmax_t(drow, V, temp, s->qd);
  if (!(top_p < 1.0)) return node_decide(s->p, s->qd, s->r, V, par, tok, n, u, b, seed, band);

  int has_child = 0;
  for (int c = u + 1; c < n; ++c) has_child |= par[c] == u;
  double tau_p = 0.0, tau_q = 0.0;
  const int np = nucleus_alternatives(s->p, V, top_p, s->sorted, s->keeps_p, &tau_p);
  int nq = 1;
  if (has_child) {
    nq = nucleus_alternatives(s->qd, V, top_p, s->sorted, s->keeps_q, &tau_q);
  } else {
    memset(s->keeps_q, 1, (size_t)V);   /* a leaf never reads q */
  }
  nucleus_apply(s->p, V, s->keeps_p, s->fp);
  nucleus_apply(s->qd, V, s->keeps_q, s->fq);
  node_outcome o = node_decide(s->fp, s->fq, s->r, V, par, tok, n, u, b, seed, band);

  /* fragile: too many plausible nuclei to compare, or two that decide differently */
  int fragile = np < 0 || nq < 0 || np * nq > 256;
  for (int i = 0; i < np && !fragile; ++i)
    for (int j = 0; j < nq && !fragile; ++j) {
      if (i == 0 && j == 0) continue;
      nucleus_apply(s->p, V, s->keeps_p + (size_t)i * V, s->vp);
      nucleus_apply(s->qd, V, s->keeps_q + (size_t)j * V, s->vq);
      const node_outcome alt = node_decide(s->vp, s->vq, s->r, V, par, tok, n, u, b, seed, band);
      fragile = alt.next != o.next || (alt.next < 0 && alt.token != o.token);
    }
  if (fragile) {
    ++o.ties;
    ++o.n_close;
    o.margin = 0.0;
  }
  /* decisions that involve an entry near tau (tested children, the drawn token) */
  for (int c = u + 1; c < n; ++c) {
    if (par[c] != u) continue;
    const int x = tok[c];
    o.n_close += near_tau(s->p, V, tau_p, x) || (has_child && near_tau(s->qd, V, tau_q, x));
    if (c == o.next) break;
  }
  if (o.next < 0)
    o.n_close += near_tau(s->p, V, tau_p, o.token) || (has_child && near_tau(s->qd, V, tau_q, o.token));
  return o;
}

/* Validation of request b for verification; *n_out receives its node count. */
static int verify_request_status(const int32_t *tokens, const int32_t *parents,
                                 const int32_t *offsets, int B, int T, int V, int W, int b,
                                 int *n_out) {
  int n = 0;
  int st = check_request(offsets, B, T, b, &n);
  if (st != OR_OK) return st;
  const int32_t *par = parents + offsets[b];
  const int32_t *tok = tokens + offsets[b];
  st = check_parents(par, n);
  if (st != OR_OK) return st;
  for (int i = 1; i < n; ++i)
    if (tok[i] < 0 || tok[i] >= V) return OR_ERR_TOKEN;
  /* the output rows must hold the deepest possible path */
  int maxd = 0;
  for (int i = 0; i < n; ++i) {
    int d = 0;
    for (int a = i; par[a] != -1; a = par[a]) ++d;
    if (d > maxd) maxd = d;
  }
  if (maxd + 1 > W) return OR_ERR_TREE;
  *n_out = n;
  return OR_OK;
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
  const int W = max_depth_plus1;
  verify_scratch s;
  if (!scratch_alloc(&s, V)) return OR_ERR_SHAPE;

  for (int b = 0; b < B; ++b) {
    int n = 0;
    const int st = verify_request_status(tokens, parents, offsets, B, T, V, W, b, &n);
    status[b] = st;
    if (st != OR_OK) continue;
    const int32_t *par = parents + offsets[b];
    const int32_t *tok = tokens + offsets[b];
    int32_t *pn = path_nodes + (size_t)b * W;
    int32_t *ot = out_tokens + (size_t)b * W;
    for (int j = 0; j < W; ++j) pn[j] = ot[j] = -1;
    int ties = 0, acc = 0, u = 0;
    pn[0] = 0;
    for (;;) {
      const size_t row = (size_t)(offsets[b] + u) * V;
      const node_outcome o =
          node_eval(target_logits + row, greedy ? NULL : draft_logits + row, V, greedy,
                    (double)temperature, top_p, par, tok, n, u, b, seed, TIE_BAND, &s);
      ties += o.ties;
      if (o.next < 0) {
        ot[acc] = o.token;
        break;
      }
      ot[acc] = tok[o.next];
      ++acc;
      pn[acc] = o.next;
      u = o.next;
    }
    accept_len[b] = acc;
    near_ties[b] = ties;
  }
  scratch_free(&s);
  return OR_OK;
}

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
 * A visited node that is fragile (see above) counts one near-tie. */
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

/* Per-node decisions, for the parity tests.  Every decision at a node
 * depends only on that node's rows, its children and its own uniforms, not
 * on how the walk reached it, so each node can be evaluated alone.  For every
 * global node t of a valid request with want[t] != 0 (want may be NULL: all
 * nodes): next[t] = the accepted child (request-local) or -1, token[t] = the
 * emitted token when next[t] == -1, margin[t] = the smallest distance of a
 * decision there from its threshold (infinite for greedy; 0 for a fragile
 * top-p node), n_close[t] = its decisions within `band` (top-p: plus those
 * that involve an entry near tau).  Nodes not evaluated get next = -2.
 * status[b] as oracle_tree_verify (max_depth_plus1 = W). */
int oracle_verify_nodes(const float *target_logits, const float *draft_logits,
                        const int32_t *tokens, const int32_t *parents, const int32_t *offsets,
                        int B, int T, int V, float temperature, double top_p, uint64_t seed,
                        int max_depth_plus1, double band, const uint8_t *want, int32_t *next,
                        int32_t *token, double *margin, int32_t *n_close, int32_t *status) {
  if (B < 1 || T < 1 || V < 1 || max_depth_plus1 < 1 || !(top_p > 0.0)) return OR_ERR_SHAPE;
  const int greedy = !(temperature > 0.0f);
  if (!greedy && draft_logits == NULL) return OR_ERR_SHAPE;
  for (int t = 0; t < T; ++t) {
    next[t] = -2;
    token[t] = -1;
    margin[t] = INFINITY;
    n_close[t] = 0;
  }
  verify_scratch s;
  if (!scratch_alloc(&s, V)) return OR_ERR_SHAPE;
  for (int b = 0; b < B; ++b) {
    int n = 0;
    status[b] = verify_request_status(tokens, parents, offsets, B, T, V, max_depth_plus1, b, &n);
    if (status[b] != OR_OK) continue;
    const int32_t *par = parents + offsets[b];
    const int32_t *tok = tokens + offsets[b];
    for (int u = 0; u < n; ++u) {
      const int t = offsets[b] + u;
      if (want && !want[t]) continue;
      const size_t row = (size_t)t * V;
      const node_outcome o =
          node_eval(target_logits + row, greedy ? NULL : draft_logits + row, V, greedy,
                    (double)temperature, top_p, par, tok, n, u, b, seed, band, &s);
      next[t] = o.next;
      token[t] = o.next < 0 ? o.token : -1;
      margin[t] = o.margin;
      n_close[t] = o.n_close;
    }
  }
  scratch_free(&s);
  return OR_OK;
}

/* The plausible top-p nuclei of one distribution, for the tests that pin
 * their enumeration: writes the exact tau and the keep-flags of every
 * plausible nucleus (keeps[NUCLEUS_MAX_ALT][V]); returns their number or -1. */
int oracle_nucleus_alternatives(const double *d, int V, double top_p, unsigned char *keeps,
                                double *tau) {
  double *sorted = (double *)malloc(sizeof(double) * (size_t)V);
  if (!sorted) return -2;
  const int n = nucleus_alternatives(d, V, top_p, sorted, keeps, tau);
  free(sorted);
  return n;
}

int oracle_nucleus_max_alternatives(void) { return NUCLEUS_MAX_ALT; }

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
/* draw lay within 1e-6 of an inverse-CDF boundary; gaps[f][j] (may be NULL)  */
/* is the draw's relative distance from the nearer boundary (infinite for a  */
/* greedy child).                                                            */
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
                       uint64_t seed, int32_t *tokens, double *scores, int32_t *ties,
                       double *gaps) {
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
      int tok;
      double gap = INFINITY;
      if (temperature > 0.0) {
        tok = sample_inverse_cdf(w, V, oracle_uniform4(seed, node_ids[f], reqs[f], 2, j), &gap);
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
      ties[(size_t)f * width + j] = gap < TIE_BAND;
      if (gaps) gaps[(size_t)f * width + j] = gap;
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

/* ------------------------------------------------------------------------ */
/* Merging two speculators' token trees (developer article, §7.2 混合推测策略: */
/* an LLM speculator's tree merged with an n-gram speculator's,             */
/* tree.merge(other)).  Both trees of request b share the root (the last     */
/* committed token; the root tokens are ignored).  The merged tree holds A's  */
/* nodes unchanged (indices 0 .. n_a - 1), then every node of B whose token  */
/* path from the root is not the path of a node already in the merged tree, */
/* in B's index order; a B node whose path is already present maps to the   */
/* present node of lowest merged index.  Outputs per request at stride cap:  */
/* out_parents (-2 past n_out), out_tokens (-1 past n_out), map_b[b][i] =    */
/* the merged index of B's node i (-1 past n_b, stride cap), n_out[b].       */
/* Errors: OR_ERR_TREE (a tree with no node or more than cap nodes, or a      */
/* merged tree larger than cap), OR_ERR_PARENT; outputs untouched then.      */
/* ------------------------------------------------------------------------ */
int oracle_tree_merge(const int32_t *parents_a, const int32_t *tokens_a, const int32_t *off_a,
                      const int32_t *parents_b, const int32_t *tokens_b, const int32_t *off_b,
                      int B, int cap, int32_t *out_parents, int32_t *out_tokens, int32_t *map_b,
                      int32_t *n_out, int32_t *status) {
  if (B < 1 || cap < 1) return OR_ERR_SHAPE;
  int32_t *mp = (int32_t *)malloc(sizeof(int32_t) * (size_t)cap * 2);
  int32_t *mt = (int32_t *)malloc(sizeof(int32_t) * (size_t)cap * 2);
  int32_t *mb = (int32_t *)malloc(sizeof(int32_t) * (size_t)cap);
  if (!mp || !mt || !mb) { free(mp); free(mt); free(mb); return OR_ERR_SHAPE; }
  for (int b = 0; b < B; ++b) {
    const int na = off_a[b + 1] - off_a[b], nb = off_b[b + 1] - off_b[b];
    const int32_t *pa = parents_a + off_a[b], *ta = tokens_a + off_a[b];
    const int32_t *pb = parents_b + off_b[b], *tb = tokens_b + off_b[b];
    int st = OR_OK;
    if (na < 1 || na > cap || nb < 1 || nb > cap) st = OR_ERR_TREE;
    if (st == OR_OK && (check_parents(pa, na) != OR_OK || check_parents(pb, nb) != OR_OK))
      st = OR_ERR_PARENT;
    int n = 0;
    if (st == OR_OK) {
      /* A unchanged */
      for (int j = 0; j < na; ++j) { mp[n] = pa[j]; mt[n] = ta[j]; ++n; }
      mb[0] = 0; /* the roots coincide */
      for (int i = 1; i < nb && st == OR_OK; ++i) {
        const int parent = mb[pb[i]];
        int found = -1;
        for (int j = 1; j < n && found < 0; ++j)
          if (mp[j] == parent && mt[j] == tb[i]) found = j;
        if (found >= 0) {
          mb[i] = found;
        } else if (n == cap) {
          st = OR_ERR_TREE;
        } else {
          mp[n] = parent;
          mt[n] = tb[i];
          mb[i] = n++;
        }
      }
    }
    status[b] = st;
    if (st != OR_OK) continue;
    for (int j = 0; j < cap; ++j) {
      out_parents[(size_t)b * cap + j] = j < n ? mp[j] : -2;
      out_tokens[(size_t)b * cap + j] = j < n ? mt[j] : -1;
      map_b[(size_t)b * cap + j] = j < nb ? mb[j] : -1;
    }
    n_out[b] = n;
  }
  free(mp); free(mt); free(mb);
  return OR_OK;
}
