/*
 * sv_oracle.c -- plain, slow, fp64 CPU oracle for the speculative-sampling
 * verification step (chain and token-tree variants).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the package smoke check and the
 * benchmark's CPU-baseline leg load this library.  It shares no source with
 * the CUDA library: no header, helper, table or constant is common to both.
 *
 * Sources (web pages, cited by title and section):
 *   [L17]  CMU 15-779 Lecture 17 notes, "LLM Serving (II): Speculative
 *          Decoding" -- sec. 2.2 (greedy verification), 2.3 (speculative
 *          sampling and its proof), 2.4 (Algorithm 1), 4.4 (VerifyGreedy on
 *          a token tree), 4.5 (multi-step speculative sampling, MSS).
 *   [S14]  "Speculative decoding" tutorial (llminference, s14), section
 *          "The idea / the solution": verify(draft_tokens, q, p, rng).
 *   [N02]  "LLM speculative decoding study notes 02: original speculative
 *          decoding, draft model and rejection sampling" -- sec. 3
 *          (notation: r_i ~ U[0,1]), 4 (complete algorithm), 5.1 (Lemma 1:
 *          residual mass), 5.4 (same decoding strategy, incl. temperature
 *          and top-k, for p and q), 10 (greedy special case), 11.3
 *          (deterministic per-request random numbers).
 *   [DVP]  "Speculative decoding: draft, verify and payoff", part II.2
 *          (algorithm and the distribution identity; KV rollback index).
 *
 * Every floating-point quantity is computed in fp64 with plain loops in the
 * order the definitions state.  Readings where the pages are silent:
 *   - accept test is  u * q(x) < p(x)  (strict; [S14] uses "<", [N02] sec. 4
 *     prints "<="; the two differ only on a measure-zero set of u);
 *   - the residual / bonus token is drawn by inverse CDF over ascending token
 *     id with one extra uniform per request: smallest t with
 *     u*S < sum_{x<=t} w(x); if rounding leaves no such t, the largest t
 *     with w(t) > 0;
 *   - argmax ties go to the lowest token id; top-k keeps exactly k entries,
 *     ties at the k-th value going to the lower token id; temperature is
 *     applied before top-k; p and q are filtered independently;
 *   - a residual of zero mass (only possible through rounding) falls back
 *     to the distribution it was formed from (p_i for a chain, r for a tree);
 *   - greedy requests (temperature 0) use only the target rows.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* oracle status codes (per request) */
#define SVO_OK 0
#define SVO_ENONFINITE 1 /* NaN or +inf logit in a row that is used */
#define SVO_ETOKEN 2     /* token id outside [0, V) */
#define SVO_EMASS 3      /* a distribution with zero total mass */
#define SVO_ETREE 4      /* malformed tree (parent, q_row, depth) */
#define SVO_EARG 5       /* bad scalar argument (temperature < 0 ...) */

/* ---------------------------------------------------------------- logits */

/* A bf16 value is the upper 16 bits of the fp32 value with the same bits. */
static double bf16_bits_to_double(uint16_t h) {
  uint32_t u = ((uint32_t)h) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* dtype 0: bf16 stored as uint16 bit patterns; dtype 1: fp32. */
static double logit_at(const void* rows, int dtype, int64_t idx) {
  if (dtype == 0) return bf16_bits_to_double(((const uint16_t*)rows)[idx]);
  return (double)((const float*)rows)[idx];
}

/* ------------------------------------------------- one row -> a distribution */

int svo_row_argmax(const void* row, int dtype, int V);

static int cmp_desc(const void* a, const void* b) {
  double x = *(const double*)a, y = *(const double*)b;
  return (x < y) - (x > y);
}

/*
 * Mark the k entries of y that come first in the order (value descending,
 * token id ascending).  k <= 0 or k >= V keeps everything.
 */
static void topk_keep(const double* y, int V, int k, unsigned char* keep) {
  if (V <= 0) return;
  if (k <= 0 || k >= V) {
    for (int j = 0; j < V; ++j) keep[j] = 1;
    return;
  }
  double* s = (double*)malloc(sizeof(double) * (size_t)V);
  memcpy(s, y, sizeof(double) * (size_t)V);
  qsort(s, (size_t)V, sizeof(double), cmp_desc);
  double thr = s[k - 1];
  free(s);
  int greater = 0;
  for (int j = 0; j < V; ++j) greater += (y[j] > thr);
  int ties_left = k - greater;
  for (int j = 0; j < V; ++j) {
    if (y[j] > thr) keep[j] = 1;
    else if (y[j] == thr && ties_left > 0) { keep[j] = 1; --ties_left; }
    else keep[j] = 0;
  }
}

/*
 * p = decoding distribution of one logit row ([N02] sec. 5.4: temperature,
 * top-k, the same for p and q).
 *   T == 0 : one-hot at argmax l (lowest id on ties)  ([L17] sec. 2.2).
 *   T  > 0 : y = l / T; keep the top-k of y; p = exp(y - max) / sum.
 * Returns an oracle status code.
 */
int svo_row_probs(const void* row, int dtype, int V, double T, int top_k,
                  double* p) {
  if (V <= 0 || !(T >= 0.0)) return SVO_EARG;
  for (int j = 0; j < V; ++j) {
    double l = logit_at(row, dtype, j);
    if (isnan(l) || l == INFINITY) return SVO_ENONFINITE;
  }
  if (T == 0.0) {
    int a = svo_row_argmax(row, dtype, V);
    if (a == -2) return SVO_EMASS;
    for (int j = 0; j < V; ++j) p[j] = (j == a) ? 1.0 : 0.0;
    return SVO_OK;
  }
  double* y = (double*)malloc(sizeof(double) * (size_t)V);
  unsigned char* keep = (unsigned char*)malloc((size_t)V);
  for (int j = 0; j < V; ++j) y[j] = logit_at(row, dtype, j) / T;
  topk_keep(y, V, top_k, keep);
  double m = -INFINITY;
  for (int j = 0; j < V; ++j)
    if (keep[j] && y[j] > m) m = y[j];
  int rc = SVO_OK;
  if (m == -INFINITY) {
    rc = SVO_EMASS;
  } else {
    double z = 0.0;
    for (int j = 0; j < V; ++j) {
      p[j] = keep[j] ? exp(y[j] - m) : 0.0;
      z += p[j];
    }
    for (int j = 0; j < V; ++j) p[j] /= z;
  }
  free(y);
  free(keep);
  return rc;
}

/*
 * argmax of a row, lowest id on ties.  Returns -1 if the row holds a NaN or
 * +inf, -2 if every entry is -inf (no mass).
 */
int svo_row_argmax(const void* row, int dtype, int V) {
  int a = -2;
  double best = -INFINITY;
  for (int j = 0; j < V; ++j) {
    double l = logit_at(row, dtype, j);
    if (isnan(l) || l == INFINITY) return -1;
    if (l > best) { best = l; a = j; }
  }
  return a;
}

/* ------------------------------------------------------- residual and ICDF */

/*
 * w = max(0, p - q) elementwise; returns S = sum w.  By [N02] sec. 5.1
 * (Lemma 1), S = 1 - sum min(p, q) = TV(p, q) when p and q are normalised.
 */
double svo_residual(const double* p, const double* q, int V, double* w) {
  double s = 0.0;
  for (int t = 0; t < V; ++t) {
    double d = p[t] - q[t];
    w[t] = d > 0.0 ? d : 0.0;
    s += w[t];
  }
  return s;
}

/*
 * Inverse-CDF draw from the unnormalised weights w (total S, computed here in
 * ascending id order): the smallest t with u*S < C(t), C(t) = sum_{x<=t} w(x).
 * If rounding leaves no such t, the largest t with w(t) > 0.
 * *margin = distance of u*S to the nearer of the two boundaries that enclose
 * it, divided by S (the decision is "near" when this is tiny).
 * Returns -1 when S is not positive.
 */
int svo_icdf(const double* w, int V, double u, double* margin) {
  double S = 0.0;
  for (int t = 0; t < V; ++t) S += w[t];
  if (!(S > 0.0)) {
    if (margin) *margin = 0.0;
    return -1;
  }
  double target = u * S;
  double c_prev = 0.0, c = 0.0;
  for (int t = 0; t < V; ++t) {
    c_prev = c;
    c += w[t];
    if (target < c) {
      if (margin) {
        double a = target - c_prev, b = c - target;
        *margin = (a < b ? a : b) / S;
      }
      return t;
    }
  }
  int last = -1;
  for (int t = 0; t < V; ++t)
    if (w[t] > 0.0) last = t;
  if (margin) *margin = 0.0;
  return last;
}

/*
 * The tokens an inverse-CDF draw can give when its target u*S is known only
 * to within radius*S: every t with w(t) > 0 whose step [C(t-1), C(t)) meets
 * [u*S - radius*S, u*S + radius*S] (C and S summed in ascending id order as
 * in svo_icdf).  *lo and *hi receive the smallest and largest such id; they
 * are equal to the svo_icdf token when no other step is that close.  With
 * radius 0 the range is the svo_icdf token alone.  Returns the number of
 * positive-weight tokens in [*lo, *hi], or -1 (and *lo = *hi = -1) when S is
 * not positive.  The parity tests use it to bound a draw whose uniform lies
 * within the kernel's rounding of a CDF step.
 */
int svo_icdf_window(const double* w, int V, double u, double radius, int* lo, int* hi) {
  double S = 0.0;
  for (int t = 0; t < V; ++t) S += w[t];
  *lo = -1;
  *hi = -1;
  if (!(S > 0.0)) return -1;
  const double a = (u - radius) * S, b = (u + radius) * S;
  double c_prev = 0.0, c = 0.0;
  int count = 0;
  for (int t = 0; t < V; ++t) {
    c_prev = c;
    c += w[t];
    if (!(w[t] > 0.0)) continue;
    if (c > a && c_prev <= b) {
      if (*lo < 0) *lo = t;
      *hi = t;
    }
  }
  /* rounding can leave u*S at or beyond the last step: svo_icdf then takes
     the last positive weight, which the window must hold too */
  if (*lo < 0) {
    for (int t = 0; t < V; ++t)
      if (w[t] > 0.0) *lo = *hi = t;
  }
  for (int t = *lo; t >= 0 && t <= *hi; ++t) count += w[t] > 0.0;
  return count;
}

/* relative distance of an accept test  u*q < p  from its boundary */
static double accept_margin(double u, double q, double p) {
  if (!(q > 0.0)) return INFINITY; /* u*0 < p is decided by p > 0 alone */
  return fabs(u * q - p) / q;
}

/* ------------------------------------------------------------------ chain */

/*
 * Chain verification (Leviathan et al. Algorithm 1 as restated in [L17]
 * sec. 2.4, [N02] sec. 4, [DVP] II.2; greedy case [L17] sec. 2.2,
 * [N02] sec. 10).
 *
 * Layouts (contiguous): target [B][K+1][V], draft [B][K][V], tokens [B][K],
 * num_drafts [B] (NULL: all K), temperature [B], top_k [B] (NULL: none),
 * uniforms [B][K+1] (u[0..K-1] accept tests, u[K] the final draw).
 * Outputs: out_tokens [B][K+1] (-1 padded), out_len [B] = accepted + 1,
 * accept_len [B] = accepted drafts = KV truncation index,
 * p_at / q_at [B][K] = p_i(x_i), q_i(x_i) for every i < num_drafts (NaN
 * elsewhere; q_at is NaN for greedy requests, whose draft rows are unused),
 * margin_accept [B] = smallest relative distance |u q - p| / q of an accept
 * test taken to its boundary, margin_draw [B] = the inverse-CDF margin of the
 * final draw (+inf where the decisions are exact, e.g. greedy), status [B].
 * draw_lo, draw_hi [B] (may be NULL): the emitted token's id, or, when the
 * final draw's margin is below `near`, the id range svo_icdf_window gives
 * for radius `near` on the same weights (-1 for a failed request).
 */
int svo_verify_chain(int B, int K, int V, int dtype, const void* target,
                     const void* draft, const int* tokens,
                     const int* num_drafts, const float* temperature,
                     const int* top_k, const float* uniforms, int* out_tokens,
                     int* out_len, int* accept_len, double* p_at,
                     double* q_at, double* margin_accept, double* margin_draw,
                     int* status, double near, int* draw_lo, int* draw_hi) {
  const size_t es = dtype == 0 ? 2 : 4;
  double* p = (double*)malloc(sizeof(double) * (size_t)V);
  double* q = (double*)malloc(sizeof(double) * (size_t)V);
  double* w = (double*)malloc(sizeof(double) * (size_t)V);
  int* amax = (int*)malloc(sizeof(int) * (size_t)(K + 1));
  int n_err = 0;
  for (int b = 0; b < B; ++b) {
    const char* trow0 = (const char*)target + (size_t)b * (K + 1) * V * es;
    const char* drow0 = (const char*)draft + (size_t)b * K * V * es;
    const int* x = tokens + (size_t)b * K;
    const float* u = uniforms + (size_t)b * (K + 1);
    int nd = num_drafts ? num_drafts[b] : K;
    double T = (double)temperature[b];
    int tk = top_k ? top_k[b] : 0;
    int* out = out_tokens + (size_t)b * (K + 1);
    for (int i = 0; i <= K; ++i) out[i] = -1;
    for (int i = 0; i < K; ++i) {
      p_at[(size_t)b * K + i] = NAN;
      q_at[(size_t)b * K + i] = NAN;
    }
    out_len[b] = 0;
    accept_len[b] = 0;
    margin_accept[b] = INFINITY;
    margin_draw[b] = INFINITY;
    status[b] = SVO_OK;
    if (draw_lo) draw_lo[b] = draw_hi[b] = -1;

    int st = SVO_OK;
    if (nd < 0 || nd > K || !(T >= 0.0)) st = SVO_EARG;
    for (int i = 0; st == SVO_OK && i < nd; ++i)
      if (x[i] < 0 || x[i] >= V) st = SVO_ETOKEN;
    if (st != SVO_OK) { status[b] = st; ++n_err; continue; }

    int n = 0, token = -1;
    if (T == 0.0) {
      /* greedy: accept x_i iff it equals argmax p_i; else emit argmax p_i */
      int* a = amax;
      for (int i = 0; i <= nd && st == SVO_OK; ++i) {
        a[i] = svo_row_argmax(trow0 + (size_t)i * V * es, dtype, V);
        if (a[i] == -1) st = SVO_ENONFINITE;
        else if (a[i] == -2) st = SVO_EMASS;
      }
      if (st != SVO_OK) { status[b] = st; ++n_err; continue; }
      for (int i = 0; i < nd; ++i) p_at[(size_t)b * K + i] = (x[i] == a[i]) ? 1.0 : 0.0;
      while (n < nd && x[n] == a[n]) ++n;
      token = a[n];
    } else {
      /* every row the step reads: target rows 0..nd, draft rows 0..nd-1;
         p_i(x_i), q_i(x_i) are reported for every draft position */
      for (int i = 0; i <= nd && st == SVO_OK; ++i) {
        st = svo_row_probs(trow0 + (size_t)i * V * es, dtype, V, T, tk, p);
        if (st == SVO_OK && i < nd) {
          st = svo_row_probs(drow0 + (size_t)i * V * es, dtype, V, T, tk, q);
          if (st == SVO_OK) {
            p_at[(size_t)b * K + i] = p[x[i]];
            q_at[(size_t)b * K + i] = q[x[i]];
          }
        }
      }
      if (st == SVO_OK) {
        /* left to right; stop at the first rejection */
        while (n < nd) {
          double pi = p_at[(size_t)b * K + n], qi = q_at[(size_t)b * K + n];
          double mg = accept_margin((double)u[n], qi, pi);
          if (mg < margin_accept[b]) margin_accept[b] = mg;
          if ((double)u[n] * qi < pi) ++n;
          else break;
        }
        double mg = INFINITY;
        st = svo_row_probs(trow0 + (size_t)n * V * es, dtype, V, T, tk, p);
        if (st == SVO_OK && n < nd) {
          /* rejected at position n: draw from norm(max(0, p_n - q_n)) */
          st = svo_row_probs(drow0 + (size_t)n * V * es, dtype, V, T, tk, q);
          if (st == SVO_OK) {
            double S = svo_residual(p, q, V, w);
            token = S > 0.0 ? svo_icdf(w, V, (double)u[K], &mg)
                            : svo_icdf(p, V, (double)u[K], &mg);
            if (draw_lo && mg < near)
              svo_icdf_window(S > 0.0 ? w : p, V, (double)u[K], near, &draw_lo[b], &draw_hi[b]);
          }
        } else if (st == SVO_OK) {
          /* all drafts accepted: bonus token from p_{nd+1} */
          token = svo_icdf(p, V, (double)u[K], &mg);
          if (draw_lo && mg < near)
            svo_icdf_window(p, V, (double)u[K], near, &draw_lo[b], &draw_hi[b]);
        }
        margin_draw[b] = mg;
        if (st == SVO_OK && token < 0) st = SVO_EMASS;
      }
      if (st != SVO_OK) { status[b] = st; ++n_err; continue; }
    }
    for (int i = 0; i < n; ++i) out[i] = x[i];
    out[n] = token;
    out_len[b] = n + 1;
    accept_len[b] = n;
    if (draw_lo && !(margin_draw[b] < near)) draw_lo[b] = draw_hi[b] = token;
  }
  free(p);
  free(q);
  free(w);
  free(amax);
  return n_err;
}

/* ------------------------------------------------------------------- tree */

/*
 * Token-tree verification ([L17] sec. 4.3-4.5): VerifyGreedy for T == 0,
 * multi-step speculative sampling (MSS) for T > 0.
 *
 * The tree of request b has num_nodes[b] nodes in depth-first order; node 0
 * is the root (the last verified token; its token id is ignored) and
 * parent[n] < n for n >= 1.  target [B][N][V]: row n is the target
 * distribution after the path root..n.  draft [B][M][V]: row q_row[n] is the
 * draft distribution that proposed node n.  u_accept [B][N] holds the accept
 * uniform of node n, u_sample [B] the final draw.
 *
 * At the current node, children are tried in ascending index order against
 * the residual r (initially p_node):  accept child c iff u_c * q_c(x_c) <
 * r(x_c); on rejection r <- norm(max(0, r - q_c)).  All children rejected:
 * draw from r.  A node without children: draw from p_node (bonus).
 * Greedy: go to the first child whose token is argmax p_node, else emit it.
 *
 * mode selects the stochastic rule (greedy walks are the same in every mode):
 *   SVO_TREE_MSS (0)   as above; the children are assumed drawn i.i.d. from
 *                      their q ([L17] sec. 4.5, the precondition of Thm 4.2).
 *   SVO_TREE_NOREPLACE (1)  multi-step speculative sampling for children
 *                      drawn WITHOUT replacement ([L17] sec. 4.5, the remark
 *                      on the proof's precondition, and sec. 10 exercise 7,
 *                      the unbiased fix): the j-th child tried at a node is
 *                      tested, and the residual formed, with q_j = q with
 *                      the tokens of the siblings tried before it set to 0,
 *                      renormalised (q = the child's own draft row).  A q_j
 *                      of zero mass is all zero (its child is accepted iff
 *                      r(x) > 0, and a rejection leaves r unchanged).
 *   SVO_TREE_NAIVE (2) naive sampling ([L17] sec. 4.5): at the current node
 *                      draw x from p_node by inverse CDF with the node's own
 *                      uniform u_accept[node]; move to the first child whose
 *                      token is x, else emit x.  u_sample is unused, and
 *                      margin_draw is the smallest margin over the draws.
 *
 * Outputs: out_tokens [B][max_depth+1], accepted_nodes [B][max_depth]
 * (-1 padded), out_len, accept_len, margin_accept, margin_draw, status as
 * for the chain.  margin_walk [B] (may be NULL): the smallest margin of the
 * draws that chose a child (naive mode; +inf otherwise), i.e. of the draws
 * that decide the path as the accept tests do in MSS.  draw_lo, draw_hi [B]
 * (may be NULL): as for the chain, for the draw of the emitted token.
 */
#define SVO_TREE_MSS 0
#define SVO_TREE_NOREPLACE 1
#define SVO_TREE_NAIVE 2

int svo_verify_tree(int B, int N, int M, int V, int dtype, int max_depth, int mode,
                    const void* target, const void* draft,
                    const int* node_tokens, const int* parent,
                    const int* q_row, const int* num_nodes,
                    const float* temperature, const int* top_k,
                    const float* u_accept, const float* u_sample,
                    int* out_tokens, int* out_len, int* accept_len,
                    int* accepted_nodes, double* margin_accept,
                    double* margin_draw, int* status, double near,
                    double* margin_walk, int* draw_lo, int* draw_hi) {
  const size_t es = dtype == 0 ? 2 : 4;
  double* p = (double*)malloc(sizeof(double) * (size_t)V);
  double* r = (double*)malloc(sizeof(double) * (size_t)V);
  double* q = (double*)malloc(sizeof(double) * (size_t)V);
  double* w = (double*)malloc(sizeof(double) * (size_t)V);
  int* depth = (int*)malloc(sizeof(int) * (size_t)(N > 0 ? N : 1));
  int* tried = (int*)malloc(sizeof(int) * (size_t)(N > 0 ? N : 1));
  int n_err = 0;
  for (int b = 0; b < B; ++b) {
    const char* trow0 = (const char*)target + (size_t)b * N * V * es;
    const char* drow0 = (const char*)draft + (size_t)b * M * V * es;
    const int* tok = node_tokens + (size_t)b * N;
    const int* par = parent + (size_t)b * N;
    const int* qr = q_row + (size_t)b * N;
    const float* ua = u_accept + (size_t)b * N;
    int nn = num_nodes ? num_nodes[b] : N;
    double T = (double)temperature[b];
    int tk = top_k ? top_k[b] : 0;
    int* out = out_tokens + (size_t)b * (max_depth + 1);
    int* acc = accepted_nodes + (size_t)b * max_depth;
    for (int i = 0; i <= max_depth; ++i) out[i] = -1;
    for (int i = 0; i < max_depth; ++i) acc[i] = -1;
    out_len[b] = 0;
    accept_len[b] = 0;
    margin_accept[b] = INFINITY;
    margin_draw[b] = INFINITY;
    status[b] = SVO_OK;
    if (margin_walk) margin_walk[b] = INFINITY;
    if (draw_lo) draw_lo[b] = draw_hi[b] = -1;
    const double* wfinal = NULL; /* weights of the final draw */
    double ufinal = 0.0, mfinal = INFINITY;

    int st = SVO_OK;
    if (nn < 1 || nn > N || !(T >= 0.0) || mode < 0 || mode > 2) st = SVO_EARG;
    else if (par[0] != -1) st = SVO_ETREE;
    if (st == SVO_OK) depth[0] = 0;
    /* q_row is checked only where the walk reads it (sampled, not naive) */
    const int use_q = T > 0.0 && mode != SVO_TREE_NAIVE;
    for (int n = 1; st == SVO_OK && n < nn; ++n) {
      if (par[n] < 0 || par[n] >= n || (use_q && (qr[n] < 0 || qr[n] >= M))) st = SVO_ETREE;
      else if (tok[n] < 0 || tok[n] >= V) st = SVO_ETOKEN;
      else {
        depth[n] = depth[par[n]] + 1;
        if (depth[n] > max_depth) st = SVO_ETREE;
      }
    }
    if (st != SVO_OK) { status[b] = st; ++n_err; continue; }

    int node = 0, L = 0, token = -1;
    for (;;) {
      st = svo_row_probs(trow0 + (size_t)node * V * es, dtype, V, T, tk, p);
      if (st != SVO_OK) break;
      if (T == 0.0) {
        int a = svo_row_argmax(trow0 + (size_t)node * V * es, dtype, V);
        int next = -1;
        for (int c = node + 1; c < nn; ++c)
          if (par[c] == node && tok[c] == a) { next = c; break; }
        if (next < 0) { token = a; break; }
        out[L] = a;
        acc[L] = next;
        ++L;
        node = next;
        continue;
      }
      if (mode == SVO_TREE_NAIVE) {
        double mgn = INFINITY;
        int x = svo_icdf(p, V, (double)ua[node], &mgn);
        if (mgn < margin_draw[b]) margin_draw[b] = mgn;
        if (x < 0) { token = -1; break; }
        int next = -1;
        for (int c = node + 1; c < nn; ++c)
          if (par[c] == node && tok[c] == x) { next = c; break; }
        if (next < 0) {
          token = x;
          wfinal = p;
          ufinal = (double)ua[node];
          mfinal = mgn;
          break;
        }
        if (margin_walk && mgn < margin_walk[b]) margin_walk[b] = mgn;
        out[L] = x;
        acc[L] = next;
        ++L;
        node = next;
        continue;
      }
      int has_child = 0;
      for (int c = node + 1; c < nn; ++c)
        if (par[c] == node) { has_child = 1; break; }
      double mg = INFINITY;
      if (!has_child) { /* leaf: bonus token from p_node */
        token = svo_icdf(p, V, (double)u_sample[b], &mg);
        margin_draw[b] = mg;
        wfinal = p;
        ufinal = (double)u_sample[b];
        mfinal = mg;
        break;
      }
      memcpy(r, p, sizeof(double) * (size_t)V);
      int next = -1, n_tried = 0;
      for (int c = node + 1; c < nn && st == SVO_OK; ++c) {
        if (par[c] != node) continue;
        st = svo_row_probs(drow0 + (size_t)qr[c] * V * es, dtype, V, T, tk, q);
        if (st != SVO_OK) break;
        if (mode == SVO_TREE_NOREPLACE) {
          /* q_j: the earlier-tried siblings' tokens removed, renormalised */
          for (int j = 0; j < n_tried; ++j) q[tried[j]] = 0.0;
          double sq = 0.0;
          for (int t = 0; t < V; ++t) sq += q[t];
          if (sq > 0.0)
            for (int t = 0; t < V; ++t) q[t] /= sq;
        }
        int xc = tok[c];
        tried[n_tried++] = xc;
        double m1 = accept_margin((double)ua[c], q[xc], r[xc]);
        if (m1 < margin_accept[b]) margin_accept[b] = m1;
        if ((double)ua[c] * q[xc] < r[xc]) { next = c; break; }
        double S = svo_residual(r, q, V, w);
        if (S > 0.0)
          for (int t = 0; t < V; ++t) r[t] = w[t] / S;
      }
      if (st != SVO_OK) break;
      if (next >= 0) {
        out[L] = tok[next];
        acc[L] = next;
        ++L;
        node = next;
        continue;
      }
      token = svo_icdf(r, V, (double)u_sample[b], &mg);
      margin_draw[b] = mg;
      wfinal = r;
      ufinal = (double)u_sample[b];
      mfinal = mg;
      break;
    }
    if (st == SVO_OK && token < 0) st = SVO_EMASS;
    if (st != SVO_OK) {
      for (int i = 0; i <= max_depth; ++i) out[i] = -1;
      for (int i = 0; i < max_depth; ++i) acc[i] = -1;
      status[b] = st;
      ++n_err;
      continue;
    }
    out[L] = token;
    out_len[b] = L + 1;
    accept_len[b] = L;
    if (draw_lo) {
      draw_lo[b] = draw_hi[b] = token;
      if (wfinal && mfinal < near) svo_icdf_window(wfinal, V, ufinal, near, &draw_lo[b], &draw_hi[b]);
    }
  }
  free(p);
  free(r);
  free(q);
  free(w);
  free(depth);
  free(tried);
  return n_err;
}

/* ------------------------------------------------- tree attention mask */

/*
 * Topology-aware causal mask and depth position ids of a depth-first
 * linearised token tree ([L17] sec. 4.3, tree attention: a node attends to
 * the verified prefix, its ancestors and itself; positions are given by
 * depth, so nodes at the same depth share one; sec. 10 exercise 5).
 *
 * Request b has n = num_nodes[b] nodes (num_nodes NULL: N), node 0 the root,
 * parent[0] == -1 and 0 <= parent[i] < i.  mask [B][N][W] (W >= ceil(N/32)
 * 32-bit words per row): bit (j % 32) of word j / 32 of row i is set iff j is
 * i or an ancestor of i.  depth [B][N]: edges from the root.  Rows i >= n and
 * every row of a malformed request are zero with depth -1; a malformed
 * request gets status SVO_ETREE (SVO_EARG for n outside [1, N]).
 */
int svo_tree_mask(int B, int N, int W, const int* parent, const int* num_nodes,
                  uint32_t* mask, int* depth, int* status) {
  int n_err = 0;
  for (int b = 0; b < B; ++b) {
    const int* par = parent + (size_t)b * N;
    uint32_t* mrow = mask + (size_t)b * N * W;
    int* dep = depth + (size_t)b * N;
    int n = num_nodes ? num_nodes[b] : N;
    for (int i = 0; i < N * W; ++i) mrow[i] = 0u;
    for (int i = 0; i < N; ++i) dep[i] = -1;
    int st = SVO_OK;
    if (n < 1 || n > N) st = SVO_EARG;
    else if (par[0] != -1) st = SVO_ETREE;
    for (int i = 1; st == SVO_OK && i < n; ++i)
      if (par[i] < 0 || par[i] >= i) st = SVO_ETREE;
    status[b] = st;
    if (st != SVO_OK) { ++n_err; continue; }
    for (int i = 0; i < n; ++i) {
      int d = -1;
      for (int j = i; j >= 0; j = (j == 0 ? -1 : par[j])) {
        mrow[(size_t)i * W + j / 32] |= 1u << (j % 32);
        ++d;
      }
      dep[i] = d;
    }
  }
  return n_err;
}

/* ------------------------------------------------- per-position statistics */

/*
 * Acceptance statistics of a chain round ([L17] sec. 2.3, Thm 3.5: the
 * acceptance rate of position i is alpha_i = sum_x min(p_i(x), q_i(x)) =
 * 1 - TV(p_i, q_i); [N02] sec. 7: E[N] = (1 - a^(K+1)) / (1 - a) for i.i.d.
 * acceptance; the per-position form sum_{j=0..nd} prod_{i<j} alpha_i, which
 * reduces to it when every alpha_i = a).
 *
 * For request b with nd = num_drafts[b] (NULL: K) and every position
 * i < nd: p_i, q_i = svo_row_probs of target row i and draft row i (greedy:
 * one-hot argmax, so alpha_i is 1 iff the argmaxes agree); alpha [B][K]
 * (NaN at i >= nd); expected [B] = sum_{j=0..nd} prod_{i<j} alpha_i, the
 * expected number of tokens the round emits.  A request with a data error
 * gets NaN everywhere and its status.
 */
int svo_row_stats(int B, int K, int V, int dtype, const void* target, const void* draft,
                  const int* num_drafts, const float* temperature, const int* top_k,
                  double* alpha, double* expected, int* status) {
  const size_t es = dtype == 0 ? 2 : 4;
  double* p = (double*)malloc(sizeof(double) * (size_t)V);
  double* q = (double*)malloc(sizeof(double) * (size_t)V);
  int n_err = 0;
  for (int b = 0; b < B; ++b) {
    int nd = num_drafts ? num_drafts[b] : K;
    double T = (double)temperature[b];
    int tk = top_k ? top_k[b] : 0;
    double* al = alpha + (size_t)b * K;
    for (int i = 0; i < K; ++i) al[i] = NAN;
    expected[b] = NAN;
    int st = SVO_OK;
    if (nd < 0 || nd > K || !(T >= 0.0) || tk < 0) st = SVO_EARG;
    for (int i = 0; st == SVO_OK && i < nd; ++i) {
      st = svo_row_probs((const char*)target + ((size_t)b * (K + 1) + i) * V * es, dtype, V,
                         T, tk, p);
      if (st != SVO_OK) break;
      st = svo_row_probs((const char*)draft + ((size_t)b * K + i) * V * es, dtype, V, T,
                         tk, q);
      if (st != SVO_OK) break;
      double a = 0.0;
      for (int t = 0; t < V; ++t) a += p[t] < q[t] ? p[t] : q[t];
      al[i] = a;
    }
    status[b] = st;
    if (st != SVO_OK) {
      for (int i = 0; i < K; ++i) al[i] = NAN;
      ++n_err;
      continue;
    }
    double e = 0.0, reach = 1.0;
    for (int j = 0; j <= nd; ++j) {
      e += reach;
      if (j < nd) reach *= al[j];
    }
    expected[b] = e;
  }
  free(p);
  free(q);
  return n_err;
}
