/*
 * Jagged generalized dot-product attention: plain CPU oracle (TEST
 * INFRASTRUCTURE ONLY).
 *
 * This file is the checker, not the product. Only the test suite, the
 * package's smoke check and the benchmark's CPU-baseline leg may build, load
 * or call it. It shares no code, header or constant with the CUDA path.
 *
 * What it computes ("GEM Training" engineering post, section "Jagged Sequence
 * Flash Attention" -- attention run directly on unpadded variable-length
 * tensors with asymmetric query/key lengths; section "Generalized Dot-Product
 * Attention (GDPA)" -- two matrix products with an element-wise activation,
 * softmax replaced by GELU or SiLU; section "BlockAttention" -- sliding
 * windows for long self-attention, then fixed blocks where each query block
 * attends only to its own key block):
 *
 *   for every sequence b and head h, rows i < Lq(b), keys j < Lkv(b),
 *   delta = Lkv - Lq (bottom-right alignment):
 *     allowed(i,j): causal  -> j <= i + delta
 *                   window  -> 0 <= i + delta - j < W  (implies causal)
 *                   block   -> floor(j / W) == floor((i + delta) / W)
 *                              (with causal: also j <= i + delta)
 *     s_ij = scale * <q_i, k_j>
 *     softmax:   p_ij = exp(s_ij - m_i) / l_i over allowed j,
 *                o_i = sum_j p_ij v_j,  lse_i = m_i + ln l_i
 *                (no allowed key: o_i = 0, lse_i = -inf)
 *     pointwise: o_i = c * sum_{allowed j} act(s_ij) v_j, c = 1/Lkv or 1
 *                act = SiLU(x) = x / (1 + e^-x)
 *                   or tanh-GELU(x) = x/2 (1 + tanh(sqrt(2/pi)(x + 0.044715 x^3)))
 *   backward (chain rule of the above):
 *     softmax:   D_i = <dO_i, o_i>, dS_ij = p_ij (<dO_i, v_j> - D_i)
 *                (o_i is the forward's output: recomputed here in double, or
 *                the stored output the caller passes in -- FlashAttention's
 *                backward, which JFA's is, reads the output the forward
 *                stored, so its rounding enters D_i and nothing else)
 *     pointwise: dS_ij = c act'(s_ij) <dO_i, v_j>,  p_ij = c act(s_ij)
 *     dV_j = sum_i p_ij dO_i, dQ_i = scale sum_j dS_ij k_j,
 *     dK_j = scale sum_i dS_ij q_i
 *
 * Inputs are double arrays (the Python wrapper decodes bf16 bit patterns to
 * double exactly); all arithmetic is in double. Rows are laid out [total, H, D]; offsets are
 * int64 prefix sums. Only allowed (i, j) pairs are visited, which is exact
 * because masked pairs contribute exactly zero. Parallel over (b, h) with
 * OpenMP; every (b, h) writes disjoint output rows.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_SOFTMAX 0
#define ORACLE_SILU 1
#define ORACLE_GELU 2
/* GELU evaluated by the GPU with a polynomial: the function it stands for
 * is tanh-GELU, which is what the oracle computes for it. */
#define ORACLE_GELU_POLY 3
#define ORACLE_CAUSAL 1
#define ORACLE_WINDOW 2
#define ORACLE_BLOCK 4

/* Block index of position x for blocks of width w (rounds toward -inf). */
static int64_t block_of(int64_t x, int64_t w) { return x >= 0 ? x / w : -((-x + w - 1) / w); }

/* Is key j visible from query i (both sequence-local)? */
static int allowed(int64_t i, int64_t j, int64_t delta, int mask, int64_t window) {
  if ((mask & (ORACLE_CAUSAL | ORACLE_WINDOW)) && j > i + delta) return 0;
  if ((mask & ORACLE_WINDOW) && i + delta - j >= window) return 0;
  if ((mask & ORACLE_BLOCK) && block_of(j, window) != block_of(i + delta, window)) return 0;
  return 1;
}

/* Half-open range of keys that can be visible from row i; every j outside it
 * fails allowed(). Each j inside is still tested with allowed(). */
static void key_range(int64_t i, int64_t delta, int64_t lkv, int mask, int64_t window, int64_t* lo,
                      int64_t* hi) {
  int64_t a = 0, b = lkv;
  if (mask & (ORACLE_CAUSAL | ORACLE_WINDOW)) {
    if (i + delta + 1 < b) b = i + delta + 1;
  }
  if (mask & ORACLE_WINDOW) {
    if (i + delta - window + 1 > a) a = i + delta - window + 1;
  }
  if (mask & ORACLE_BLOCK) {
    const int64_t start = block_of(i + delta, window) * window;
    if (start > a) a = start;
    if (start + window < b) b = start + window;
  }
  if (b < a) b = a;
  *lo = a;
  *hi = b;
}

static double silu(double x) { return x / (1.0 + exp(-x)); }
static double silu_grad(double x) {
  double sg = 1.0 / (1.0 + exp(-x));
  return sg * (1.0 + x * (1.0 - sg));
}
static const double GELU_K = 0.7978845608028654; /* sqrt(2/pi) */
static const double GELU_C = 0.044715;
static double gelu(double x) { return 0.5 * x * (1.0 + tanh(GELU_K * (x + GELU_C * x * x * x))); }
static double gelu_grad(double x) {
  double t = tanh(GELU_K * (x + GELU_C * x * x * x));
  return 0.5 * (1.0 + t) + 0.5 * x * (1.0 - t * t) * GELU_K * (1.0 + 3.0 * GELU_C * x * x);
}
/* act is ORACLE_SILU, ORACLE_GELU or ORACLE_GELU_POLY (the last two both tanh-GELU) */
static double act_fn(int act, double x) { return act == ORACLE_SILU ? silu(x) : gelu(x); }
static double act_grad(int act, double x) { return act == ORACLE_SILU ? silu_grad(x) : gelu_grad(x); }

typedef struct {
  int64_t B;
  int H, D, act, mask;
  int64_t window;
  double scale;
  int norm_by_lkv;
} oracle_params;

/* Copy one (row, head) vector of D values. */
static void load_vec(const double* base, int64_t row, int h, int H, int D, double* out) {
  const double* p = base + ((size_t)row * H + h) * D;
  for (int d = 0; d < D; ++d) out[d] = p[d];
}

static double dot(const double* a, const double* b, int D) {
  double s = 0.0;
  for (int d = 0; d < D; ++d) s += a[d] * b[d];
  return s;
}

/* Scores of row i against its key range, written to s[0 .. hi-lo); returns
 * whether any key is allowed. Also fills vis[] (1 = allowed). */
static int row_scores(const oracle_params* P, const double* qi, const double* kbuf, int64_t i, int64_t delta,
                      int64_t lkv, int64_t lo, int64_t hi, double* s, unsigned char* vis) {
  int any = 0;
  for (int64_t j = lo; j < hi; ++j) {
    vis[j - lo] = (unsigned char)allowed(i, j, delta, P->mask, P->window);
    s[j - lo] = vis[j - lo] ? P->scale * dot(qi, kbuf + (size_t)j * P->D, P->D) : 0.0;
    any |= vis[j - lo];
  }
  (void)lkv;
  return any;
}

/* Probabilities p_ij (softmax) or c*act(s_ij) (pointwise) for one row. */
static void row_probs(const oracle_params* P, int64_t lkv, int64_t n, const double* s, const unsigned char* vis,
                      double* p, double* lse_out) {
  if (P->act == ORACLE_SOFTMAX) {
    double m = -INFINITY;
    for (int64_t t = 0; t < n; ++t)
      if (vis[t] && s[t] > m) m = s[t];
    double l = 0.0;
    for (int64_t t = 0; t < n; ++t) l += vis[t] ? exp(s[t] - m) : 0.0;
    for (int64_t t = 0; t < n; ++t) p[t] = (vis[t] && l > 0.0) ? exp(s[t] - m) / l : 0.0;
    if (lse_out) *lse_out = (l > 0.0) ? m + log(l) : -INFINITY;
  } else {
    double c = (P->norm_by_lkv && lkv > 0) ? 1.0 / (double)lkv : 1.0;
    for (int64_t t = 0; t < n; ++t) p[t] = vis[t] ? c * act_fn(P->act, s[t]) : 0.0;
    if (lse_out) *lse_out = 0.0;
  }
}

static void fill_kv(const double* src, int64_t off, int64_t len, int h, int H, int D, double* dst) {
  for (int64_t j = 0; j < len; ++j) load_vec(src, off + j, h, H, D, dst + (size_t)j * D);
}

/* Forward. o: [total_q, H, D] doubles; lse: [total_q, H] doubles (softmax
 * only; may be NULL). Returns 0. */
int oracle_fwd(const oracle_params* P, const int64_t* q_off, const int64_t* kv_off, const double* q,
               const double* k, const double* v, double* o, double* lse) {
  const int H = P->H, D = P->D;
  const int64_t nbh = P->B * (int64_t)H;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t bh = 0; bh < nbh; ++bh) {
    const int64_t b = bh / H;
    const int h = (int)(bh % H);
    const int64_t lq = q_off[b + 1] - q_off[b], lkv = kv_off[b + 1] - kv_off[b];
    const int64_t delta = lkv - lq;
    double* kb = (double*)malloc(sizeof(double) * (size_t)(lkv > 0 ? lkv : 1) * D);
    double* vb = (double*)malloc(sizeof(double) * (size_t)(lkv > 0 ? lkv : 1) * D);
    double* s = (double*)malloc(sizeof(double) * (size_t)(lkv > 0 ? lkv : 1));
    double* p = (double*)malloc(sizeof(double) * (size_t)(lkv > 0 ? lkv : 1));
    unsigned char* vis = (unsigned char*)malloc((size_t)(lkv > 0 ? lkv : 1));
    double* qi = (double*)malloc(sizeof(double) * D);
    fill_kv(k, kv_off[b], lkv, h, H, D, kb);
    fill_kv(v, kv_off[b], lkv, h, H, D, vb);
    for (int64_t i = 0; i < lq; ++i) {
      int64_t lo, hi;
      key_range(i, delta, lkv, P->mask, P->window, &lo, &hi);
      load_vec(q, q_off[b] + i, h, H, D, qi);
      row_scores(P, qi, kb, i, delta, lkv, lo, hi, s, vis);
      double l_se;
      row_probs(P, lkv, hi - lo, s, vis, p, &l_se);
      double* oi = o + ((size_t)(q_off[b] + i) * H + h) * D;
      for (int d = 0; d < D; ++d) oi[d] = 0.0;
      for (int64_t t = 0; t < hi - lo; ++t) {
        if (!vis[t]) continue;
        const double* vj = vb + (size_t)(lo + t) * D;
        for (int d = 0; d < D; ++d) oi[d] += p[t] * vj[d];
      }
      if (lse) lse[(size_t)(q_off[b] + i) * H + h] = l_se;
    }
    free(kb); free(vb); free(s); free(p); free(vis); free(qi);
  }
  return 0;
}

/* Backward. dq: [total_q,H,D], dk/dv: [total_kv,H,D] doubles, fully written.
 * o_stored: NULL (D_i from the output recomputed here) or the forward output
 * [total_q,H,D] to form D_i from (softmax only; ignored otherwise). */
int oracle_bwd(const oracle_params* P, const int64_t* q_off, const int64_t* kv_off, const double* q,
               const double* k, const double* v, const double* dout, const double* o_stored, double* dq,
               double* dk, double* dv) {
  const int H = P->H, D = P->D;
  const int64_t nbh = P->B * (int64_t)H;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t bh = 0; bh < nbh; ++bh) {
    const int64_t b = bh / H;
    const int h = (int)(bh % H);
    const int64_t lq = q_off[b + 1] - q_off[b], lkv = kv_off[b + 1] - kv_off[b];
    const int64_t delta = lkv - lq;
    const size_t nk = (size_t)(lkv > 0 ? lkv : 1);
    double* kb = (double*)malloc(sizeof(double) * nk * D);
    double* vb = (double*)malloc(sizeof(double) * nk * D);
    double* s = (double*)malloc(sizeof(double) * nk);
    double* p = (double*)malloc(sizeof(double) * nk);
    unsigned char* vis = (unsigned char*)malloc(nk);
    double* qi = (double*)malloc(sizeof(double) * D);
    double* gi = (double*)malloc(sizeof(double) * D);
    double* oi = (double*)malloc(sizeof(double) * D);
    fill_kv(k, kv_off[b], lkv, h, H, D, kb);
    fill_kv(v, kv_off[b], lkv, h, H, D, vb);
    for (int64_t j = 0; j < lkv; ++j) {
      double* a = dk + ((size_t)(kv_off[b] + j) * H + h) * D;
      double* c = dv + ((size_t)(kv_off[b] + j) * H + h) * D;
      for (int d = 0; d < D; ++d) a[d] = c[d] = 0.0;
    }
    for (int64_t i = 0; i < lq; ++i) {
      int64_t lo, hi;
      key_range(i, delta, lkv, P->mask, P->window, &lo, &hi);
      load_vec(q, q_off[b] + i, h, H, D, qi);
      load_vec(dout, q_off[b] + i, h, H, D, gi);
      row_scores(P, qi, kb, i, delta, lkv, lo, hi, s, vis);
      row_probs(P, lkv, hi - lo, s, vis, p, NULL);
      double di = 0.0;
      if (P->act == ORACLE_SOFTMAX) {
        if (o_stored) {
          load_vec(o_stored, q_off[b] + i, h, H, D, oi);
        } else {
          for (int d = 0; d < D; ++d) oi[d] = 0.0;
          for (int64_t t = 0; t < hi - lo; ++t)
            if (vis[t])
              for (int d = 0; d < D; ++d) oi[d] += p[t] * vb[(size_t)(lo + t) * D + d];
        }
        di = dot(gi, oi, D);
      }
      const double c = (P->norm_by_lkv && lkv > 0) ? 1.0 / (double)lkv : 1.0;
      double* dqi = dq + ((size_t)(q_off[b] + i) * H + h) * D;
      for (int d = 0; d < D; ++d) dqi[d] = 0.0;
      for (int64_t t = 0; t < hi - lo; ++t) {
        if (!vis[t]) continue;
        const int64_t j = lo + t;
        const double* kj = kb + (size_t)j * D;
        const double* vj = vb + (size_t)j * D;
        const double dp = dot(gi, vj, D);
        const double ds = (P->act == ORACLE_SOFTMAX) ? p[t] * (dp - di) : c * act_grad(P->act, s[t]) * dp;
        double* dkj = dk + ((size_t)(kv_off[b] + j) * H + h) * D;
        double* dvj = dv + ((size_t)(kv_off[b] + j) * H + h) * D;
        for (int d = 0; d < D; ++d) {
          dvj[d] += p[t] * gi[d];
          dqi[d] += P->scale * ds * kj[d];
          dkj[d] += P->scale * ds * qi[d];
        }
      }
    }
    free(kb); free(vb); free(s); free(p); free(vis); free(qi); free(gi); free(oi);
  }
  return 0;
}

/* Number of allowed (i, j) pairs summed over sequences (one head), counted by
 * visiting every pair of every sequence: O(sum Lq*Lkv). */
int64_t oracle_count_pairs(int64_t B, const int64_t* q_off, const int64_t* kv_off, int mask, int64_t window) {
  int64_t total = 0;
  for (int64_t b = 0; b < B; ++b) {
    const int64_t lq = q_off[b + 1] - q_off[b], lkv = kv_off[b + 1] - kv_off[b];
    for (int64_t i = 0; i < lq; ++i)
      for (int64_t j = 0; j < lkv; ++j) total += allowed(i, j, lkv - lq, mask, window);
  }
  return total;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  extern int omp_get_max_threads(void);
  return omp_get_max_threads();
#else
  return 1;
#endif
}
