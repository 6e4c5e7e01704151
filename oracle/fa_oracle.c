/*
 * Oracle for exact attention — TEST INFRASTRUCTURE, NOT PRODUCT CODE.
 *
 * Only the test suite, the smoke check and the benchmark's CPU-baseline /
 * reference arm may load this library.  The CUDA library never calls it and
 * shares no code, header, table or constant with it.
 *
 * Everything is fp64 and follows the reference pages in their own order:
 *
 *   oracle_attention        the plain definition written out
 *                           ("hs-black: FlashAttention 1/2/3", section
 *                           "Shapes": S = QK^T/sqrt(d), P = softmax_rows(S+mask),
 *                           O = PV; LSE = m + log l from the section
 *                           "One row of runnable logic"), with the causal
 *                           visibility rule of "flash attention V2 code walkthrough"
 *                           (Is_causal: bottom-right aligned mask pictures) and
 *                           the GQA head mapping kv_head = h / (hq/hkv).
 *   oracle_attention_tiled  the online-softmax recurrence of the section
 *                           "Online softmax: merge while reading" / "One row of
 *                           runnable logic" (carry m, l, o; alpha = exp(m-m');
 *                           alpha = 0 on the first block with a valid key; skip
 *                           fully masked blocks; divide at the end), applied tile
 *                           by tile and optionally per KV split, whose partial
 *                           results are then merged by oracle_combine.  Used only
 *                           to check the direct oracle against the method.
 *   oracle_combine          the split-KV merge of "ai-reference-codex: forward
 *                           CUDA kernel", section 7.3: logsumexp of the partial
 *                           LSEs over the split axis, then weights
 *                           e^(LSE_s - LSE_total); a split with no contribution
 *                           carries LSE = -inf.
 *   oracle_num_splits       section 7.2 of the same page: the smallest split
 *                           count whose occupancy is at least 85% of the best.
 *   oracle_attention_bwd    the recompute-based backward pass of "hs-black",
 *                           sections "Backward: ..." (dV = P^T dO, dP = dO V^T,
 *                           D = rowsum(dO * O), dS = P (dP - D), dQ = dS K * scale,
 *                           dK = dS^T Q * scale), written out row by row.
 *
 * Softcap follows the same page's template flag Is_softcap ("a nonlinear
 * transform of the attention scores: tanh softly limits the logits, when
 * softcap > 0"); the page gives no formula, and the reading used here is the
 * plainest one: each scaled score s becomes c * tanh(s / c) (c = softcap), which
 * keeps small scores and bounds every score to (-c, c); masking, the maximum and
 * the softmax then act on the capped scores.  In the backward pass the chain rule
 * adds the factor dc*tanh(s/c)/ds = 1 - tanh^2(s/c) to dS.  c = 0 turns it off.
 *
 * Sliding-window (local) attention follows "flash attention V2 code walkthrough",
 * template flag Is_local: query i sees keys in [i + skv - sq - window_left,
 * i + skv - sq + window_right], written here with the general query offset off
 * in place of skv - sq; a negative window width leaves that side unbounded.
 *
 * Conventions for what the pages leave open (each is listed in the design notes):
 *   - a query row i sees key j iff j < skv and (not causal or j <= i + off)
 *     and, with a window, i + off - window_left <= j <= i + off + window_right;
 *   - a row that sees no key gets O = 0 and LSE = -inf;
 *   - the scale multiplies the raw dot product before mask and max; LSE is in
 *     natural-log units of the scaled scores;
 *   - split partials are normalised (O_s = o_s / l_s) with LSE_s = m_s + log l_s.
 *
 * Mutations (test only): the `mutation` bit mask plants the mistakes the
 * "hs-black" page's lab asks a reader to predict, so that tests can show that
 * the pins catch them.  0 = the correct oracle.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_MUT_NO_ALPHA_ON_O 1   /* tiled: old numerator not rescaled by alpha   */
#define ORACLE_MUT_NO_SCALE 2        /* both: 1/sqrt(d) (the scale) dropped          */
#define ORACLE_MUT_STRICT_CAUSAL 4   /* both: causal j <= i + off replaced by j < ... */
#define ORACLE_MUT_NO_ALPHA_ON_L 8   /* tiled: old denominator not rescaled by alpha */
#define ORACLE_MUT_CAP_BEFORE_SCALE 128  /* softcap applied to the raw dot product, then scaled */
#define ORACLE_MUT_CAP_NO_DERIV 256      /* backward: the softcap factor 1 - tanh^2 dropped */

int oracle_version(void) { return 4; }

/* The score of one (query, key) pair: the scaled dot product, capped when c > 0. */
static double capped(double dotv, double sc, double c, int mutation) {
  if (c <= 0.0) return sc * dotv;
  if (mutation & ORACLE_MUT_CAP_BEFORE_SCALE) return sc * (c * tanh(dotv / c));
  return c * tanh(sc * dotv / c);
}

/* Visibility of key j to query row i; wl / wr < 0: that side of the window is unbounded. */
int oracle_visible_window(int64_t i, int64_t j, int64_t skv, int causal, int64_t off, int64_t wl, int64_t wr,
                          int mutation) {
  if (j < 0 || j >= skv) return 0;
  if (wl >= 0 && j < i + off - wl) return 0;
  if (wr >= 0 && j > i + off + wr) return 0;
  if (!causal) return 1;
  if (mutation & ORACLE_MUT_STRICT_CAUSAL) return j < i + off;
  return j <= i + off;
}

int oracle_visible(int64_t i, int64_t j, int64_t skv, int causal, int64_t off, int mutation) {
  return oracle_visible_window(i, j, skv, causal, off, -1, -1, mutation);
}

static double dot(const double* a, const double* b, int64_t d) {
  double s = 0.0;
  for (int64_t t = 0; t < d; ++t) s += a[t] * b[t];
  return s;
}

/*
 * Direct definition for a list of query rows.
 *   q: [b][sq][hq][d], k, v: [b][skv][hkv][d], contiguous fp64.
 *   rows: nrows triples (batch, q_head, query index).
 *   o: [nrows][d], lse: [nrows].
 * Returns 0 on success, -1 on bad arguments.
 */
int oracle_attention_ex(const double* q, const double* k, const double* v, int64_t b, int64_t sq, int64_t skv,
                        int64_t hq, int64_t hkv, int64_t d, int causal, int64_t off, int64_t wl, int64_t wr,
                        double scale, double softcap, const int64_t* rows, int64_t nrows, double* o, double* lse,
                        int mutation) {
  if (hkv <= 0 || hq % hkv != 0 || d <= 0) return -1;
  const int64_t g = hq / hkv;
  const double sc = (mutation & ORACLE_MUT_NO_SCALE) ? 1.0 : scale;
  int bad = 0;
#pragma omp parallel
  {
    double* s = (double*)malloc(sizeof(double) * (size_t)(skv > 0 ? skv : 1));
    if (!s) {
#pragma omp atomic write
      bad = 1;
    }
#pragma omp for schedule(dynamic, 4)
    for (int64_t r = 0; r < nrows; ++r) {
      if (!s) continue;
      const int64_t bi = rows[3 * r], hi = rows[3 * r + 1], i = rows[3 * r + 2];
      double* orow = o + r * d;
      if (bi < 0 || bi >= b || hi < 0 || hi >= hq || i < 0 || i >= sq) {
#pragma omp atomic write
        bad = 1;
        continue;
      }
      const int64_t kvh = hi / g;
      const double* qrow = q + ((bi * sq + i) * hq + hi) * d;
      double m = -INFINITY;
      int64_t nvis = 0;
      for (int64_t j = 0; j < skv; ++j) {
        if (!oracle_visible_window(i, j, skv, causal, off, wl, wr, mutation)) continue;
        s[j] = capped(dot(qrow, k + ((bi * skv + j) * hkv + kvh) * d, d), sc, softcap, mutation);
        if (s[j] > m) m = s[j];
        ++nvis;
      }
      for (int64_t t = 0; t < d; ++t) orow[t] = 0.0;
      if (nvis == 0) {
        lse[r] = -INFINITY;
        continue;
      }
      double l = 0.0;
      for (int64_t j = 0; j < skv; ++j) {
        if (!oracle_visible_window(i, j, skv, causal, off, wl, wr, mutation)) continue;
        const double p = exp(s[j] - m);
        const double* vrow = v + ((bi * skv + j) * hkv + kvh) * d;
        l += p;
        for (int64_t t = 0; t < d; ++t) orow[t] += p * vrow[t];
      }
      for (int64_t t = 0; t < d; ++t) orow[t] /= l;
      lse[r] = m + log(l);
    }
    free(s);
  }
  return bad ? -1 : 0;
}

int oracle_attention_window(const double* q, const double* k, const double* v, int64_t b, int64_t sq, int64_t skv,
                            int64_t hq, int64_t hkv, int64_t d, int causal, int64_t off, int64_t wl, int64_t wr,
                            double scale, const int64_t* rows, int64_t nrows, double* o, double* lse, int mutation) {
  return oracle_attention_ex(q, k, v, b, sq, skv, hq, hkv, d, causal, off, wl, wr, scale, 0.0, rows, nrows, o, lse,
                             mutation);
}

int oracle_attention(const double* q, const double* k, const double* v, int64_t b, int64_t sq, int64_t skv,
                     int64_t hq, int64_t hkv, int64_t d, int causal, int64_t off, double scale,
                     const int64_t* rows, int64_t nrows, double* o, double* lse, int mutation) {
  return oracle_attention_ex(q, k, v, b, sq, skv, hq, hkv, d, causal, off, -1, -1, scale, 0.0, rows, nrows, o, lse,
                             mutation);
}

/*
 * Split-KV merge for nrows rows of width d.
 *   o_part: [ns][nrows][d] (normalised partial outputs), lse_part: [ns][nrows].
 *   o: [nrows][d], lse: [nrows].
 */
void oracle_combine(const double* o_part, const double* lse_part, int64_t ns, int64_t nrows, int64_t d,
                    double* o, double* lse) {
  for (int64_t r = 0; r < nrows; ++r) {
    double M = -INFINITY;
    for (int64_t s = 0; s < ns; ++s)
      if (lse_part[s * nrows + r] > M) M = lse_part[s * nrows + r];
    double* orow = o + r * d;
    for (int64_t t = 0; t < d; ++t) orow[t] = 0.0;
    if (M == -INFINITY) {
      lse[r] = -INFINITY;
      continue;
    }
    double sum = 0.0;
    for (int64_t s = 0; s < ns; ++s) sum += exp(lse_part[s * nrows + r] - M);
    const double total = M + log(sum);
    for (int64_t s = 0; s < ns; ++s) {
      const double w = exp(lse_part[s * nrows + r] - total);
      if (w == 0.0) continue;
      const double* op = o_part + (s * nrows + r) * d;
      for (int64_t t = 0; t < d; ++t) orow[t] += w * op[t];
    }
    lse[r] = total;
  }
}

/*
 * The tile-by-tile recurrence for one query row over key tiles
 * [t*tile, min((t+1)*tile, skv)) for t in [t_lo, t_hi).  Writes the normalised
 * output and the LSE of this range (0 / -inf when nothing in it is visible).
 */
static void one_row_tiled(const double* qrow, const double* k, const double* v, int64_t bi, int64_t i,
                          int64_t skv, int64_t hkv, int64_t kvh, int64_t d, int causal, int64_t off, int64_t wl,
                          int64_t wr, double sc, double softcap,
                          int64_t tile, int64_t t_lo, int64_t t_hi, int mutation, double* s, double* p, double* o,
                          double* lse) {
  double m = -INFINITY, l = 0.0;
  for (int64_t t = 0; t < d; ++t) o[t] = 0.0;
  for (int64_t tb = t_lo; tb < t_hi; ++tb) {
    const int64_t j0 = tb * tile;
    const int64_t j1 = (j0 + tile < skv) ? j0 + tile : skv;
    int any = 0;
    double bmax = -INFINITY;
    for (int64_t j = j0; j < j1; ++j) {
      if (oracle_visible_window(i, j, skv, causal, off, wl, wr, mutation)) {
        s[j - j0] = capped(dot(qrow, k + ((bi * skv + j) * hkv + kvh) * d, d), sc, softcap, mutation);
        if (s[j - j0] > bmax) bmax = s[j - j0];
        any = 1;
      } else {
        s[j - j0] = -INFINITY;
      }
    }
    if (!any) continue; /* a fully masked block is skipped */
    const double m2 = (bmax > m) ? bmax : m;
    const double alpha = (l != 0.0) ? exp(m - m2) : 0.0;
    double psum = 0.0;
    for (int64_t j = j0; j < j1; ++j) {
      p[j - j0] = (s[j - j0] == -INFINITY) ? 0.0 : exp(s[j - j0] - m2);
      psum += p[j - j0];
    }
    const double ao = (mutation & ORACLE_MUT_NO_ALPHA_ON_O) ? 1.0 : alpha;
    for (int64_t t = 0; t < d; ++t) o[t] *= ao;
    for (int64_t j = j0; j < j1; ++j) {
      if (p[j - j0] == 0.0) continue;
      const double* vrow = v + ((bi * skv + j) * hkv + kvh) * d;
      for (int64_t t = 0; t < d; ++t) o[t] += p[j - j0] * vrow[t];
    }
    const double al = (mutation & ORACLE_MUT_NO_ALPHA_ON_L) ? 1.0 : alpha;
    l = al * l + psum;
    m = m2;
  }
  if (l == 0.0) {
    for (int64_t t = 0; t < d; ++t) o[t] = 0.0;
    *lse = -INFINITY;
    return;
  }
  for (int64_t t = 0; t < d; ++t) o[t] /= l;
  *lse = m + log(l);
}

/*
 * Tiled model: key tiles of `tile` keys, grouped into `num_splits` contiguous
 * ranges of ceil(nblk / num_splits) tiles each; each range is reduced by the
 * one-row recurrence and the ranges are merged by oracle_combine.  Same layouts
 * as oracle_attention.  If o_part / lse_part are non-NULL they receive the
 * per-split partials, [num_splits][nrows][d] and [num_splits][nrows].
 */
int oracle_attention_tiled(const double* q, const double* k, const double* v, int64_t b, int64_t sq, int64_t skv,
                           int64_t hq, int64_t hkv, int64_t d, int causal, int64_t off, int64_t wl, int64_t wr,
                           double scale, double softcap, const int64_t* rows, int64_t nrows, int64_t tile,
                           int64_t num_splits, double* o, double* lse, double* o_part, double* lse_part,
                           int mutation) {
  if (hkv <= 0 || hq % hkv != 0 || d <= 0 || tile <= 0 || num_splits <= 0) return -1;
  const int64_t g = hq / hkv;
  const double sc = (mutation & ORACLE_MUT_NO_SCALE) ? 1.0 : scale;
  const int64_t nblk = (skv + tile - 1) / tile;
  const int64_t nbps = (nblk + num_splits - 1) / num_splits;
  int own = 0;
  if (o_part == NULL || lse_part == NULL) {
    o_part = (double*)malloc(sizeof(double) * (size_t)(num_splits * nrows * d + 1));
    lse_part = (double*)malloc(sizeof(double) * (size_t)(num_splits * nrows + 1));
    if (!o_part || !lse_part) {
      free(o_part);
      free(lse_part);
      return -1;
    }
    own = 1;
  }
  int bad = 0;
#pragma omp parallel
  {
    double* s = (double*)malloc(sizeof(double) * (size_t)tile);
    double* p = (double*)malloc(sizeof(double) * (size_t)tile);
#pragma omp for schedule(dynamic, 4)
    for (int64_t r = 0; r < nrows; ++r) {
      const int64_t bi = rows[3 * r], hi = rows[3 * r + 1], i = rows[3 * r + 2];
      if (!s || !p || bi < 0 || bi >= b || hi < 0 || hi >= hq || i < 0 || i >= sq) {
#pragma omp atomic write
        bad = 1;
        continue;
      }
      const double* qrow = q + ((bi * sq + i) * hq + hi) * d;
      for (int64_t sp = 0; sp < num_splits; ++sp) {
        int64_t t_lo = sp * nbps, t_hi = (sp + 1) * nbps;
        if (t_hi > nblk) t_hi = nblk;
        if (t_lo > t_hi) t_lo = t_hi;
        one_row_tiled(qrow, k, v, bi, i, skv, hkv, hi / g, d, causal, off, wl, wr, sc, softcap, tile, t_lo, t_hi,
                      mutation, s, p,
                      o_part + (sp * nrows + r) * d, lse_part + sp * nrows + r);
      }
    }
    free(s);
    free(p);
  }
  if (!bad) oracle_combine(o_part, lse_part, num_splits, nrows, d, o, lse);
  if (own) {
    free(o_part);
    free(lse_part);
  }
  return bad ? -1 : 0;
}

/* Occupancy of `units` independent work items cut into `s` splits each, on
 * `slots` concurrent CTA slots: w / ceil(w) with w = units * s / slots. */
double oracle_split_efficiency(int64_t units, int64_t slots, int64_t s) {
  const double w = (double)(units * s) / (double)slots;
  return w / ceil(w);
}

/* The smallest split count whose efficiency reaches 85% of the best one over
 * s in [1, min(max_splits, nblk)]. */
int64_t oracle_num_splits(int64_t units, int64_t slots, int64_t nblk, int64_t max_splits) {
  if (units <= 0 || slots <= 0) return 1;
  int64_t smax = max_splits < nblk ? max_splits : nblk;
  if (smax < 1) smax = 1;
  double best = 0.0;
  for (int64_t s = 1; s <= smax; ++s) {
    const double e = oracle_split_efficiency(units, slots, s);
    if (e > best) best = e;
  }
  for (int64_t s = 1; s <= smax; ++s)
    if (oracle_split_efficiency(units, slots, s) >= 0.85 * best) return s;
  return 1;
}

/*
 * Backward pass, recompute form ("hs-black: FlashAttention 1/2/3", sections
 * "Backward: from the softmax derivative", "Training: recompute in backward" and
 * "Backward: back to Q, K, V").  For every row the scores are recomputed, the
 * probabilities recovered as P = exp(S - L) with L = m + log l, and
 *   D_i   = sum_t dO_it O_it              (one scalar per row)
 *   dP_ij = dO_i . V_j
 *   dS_ij = P_ij (dP_ij - D_i)            (zero where the mask hides j)
 *   dV_j += P_ij dO_i
 *   dQ_i += scale dS_ij K_j
 *   dK_j += scale dS_ij Q_i
 * with the same visibility rule as the forward pass; the query heads that share
 * a key/value head add their contributions to its dK / dV.
 *   q, dout: [b][sq][hq][d]; k, v: [b][skv][hkv][d]; outputs dq like q, dk / dv like k.
 * With softcap c > 0 the scores are capped as in the forward pass and dS gains the
 * factor 1 - tanh^2(s / c) (the derivative of the cap), read off the capped score.
 * Mutations (test only): 16 drops D, 32 drops the scale from dQ / dK, 64 uses P
 * in place of dS for dK, 256 drops the softcap factor.  Returns 0, or -1 on bad
 * arguments / allocation failure.
 */
#define ORACLE_MUT_BWD_NO_D 16
#define ORACLE_MUT_BWD_NO_SCALE 32
#define ORACLE_MUT_BWD_DK_FROM_P 64

int oracle_attention_bwd(const double* q, const double* k, const double* v, const double* dout, int64_t b,
                         int64_t sq, int64_t skv, int64_t hq, int64_t hkv, int64_t d, int causal, int64_t off,
                         int64_t wl, int64_t wr, double scale, double softcap, double* dq, double* dk, double* dv,
                         int mutation) {
  if (hkv <= 0 || hq % hkv != 0 || d <= 0 || b < 0 || sq < 0 || skv < 0) return -1;
  const int64_t g = hq / hkv;
  const double gscale = (mutation & ORACLE_MUT_BWD_NO_SCALE) ? 1.0 : scale;
  memset(dq, 0, sizeof(double) * (size_t)(b * sq * hq * d));
  memset(dk, 0, sizeof(double) * (size_t)(b * skv * hkv * d));
  memset(dv, 0, sizeof(double) * (size_t)(b * skv * hkv * d));
  int bad = 0;
  /* one (batch, key/value head) per task: its dK / dV rows are written by no other task */
#pragma omp parallel
  {
    double* s = (double*)malloc(sizeof(double) * (size_t)(skv > 0 ? skv : 1));
    double* o = (double*)malloc(sizeof(double) * (size_t)d);
    if (!s || !o) {
#pragma omp atomic write
      bad = 1;
    }
#pragma omp for schedule(dynamic, 1)
    for (int64_t task = 0; task < b * hkv; ++task) {
      if (!s || !o) continue;
      const int64_t bi = task / hkv, kvh = task % hkv;
      for (int64_t hi = kvh * g; hi < (kvh + 1) * g; ++hi) {
        for (int64_t i = 0; i < sq; ++i) {
          const double* qrow = q + ((bi * sq + i) * hq + hi) * d;
          const double* dorow = dout + ((bi * sq + i) * hq + hi) * d;
          double* dqrow = dq + ((bi * sq + i) * hq + hi) * d;
          /* forward recomputed: scores, L = m + log l, O */
          double m = -INFINITY;
          int64_t nvis = 0;
          for (int64_t j = 0; j < skv; ++j) {
            if (!oracle_visible_window(i, j, skv, causal, off, wl, wr, 0)) continue;
            s[j] = capped(dot(qrow, k + ((bi * skv + j) * hkv + kvh) * d, d), scale, softcap, 0);
            if (s[j] > m) m = s[j];
            ++nvis;
          }
          if (nvis == 0) continue; /* no key: O = 0 and every gradient term is zero */
          double l = 0.0;
          for (int64_t j = 0; j < skv; ++j)
            if (oracle_visible_window(i, j, skv, causal, off, wl, wr, 0)) l += exp(s[j] - m);
          const double L = m + log(l);
          for (int64_t t = 0; t < d; ++t) o[t] = 0.0;
          for (int64_t j = 0; j < skv; ++j) {
            if (!oracle_visible_window(i, j, skv, causal, off, wl, wr, 0)) continue;
            const double p = exp(s[j] - L);
            const double* vrow = v + ((bi * skv + j) * hkv + kvh) * d;
            for (int64_t t = 0; t < d; ++t) o[t] += p * vrow[t];
          }
          const double D = (mutation & ORACLE_MUT_BWD_NO_D) ? 0.0 : dot(dorow, o, d);
          for (int64_t j = 0; j < skv; ++j) {
            if (!oracle_visible_window(i, j, skv, causal, off, wl, wr, 0)) continue;
            const double p = exp(s[j] - L);
            const double* krow = k + ((bi * skv + j) * hkv + kvh) * d;
            const double* vrow = v + ((bi * skv + j) * hkv + kvh) * d;
            double* dkrow = dk + ((bi * skv + j) * hkv + kvh) * d;
            double* dvrow = dv + ((bi * skv + j) * hkv + kvh) * d;
            const double dp = dot(dorow, vrow, d);
            double ds = p * (dp - D);
            if (softcap > 0.0 && !(mutation & ORACLE_MUT_CAP_NO_DERIV)) {
              const double t = s[j] / softcap; /* tanh of the scaled score over c */
              ds *= 1.0 - t * t;
            }
            const double dk_coef = (mutation & ORACLE_MUT_BWD_DK_FROM_P) ? p : ds;
            for (int64_t t = 0; t < d; ++t) {
              dvrow[t] += p * dorow[t];
              dqrow[t] += gscale * ds * krow[t];
              dkrow[t] += gscale * dk_coef * qrow[t];
            }
          }
        }
      }
    }
    free(s);
    free(o);
  }
  return bad ? -1 : 0;
}
