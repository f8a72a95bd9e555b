/*
 * Skip-softmax (BLASST) attention oracle: plain fp64 CPU implementation.
 * TEST INFRASTRUCTURE ONLY (see oracle.h): never on the product path.
 *
 * The algorithm is taken in the order the "Skip-Softmax" design doc gives it:
 *   §The online-softmax pass: one streaming pass over key tiles, keeping per
 *     query row the running maximum m, the denominator l = sum exp(s - m) and
 *     the numerator O = sum exp(s - m) v, rescaling l and O when m grows and
 *     returning O / l.
 *   §The skip test: after a tile's scores are known, the tile is skipped when
 *     exp(tile_max - running_max) < threshold; a skipped tile adds nothing to
 *     l or O.  The BLASST summary (§Methodologie) states the same test in log
 *     form: local maximum minus running maximum below ln(lambda).
 *   §What this bounds: the decision is per tile; one important key keeps the
 *     whole tile.  Read here as a unanimous vote of the rows of the query
 *     block (decode: of the query heads sharing the KV head).
 *
 * Readings where the pages leave a step open (each one also listed in the
 * design notes of the repository):
 *   - "running_max" is the maximum over the tiles before this one (for
 *     lambda <= 1 the "after" reading gives the same decisions);
 *   - the comparison is strict: a tie keeps the tile;
 *   - masked scores are -inf, a row with no visible key in a tile does not
 *     veto a skip, and a tile with no visible key for any row is not
 *     evaluated (not counted, state unchanged);
 *   - causal masking is bottom-right aligned (key k visible to row r iff
 *     k <= r + Lk - Lq);
 *   - decode splits are contiguous ranges of ceil(nT/S) tiles, each starting
 *     from an empty state, merged by log-sum-exp.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* bf16 is the upper half of an IEEE binary32; the decode is exact. */
static double bf16_to_double(uint16_t bits) {
  uint32_t w = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &w, sizeof f);
  return (double)f;
}

static double dot_bf16(const uint16_t* a, const uint16_t* b, int d) {
  double s = 0.0;
  for (int e = 0; e < d; ++e) s += bf16_to_double(a[e]) * bf16_to_double(b[e]);
  return s;
}

static int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

/*
 * The per-row running state of the online pass and one tile of it.
 *
 * `rows` query rows (pointers into q, each dk long), keys [k0, k0 + nk) of one
 * head (pointers kh, vh to row 0 of that head; key rows are dk long, value
 * rows d = st->d long).  visible(r, key) is given by `last_visible[r]`: keys
 * with index > last_visible[r] are masked.
 * Returns ORC_KEPT / ORC_SKIPPED / ORC_NOT_EVALUATED and writes c_j.
 */
typedef struct {
  int rows, d; /* d: value width (columns of O) */
  double* m; /* [rows] */
  double* l; /* [rows] */
  double* O; /* [rows][d] */
} run_state;

static void state_reset(run_state* st) {
  for (int r = 0; r < st->rows; ++r) {
    st->m[r] = -INFINITY;
    st->l[r] = 0.0;
  }
  memset(st->O, 0, sizeof(double) * (size_t)st->rows * (size_t)st->d);
}

static int tile_step(run_state* st, const uint16_t* const* qrows, const int64_t* last_visible,
                     const uint16_t* kh, int dk, const uint16_t* vh, int64_t k0, int64_t nk,
                     double scale, double ln_lambda, int have_override, int override_skip,
                     double* s /* scratch [rows][nk] */, double* tmax /* scratch [rows] */,
                     double* c_out) {
  const int d = st->d;
  /* Scores S_j = Q K_j^T * scale, masked keys at -inf, and the row maxima. */
  int any_visible = 0;
  for (int r = 0; r < st->rows; ++r) {
    tmax[r] = -INFINITY;
    for (int64_t t = 0; t < nk; ++t) {
      const int64_t key = k0 + t;
      double x = -INFINITY;
      if (key <= last_visible[r]) x = scale * dot_bf16(qrows[r], kh + (size_t)key * dk, dk);
      s[(size_t)r * nk + t] = x;
      if (x > tmax[r]) tmax[r] = x;
    }
    if (tmax[r] > -INFINITY) any_visible = 1;
  }
  if (!any_visible) {
    *c_out = NAN;
    return ORC_NOT_EVALUATED;
  }
  /* Vote statistic c_j = max over rows of (tile_max - running_max). */
  double c = -INFINITY;
  for (int r = 0; r < st->rows; ++r) {
    if (tmax[r] == -INFINITY) continue; /* no visible key: no veto */
    const double diff = (st->m[r] == -INFINITY) ? INFINITY : tmax[r] - st->m[r];
    if (diff > c) c = diff;
  }
  *c_out = c;
  /* exp(tile_max - running_max) < lambda for every row  <=>  c < ln(lambda). */
  const int skip = have_override ? (override_skip != 0) : (c < ln_lambda);
  if (skip) return ORC_SKIPPED;

  /* Kept tile: fold it into m, l, O with the usual rescaling. */
  for (int r = 0; r < st->rows; ++r) {
    if (tmax[r] == -INFINITY) continue; /* contributes nothing, state unchanged */
    const double m_new = (tmax[r] > st->m[r]) ? tmax[r] : st->m[r];
    const double alpha = (st->m[r] == -INFINITY) ? 0.0 : exp(st->m[r] - m_new);
    double* Or = st->O + (size_t)r * d;
    st->l[r] *= alpha;
    for (int e = 0; e < d; ++e) Or[e] *= alpha;
    for (int64_t t = 0; t < nk; ++t) {
      const double x = s[(size_t)r * nk + t];
      if (x == -INFINITY) continue;
      const double p = exp(x - m_new);
      st->l[r] += p;
      const uint16_t* vk = vh + (size_t)(k0 + t) * d;
      for (int e = 0; e < d; ++e) Or[e] += p * bf16_to_double(vk[e]);
    }
    st->m[r] = m_new;
  }
  return ORC_KEPT;
}

int orc_prefill(const orc_prefill_problem* p, const uint16_t* q, const uint16_t* k,
                const uint16_t* v, const int64_t* units, int64_t n_units,
                const uint8_t* mask_override, double* o, uint8_t* mask, double* margin,
                uint32_t* counts) {
  if (!p || !q || !k || !v) return -1;
  if (p->B < 1 || p->Hq < 1 || p->Hkv < 1 || p->Hq % p->Hkv != 0 || p->Lq < 1 || p->Lk < 1 ||
      p->d < 1 || p->dv < 0 || p->Bq < 1 || p->Bk < 1 || !(p->lambda >= 0.0) || p->lambda > 1.0)
    return -1;
  /* dk: width of q and k rows; d: width of v rows and of O */
  const int G = p->Hq / p->Hkv, dk = p->d, d = (p->dv > 0) ? p->dv : p->d, Bq = p->Bq, Bk = p->Bk;
  const int64_t nQB = ceil_div(p->Lq, Bq), nT = ceil_div(p->Lk, Bk);
  const int64_t total = (int64_t)p->B * p->Hq * nQB;
  if (units == NULL) n_units = total;
  const double ln_lambda = (p->lambda > 0.0) ? log(p->lambda) : -INFINITY;
  const int64_t off = (int64_t)p->Lk - p->Lq;
  int bad = 0;

#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < n_units; ++i) {
    const int64_t u = units ? units[i] : i;
    if (u < 0 || u >= total) {
      bad = 1;
      continue;
    }
    const int64_t qb = u % nQB, bh = u / nQB;
    const int64_t h = bh % p->Hq, b = bh / p->Hq, kvh = h / G;
    const int64_t r0 = qb * Bq;
    const int rows = (int)((r0 + Bq <= p->Lq) ? Bq : p->Lq - r0);

    double* mbuf = malloc(sizeof(double) * (size_t)rows * (3 + (size_t)d + (size_t)Bk));
    int64_t* last_vis = malloc(sizeof(int64_t) * (size_t)rows);
    const uint16_t** qrows = malloc(sizeof(uint16_t*) * (size_t)rows);
    run_state st = {rows, d, mbuf, mbuf + rows, mbuf + 2 * (size_t)rows};
    double* s = st.O + (size_t)rows * d;
    double* tmax = s + (size_t)rows * Bk;
    state_reset(&st);
    for (int r = 0; r < rows; ++r) {
      const int64_t row = r0 + r;
      qrows[r] = q + ((size_t)(b * p->Hq + h) * p->Lq + (size_t)row) * dk;
      last_vis[r] = p->causal ? row + off : (int64_t)p->Lk - 1;
      if (last_vis[r] > (int64_t)p->Lk - 1) last_vis[r] = p->Lk - 1;
    }
    const uint16_t* kh = k + (size_t)(b * p->Hkv + kvh) * p->Lk * dk;
    const uint16_t* vh = v + (size_t)(b * p->Hkv + kvh) * p->Lk * d;
    uint32_t skipped = 0;

    /* Key tiles in ascending order (§The online-softmax pass: one pass). */
    for (int64_t j = 0; j < nT; ++j) {
      const int64_t k0 = j * Bk;
      const int64_t nk = (k0 + Bk <= p->Lk) ? Bk : p->Lk - k0;
      const int have_ov = mask_override != NULL;
      const int ov = have_ov ? mask_override[(size_t)i * nT + j] : 0;
      double c;
      const int dec =
          tile_step(&st, qrows, last_vis, kh, dk, vh, k0, nk, p->scale, ln_lambda, have_ov, ov, s, tmax, &c);
      if (dec == ORC_SKIPPED) ++skipped;
      if (mask) mask[(size_t)i * nT + j] = (uint8_t)dec;
      if (margin) margin[(size_t)i * nT + j] = c;
    }
    /* Return O / l (a row that saw no key at all yields 0). */
    if (o) {
      double* ou = o + (size_t)i * Bq * d;
      memset(ou, 0, sizeof(double) * (size_t)Bq * d);
      for (int r = 0; r < rows; ++r)
        if (st.l[r] > 0.0)
          for (int e = 0; e < d; ++e) ou[(size_t)r * d + e] = st.O[(size_t)r * d + e] / st.l[r];
    }
    if (counts) counts[i] = skipped;
    free(mbuf);
    free(last_vis);
    free(qrows);
  }
  return bad ? -1 : 0;
}

int orc_decode(const orc_decode_problem* p, const uint16_t* q, const uint16_t* k,
               const uint16_t* v, const int64_t* units, int64_t n_units,
               const uint8_t* mask_override, double* o, uint8_t* mask, double* margin,
               uint32_t* counts, double* part_m, double* part_l, double* part_o) {
  if (!p || !q || !k || !v) return -1;
  if (p->B < 1 || p->Hq < 1 || p->Hkv < 1 || p->Hq % p->Hkv != 0 || p->Lk < 1 || p->d < 1 ||
      p->dv < 0 || p->Bk < 1 || p->num_splits < 1 || !(p->lambda >= 0.0) || p->lambda > 1.0)
    return -1;
  /* dk: query/key width; d: value width (the MLA reading gives them apart) */
  const int G = p->Hq / p->Hkv, dk = p->d, d = (p->dv > 0) ? p->dv : p->d, Bk = p->Bk,
            S = p->num_splits;
  const int64_t nT = ceil_div(p->Lk, Bk), T = ceil_div(nT, S);
  const int64_t total = (int64_t)p->B * p->Hkv;
  if (units == NULL) n_units = total;
  const double ln_lambda = (p->lambda > 0.0) ? log(p->lambda) : -INFINITY;
  int bad = 0;

#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < n_units; ++i) {
    const int64_t u = units ? units[i] : i;
    if (u < 0 || u >= total) {
      bad = 1;
      continue;
    }
    const int64_t b = u / p->Hkv, kvh = u % p->Hkv;
    double* buf = malloc(sizeof(double) * (size_t)G * (3 + (size_t)d + (size_t)Bk + 3 + (size_t)d) * (size_t)S);
    int64_t* last_vis = malloc(sizeof(int64_t) * (size_t)G);
    const uint16_t** qrows = malloc(sizeof(uint16_t*) * (size_t)G);
    double* sm = buf;                              /* [G][S] */
    double* sl = sm + (size_t)G * S;               /* [G][S] */
    double* sO = sl + (size_t)G * S;               /* [G][S][d] */
    double* work = sO + (size_t)G * S * d;
    run_state st = {G, d, work, work + G, work + 2 * (size_t)G};
    double* s = st.O + (size_t)G * d;
    double* tmax = s + (size_t)G * Bk;
    for (int g = 0; g < G; ++g) {
      qrows[g] = q + ((size_t)b * p->Hq + (size_t)kvh * G + g) * dk;
      last_vis[g] = p->Lk - 1;
    }
    const uint16_t* kh = k + (size_t)(b * p->Hkv + kvh) * p->Lk * dk;
    const uint16_t* vh = v + (size_t)(b * p->Hkv + kvh) * p->Lk * d;

    for (int sp = 0; sp < S; ++sp) {
      /* Each split runs its own online pass from an empty state. */
      state_reset(&st);
      uint32_t skipped = 0;
      const int64_t j0 = sp * T, j1 = (j0 + T < nT) ? j0 + T : nT;
      for (int64_t j = j0; j < j1; ++j) {
        const int64_t k0 = j * Bk;
        const int64_t nk = (k0 + Bk <= p->Lk) ? Bk : p->Lk - k0;
        const int have_ov = mask_override != NULL;
        const int ov = have_ov ? mask_override[(size_t)i * nT + j] : 0;
        double c;
        const int dec = tile_step(&st, qrows, last_vis, kh, dk, vh, k0, nk, p->scale, ln_lambda,
                                  have_ov, ov, s, tmax, &c);
        if (dec == ORC_SKIPPED) ++skipped;
        if (mask) mask[(size_t)i * nT + j] = (uint8_t)dec;
        if (margin) margin[(size_t)i * nT + j] = c;
      }
      if (counts) counts[(size_t)i * S + sp] = skipped;
      for (int g = 0; g < G; ++g) {
        sm[(size_t)g * S + sp] = st.m[g];
        sl[(size_t)g * S + sp] = st.l[g];
        memcpy(sO + ((size_t)g * S + sp) * d, st.O + (size_t)g * d, sizeof(double) * (size_t)d);
      }
    }
    /* Log-sum-exp merge of the splits: m* = max m_s, l = sum l_s e^(m_s - m*),
       O = sum O_s e^(m_s - m*), output O / l.  Empty splits (l = 0) drop out. */
    for (int g = 0; g < G; ++g) {
      double mstar = -INFINITY;
      for (int sp = 0; sp < S; ++sp)
        if (sl[(size_t)g * S + sp] > 0.0 && sm[(size_t)g * S + sp] > mstar) mstar = sm[(size_t)g * S + sp];
      double l = 0.0;
      double* og = o ? o + ((size_t)i * G + g) * d : NULL;
      if (og) memset(og, 0, sizeof(double) * (size_t)d);
      for (int sp = 0; sp < S; ++sp) {
        const double ls = sl[(size_t)g * S + sp];
        if (!(ls > 0.0)) continue;
        const double w = exp(sm[(size_t)g * S + sp] - mstar);
        l += ls * w;
        if (og)
          for (int e = 0; e < d; ++e) og[e] += sO[((size_t)g * S + sp) * d + e] * w;
      }
      if (og && l > 0.0)
        for (int e = 0; e < d; ++e) og[e] /= l;
      for (int sp = 0; sp < S; ++sp) {
        const size_t gi = ((size_t)i * G + g) * S + sp;
        if (part_m) part_m[gi] = sm[(size_t)g * S + sp];
        if (part_l) part_l[gi] = sl[(size_t)g * S + sp];
        if (part_o) memcpy(part_o + gi * d, sO + ((size_t)g * S + sp) * d, sizeof(double) * (size_t)d);
      }
    }
    free(buf);
    free(last_vis);
    free(qrows);
  }
  return bad ? -1 : 0;
}

static int cmp_double(const void* a, const void* b) {
  const double x = *(const double*)a, y = *(const double*)b;
  return (x > y) - (x < y);
}

int orc_calibrate(const double* margin, const uint8_t* mask, int64_t n, double target, double L,
                  double* a_out, int64_t* k_out, int64_t* n_out) {
  if (!margin || !mask || !a_out || n < 0 || !(target >= 0.0) || target > 1.0 || !(L > 0.0))
    return -1;
  double* c = malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
  int64_t N = 0;
  for (int64_t i = 0; i < n; ++i)
    if (mask[i] != ORC_NOT_EVALUATED) c[N++] = margin[i];
  qsort(c, (size_t)N, sizeof(double), cmp_double);
  /* §Calibratie: choose a so that a fixed fraction of tiles is skipped.
     With lambda = a/L, tile j is skipped iff c_j < ln(lambda), so any
     ln(lambda) in (c_(k), c_(k+1)] skips exactly k tiles (k-th smallest c,
     1-based); the midpoint leaves the widest margin on both sides. */
  int64_t k = (int64_t)floor(target * (double)N + 0.5);
  double a = 0.0;
  if (k > 0) {
    double lo = c[k - 1];
    double hi = (k < N) ? c[k] : INFINITY;
    if (hi > 0.0) hi = 0.0; /* lambda <= 1 */
    if (lo >= hi) {
      /* Unreachable under lambda <= 1: skip as many tiles as lambda = 1 allows. */
      a = L;
    } else {
      a = L * exp(0.5 * (lo + hi));
    }
  }
  const double ln_lambda = (a > 0.0) ? log(a / L) : -INFINITY;
  int64_t achieved = 0;
  for (int64_t i = 0; i < N; ++i)
    if (c[i] < ln_lambda) ++achieved;
  free(c);
  *a_out = a;
  if (k_out) *k_out = achieved;
  if (n_out) *n_out = N;
  return 0;
}
