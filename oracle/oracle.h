/*
 * Skip-softmax (BLASST) attention oracle: plain, slow, fp64 CPU code.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this library: it exists so that tests/, the bench's CPU-baseline leg
 * and the package smoke check can compare the CUDA kernels against an
 * independent restatement of the method.  It shares no code, header, table
 * or constant with the CUDA path.
 *
 * Sources (web pages; cited by title and section):
 *   [SS]    "Skip-Softmax" (vllm-omni design doc, docs/design/feature/skip_softmax.md):
 *           §The online-softmax pass, §The skip test, §What this bounds,
 *           §The threshold.
 *   [BLASST] "BLASST: Dynamic BLocked Attention Sparsity via Softmax
 *           Thresholding" (gist.science summary of arXiv 2512.12087):
 *           §Methodologie (ln(lambda) test, three skipped operations),
 *           §Calibratie (lambda = a / L, automated calibration of a).
 *
 * Inputs are bf16 bit patterns (uint16), decoded exactly to fp64; every
 * arithmetic step runs in fp64 with the C library's exp/log.
 *
 * Parity status: every function here is pinned by CPU tests against closed
 * forms, brute force and invariants (two-pass softmax at lambda = 0, the
 * prefix-maximum form of the skip decision, the kept-keys restriction, the
 * exact error identity, split-merge invariance, order-statistic calibration).
 */
#ifndef SSATTN_ORACLE_H
#define SSATTN_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Decision codes per (unit, tile). */
enum { ORC_KEPT = 0, ORC_SKIPPED = 1, ORC_NOT_EVALUATED = 2 };

typedef struct {
  int B, Hq, Hkv, Lq, Lk, d; /* d: width of q and k rows */
  double scale;   /* s = scale * q.k */
  int causal;     /* bottom-right aligned: key k visible to row r iff k <= r + (Lk - Lq) */
  double lambda;  /* skip iff exp(tile_max - running_max) < lambda; 0 = dense */
  int Bq, Bk;     /* query-block rows, key-tile size (128 and 128 on the GPU path) */
  int dv;         /* width of v rows and of o; 0: the same as d (multi-head latent
                     attention in its unabsorbed prefill form has wider keys than values) */
} orc_prefill_problem;

/*
 * Prefill.  A unit is one (b, h_q, query block); unit id
 * u = (b*Hq + h)*nQB + qb with nQB = ceil(Lq/Bq).  `units` lists the unit ids
 * to compute (NULL: all, in order).  q and k rows are d wide, v rows dv wide.
 * Outputs are packed per listed unit:
 *   o      [n][Bq][dv]  attention output (rows past Lq left at 0)
 *   mask   [n][nT]      ORC_KEPT / ORC_SKIPPED / ORC_NOT_EVALUATED, nT = ceil(Lk/Bk)
 *   margin [n][nT]      c_j = max over rows (tile_max - running_max), natural-log
 *                       units; +INF when some row has no running max yet; NAN
 *                       when not evaluated
 *   counts [n]          skipped tiles of the unit
 * mask_override [n][nT] (nullable): forces each evaluated tile's decision
 * (nonzero = skip) so that arithmetic can be compared under another
 * implementation's decisions.  Any output pointer may be NULL.
 * Returns 0, or -1 on invalid arguments.
 */
int orc_prefill(const orc_prefill_problem* p, const uint16_t* q, const uint16_t* k,
                const uint16_t* v, const int64_t* units, int64_t n_units,
                const uint8_t* mask_override, double* o, uint8_t* mask, double* margin,
                uint32_t* counts);

typedef struct {
  int B, Hq, Hkv, Lk, d; /* d: width of q and k rows */
  double scale;
  double lambda;
  int num_splits; /* contiguous ranges of T = ceil(nT/S) tiles */
  int Bk;
  int dv;         /* width of v rows and of o; 0: the same as d */
} orc_decode_problem;

/*
 * Decode (one query token per sequence).  A unit is one (b, kv head) with
 * its G = Hq/Hkv query heads; unit id u = b*Hkv + kvh.  Packed outputs:
 * q is [B][Hq][d], k [B][Hkv][Lk][d], v [B][Hkv][Lk][dv] (dv = d unless set:
 * multi-head latent attention reads values of another width than keys).
 *   o      [n][G][dv]
 *   mask   [n][nT]   (tiles indexed globally; splits partition them)
 *   margin [n][nT]
 *   counts [n][S]    skipped tiles per split
 *   part_m, part_l [n][G][S], part_o [n][G][S][dv]: per-split running state
 *          (m in natural-log units, -INF for an empty split), nullable.
 */
int orc_decode(const orc_decode_problem* p, const uint16_t* q, const uint16_t* k,
               const uint16_t* v, const int64_t* units, int64_t n_units,
               const uint8_t* mask_override, double* o, uint8_t* mask, double* margin,
               uint32_t* counts, double* part_m, double* part_l, double* part_o);

/*
 * Calibration by order statistic.  Given the margins c_j of all evaluated
 * tiles (entries whose mask is ORC_NOT_EVALUATED are ignored) and a target
 * sparsity s, let k = round(s*N).  Returns a = L*exp((c_(k) + c_(k+1))/2),
 * the log-midpoint of the interval of ln(lambda) that skips exactly k tiles
 * (upper end clamped to lambda <= 1), or a = 0 when k = 0.  *k_out receives
 * the number of tiles that a skips, *n_out the number N of evaluated tiles.
 */
int orc_calibrate(const double* margin, const uint8_t* mask, int64_t n, double target, double L,
                  double* a_out, int64_t* k_out, int64_t* n_out);

#ifdef __cplusplus
}
#endif
#endif
