/*
 * ssattn -- skip-softmax (BLASST) attention forward for NVIDIA GB300 (sm_103a).
 *
 * C ABI.  Plain pointers and sizes only; every device pointer is memory the
 * caller owns (e.g. a framework tensor's data pointer), and the library
 * allocates no device memory.  Every compute call is asynchronous on the
 * caller's stream (`stream` is a cudaStream_t passed as void*, NULL meaning
 * the legacy default stream); a returned SS_OK means the work was validated
 * and launched.  Errors found on the device (a bounded wait that expired)
 * are recorded in a library-wide device status word read by
 * ss_stream_status().
 *
 * The method (cited by page title and section):
 *   "Skip-Softmax" (vllm-omni design doc):
 *     §The online-softmax pass -- one streaming pass over 128-key tiles
 *       keeping the running max m, the denominator l = sum exp(s - m) and the
 *       numerator O = sum exp(s - m) v, returning O / l;
 *     §The skip test -- once tile j's scores Q K_j^T * scale are known, the
 *       tile is skipped when exp(tile_max - running_max) < threshold: no
 *       exponentials, no P.V accumulation, no contribution to l or O;
 *     §What this bounds -- Q K^T always runs; the decision is per tile;
 *     §The threshold -- threshold = factor / seqlen, factor either calibrated
 *       (factor = a * exp(b * target_sparsity)) or direct.
 *   "BLASST: Dynamic BLocked Attention Sparsity via Softmax Thresholding"
 *   (summary of arXiv 2512.12087):
 *     §Methodologie -- the test in log form (local max - running max < ln
 *       lambda); in decode a skipped tile's V block is never loaded;
 *     §Calibratie -- lambda = a / L; an automated procedure picks a so that
 *       a fixed fraction of tiles is skipped at any context length;
 *     §Kernel-ontwerp -- prefill skips softmax and P.V MMA, decode skips V
 *       loads with batched loading of surviving tiles.
 *
 * Conventions shared by all entry points:
 *   - q, k, v, o are bf16, contiguous, 16-byte aligned.  Prefill layouts:
 *     q, o [B, Hq, Lq, d]; k, v [B, Hkv, Lk, d].  Decode: q, o [B, Hq, d],
 *     k, v [B, Hkv, Lk, d].
 *   - d is 64 or 128.  Hq must be a multiple of Hkv; query head h reads KV
 *     head h / (Hq / Hkv) (MHA: Hkv = Hq, GQA, MQA: Hkv = 1).
 *   - Key tiles and prefill query blocks are 128 wide; Lq and Lk need not be
 *     multiples of 128 (tails are masked).
 *   - Causal masking is bottom-right aligned: key k is visible to query row r
 *     iff k <= r + (Lk - Lq).
 *   - lambda in [0, 1]; lambda = 0 runs the dense path (no vote at all).
 *     A tile is skipped iff every query row of the block (decode: every query
 *     head sharing the KV head) has exp(scale*(tile_max - running_max)) <
 *     lambda, the running max being the maximum over the earlier tiles of the
 *     same pass (decode: the same split).  A row with no visible key in the
 *     tile does not veto.  The first tile of a pass is never skipped.
 */
#ifndef SSATTN_H
#define SSATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SS_OK = 0,
  SS_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad shape, lambda or scale */
  SS_ERR_UNSUPPORTED = 2,  /* d not in {64,128}, decode with Hq/Hkv > 128 (> 32 at
                              d = 64), latent decode with other widths or Hq > 64,
                              latent prefill with widths other than 192/128, or the
                              current device is not sm_103 */
  SS_ERR_CUDA = 3,         /* a CUDA runtime call failed (launch, copy, sync) */
  SS_ERR_TIMEOUT = 4,      /* a kernel's bounded wait expired (logic error; reported, not hung) */
  SS_ERR_WORKSPACE = 5     /* decode workspace missing or too small */
} ss_status;

/* Optional debug / calibration outputs, all device pointers, all nullable. */
typedef struct {
  /* One byte per (unit, key tile): 0 kept, 1 skipped, 2 not evaluated
     (causal tiles past the diagonal).  Prefill: [B*Hq*ceil(Lq/128)][nT];
     decode: [B*Hkv][nT] with tiles indexed globally. */
  uint8_t* skip_mask;
  /* Vote statistic c_j = max over rows of scale*(tile_max - running_max) in
     natural-log units, same indexing as skip_mask; +INF when some row has no
     running max yet, NAN when not evaluated.  The tile is skipped iff
     c_j < ln(lambda). */
  float* vote_margin;
  /* Nonzero: compute scores, the vote and the counters only -- no
     exponentials, no P.V, no V loads, no output written (o may be NULL).
     Decisions equal those of the full pass: a skipped tile never raises the
     running max when lambda <= 1. */
  int count_only;
  /* Test only, decode only (0 otherwise).  1: the copy of each split's
     second K tile is never issued, so the kernel's bounded wait for it
     expires (after about a second); the kernel then lets its other copies
     land, returns, and ss_stream_status() reports SS_ERR_TIMEOUT.  The
     output is unspecified; the context stays usable. */
  int fault_inject;
  /* Test only, prefill only (0 otherwise).  The prefill kernel decides a
     run of key tiles (by default 2048) before it computes the run's kept
     tiles, and carries the softmax state from run to run; a value in
     [1, 2048] shortens the run so that short inputs take the multi-run
     path.  Results do not depend on it (up to rounding).  It applies to the
     one-CTA kernel, which a nonzero value selects at d = 64 and 128 (unless
     prefill_kernel asks for the pair kernel, which ignores it). */
  int vote_chunk_tiles;
  /* Prefill only (0 otherwise): which of the library's two prefill kernels
     computes the pass.  1 selects the one-CTA kernel (two query blocks per
     CTA; the decisions of a run of tiles first, kept tiles second), 2 the
     CTA-pair kernel (two-SM MMAs, one pass).  0 chooses automatically: at
     d = 128 the pair kernel for the dense and voting paths (ahead from dense
     up to ~70% skipped tiles) and the one-CTA kernel for counting; at d = 64
     the one-CTA kernel (ahead at ~70% skipped tiles; the pair kernel leads
     at ~50%).  At ~90% skipped tiles and above the one-CTA kernel is the
     faster one.  Decisions and counts do not depend on the kernel; outputs
     agree up to rounding.  d_qk = 192 has only the pair kernel: asking for
     the other returns SS_ERR_UNSUPPORTED. */
  int prefill_kernel;
} ss_debug_opts;

/*
 * Prefill forward (all §8 prefill steps: TMA staging, Q K^T on tcgen05,
 * mask + tile max, skip vote, online softmax on kept tiles, P.V on tcgen05,
 * O / l epilogue).
 *   skip_counts: nullable device buffer [B*Hq*ceil(Lq/128)], one uint32 per
 *   (b, h_q, query block) = skipped tiles of that unit; overwritten.
 * Returns SS_OK, SS_ERR_INVALID_ARG, SS_ERR_UNSUPPORTED or SS_ERR_CUDA.
 */
ss_status ss_attn_prefill(const void* q, const void* k, const void* v, void* o, int B, int Hq,
                          int Hkv, int Lq, int Lk, int d, float scale, int causal, float lambda,
                          uint32_t* skip_counts, void* stream);

ss_status ss_attn_prefill_ex(const void* q, const void* k, const void* v, void* o, int B,
                             int Hq, int Hkv, int Lq, int Lk, int d, float scale, int causal,
                             float lambda, uint32_t* skip_counts, const ss_debug_opts* dbg,
                             void* stream);

/*
 * Latent-attention (MLA) prefill: the skip test on multi-head latent
 * attention in its unabsorbed prefill form, which the BLASST summary names
 * among the attention kinds its prefill kernels support (§Belangrijkste
 * Bijdragen, item 4: MHA, GQA, MQA and MLA).  Read as attention whose query
 * and key rows (non-rotary latent projection followed by the rotary part) are
 * wider than the value rows; the pages give no shapes, and the widths
 * supported are DeepSeek-V2/V3's published ones: d_qk = 128 + 64 = 192,
 * d_v = 128.  Everything else -- tiles, vote, causal alignment, GQA/MQA
 * head map, counters, debug outputs -- is that of ss_attn_prefill.
 *   q [B, Hq, Lq, d_qk], k [B, Hkv, Lk, d_qk], v [B, Hkv, Lk, d_v],
 *   o [B, Hq, Lq, d_v]; bf16, contiguous, 16-byte aligned.
 * Returns SS_OK, SS_ERR_INVALID_ARG, SS_ERR_UNSUPPORTED (other widths, or
 * the current device is not sm_103) or SS_ERR_CUDA.
 */
ss_status ss_attn_mla_prefill(const void* q, const void* k, const void* v, void* o, int B, int Hq,
                              int Hkv, int Lq, int Lk, int d_qk, int d_v, float scale, int causal,
                              float lambda, uint32_t* skip_counts, void* stream);

ss_status ss_attn_mla_prefill_ex(const void* q, const void* k, const void* v, void* o, int B,
                                 int Hq, int Hkv, int Lq, int Lk, int d_qk, int d_v, float scale,
                                 int causal, float lambda, uint32_t* skip_counts,
                                 const ss_debug_opts* dbg, void* stream);

/*
 * Bytes of device workspace ss_attn_decode needs for the per-split partial
 * states (m, l, O in fp32): 0 when num_kv_splits == 1.
 */
size_t ss_attn_decode_workspace_size(int B, int Hq, int d, int num_kv_splits);

/*
 * Split-KV decode forward (one query token per sequence).  The nT =
 * ceil(Lk/128) key tiles are cut into num_kv_splits contiguous ranges of
 * ceil(nT/num_kv_splits) tiles; each range runs its own online pass (its
 * first tile is always kept), streams all of its K, loads V only for kept
 * tiles, and writes a partial (m, l, O); a second kernel merges the
 * partials by log-sum-exp into bf16 o.  The G = Hq/Hkv query heads of a KV
 * head vote together on each tile; G <= 128 at d = 128 (groups above 16
 * heads run with the heads as the rows of the MMAs), G <= 32 at d = 64
 * (SS_ERR_UNSUPPORTED above).
 *   skip_counts: nullable device buffer [B*Hkv*num_kv_splits] (skipped tiles
 *     per (sequence, KV head, split)); overwritten.
 *   workspace: device buffer of at least
 *     ss_attn_decode_workspace_size(B, Hq, d, num_kv_splits) bytes, 16-byte
 *     aligned (may be NULL when that size is 0); contents need not be
 *     initialised and are clobbered.
 * Returns SS_OK, SS_ERR_INVALID_ARG, SS_ERR_UNSUPPORTED, SS_ERR_WORKSPACE or
 * SS_ERR_CUDA.
 */
ss_status ss_attn_decode(const void* q, const void* k_cache, const void* v_cache, void* o, int B,
                         int Hq, int Hkv, int Lk, int d, float scale, float lambda,
                         int num_kv_splits, uint32_t* skip_counts, void* workspace,
                         size_t workspace_bytes, void* stream);

ss_status ss_attn_decode_ex(const void* q, const void* k_cache, const void* v_cache, void* o,
                            int B, int Hq, int Hkv, int Lk, int d, float scale, float lambda,
                            int num_kv_splits, uint32_t* skip_counts, void* workspace,
                            size_t workspace_bytes, const ss_debug_opts* dbg, void* stream);

/*
 * Split-KV decode over a paged, variable-length KV cache (the serving
 * layout the pages' engine integrations imply: BLASST summary,
 * §Belangrijkste Bijdragen -- TensorRT-LLM / FlashInfer; the skip test per
 * sequence follows "Skip-Softmax" §The threshold).
 *   k_pages, v_pages: bf16 [num_pages][Hkv][128][d], 16-byte aligned; a page
 *     holds one 128-key tile of one sequence for every KV head.
 *   page_table: device int32 [B][max_pages]; entry j of row b is the page of
 *     sequence b's keys [128j, 128j + 128).  Entries past a sequence's last
 *     page are not read.  An entry outside [0, num_pages) reads zeros.
 *   seq_lens: device int32 [B], keys per sequence (0 .. 128*max_pages; larger
 *     values are clamped).  The rows of a sequence's last page past its end
 *     are ignored, whatever they hold.
 *   lambda_a: the a of lambda = a / L, applied per sequence with L its own
 *     length: lambda_b = min(1, lambda_a / seq_lens[b]); 0 keeps every tile.
 *   num_kv_splits: each sequence's ceil(L_b/128) tiles are cut into this
 *     many contiguous ranges of ceil(tiles_b / num_kv_splits) tiles (ranges
 *     past the end are empty).
 *   skip_counts: nullable, [B*Hkv*num_kv_splits] as in ss_attn_decode.
 *   workspace: as in ss_attn_decode (ss_attn_decode_workspace_size).
 *   dbg: nullable; skip_mask / vote_margin are [B*Hkv][max_pages] (tiles past
 *     a sequence's end are marked not evaluated); count_only as elsewhere.
 * Returns SS_OK, SS_ERR_INVALID_ARG (null pointer, misalignment, B, Hq, Hkv,
 * num_pages, max_pages or num_kv_splits < 1, Hq % Hkv != 0, scale <= 0,
 * lambda_a < 0 or not finite), SS_ERR_UNSUPPORTED, SS_ERR_WORKSPACE or
 * SS_ERR_CUDA.
 */
ss_status ss_attn_decode_paged(const void* q, const void* k_pages, const void* v_pages,
                               const int32_t* page_table, const int32_t* seq_lens, void* o,
                               int B, int Hq, int Hkv, int num_pages, int max_pages, int d,
                               float scale, float lambda_a, int num_kv_splits,
                               uint32_t* skip_counts, void* workspace, size_t workspace_bytes,
                               const ss_debug_opts* dbg, void* stream);

/*
 * Decode for callers that cannot allocate device memory.  The pages have no
 * counterpart to this entry point; it exists for users of this library, not
 * for the method.
 *
 * Some callers of a decode step are handed their input and output buffers
 * and nothing else -- a kernel plugin inside an inference engine that owns
 * all device memory, or a latency-critical serving loop that must not call
 * cudaMalloc (an allocation can synchronise the device and may fail under
 * memory pressure).  They cannot provide ss_attn_decode's workspace.  This
 * variant runs the same kernels as ss_attn_decode, but keeps the per-split
 * partial states in a fixed device array that is part of the library itself
 * (SS_DECODE_STATIC_SCRATCH_BYTES, held by every GPU that loads the library
 * until the process exits).  It calls no cudaMalloc, cudaFree or other
 * allocating routine.
 *
 * Arguments, layouts and results are those of ss_attn_decode without the
 * workspace.  Calls whose partials need more than
 * SS_DECODE_STATIC_SCRATCH_BYTES (B*Hq*num_kv_splits*(d+2)*4 bytes when
 * num_kv_splits > 1) return SS_ERR_WORKSPACE without launching anything.
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture on that device.  Every call on a device shares the one array and
 * it keeps the previous call's contents; each launch writes every partial it
 * later reads, so nothing has to be cleared between calls.  Calls whose
 * execution overlaps on the GPU (different streams, or several host threads)
 * race on the array: serialise them.
 */
#define SS_DECODE_STATIC_SCRATCH_BYTES (16u << 20)
/* The size of that array in the library as built (SS_DECODE_STATIC_SCRATCH_BYTES
   of the header it was compiled with); host only, needs no GPU. */
size_t ss_decode_static_scratch_bytes(void);
ss_status ss_attn_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                 void* o, int B, int Hq, int Hkv, int Lk, int d, float scale,
                                 float lambda, int num_kv_splits, uint32_t* skip_counts,
                                 void* stream);

/*
 * Latent-attention (MLA) decode: the skip test on multi-head latent
 * attention, which the BLASST summary names among the attention kinds its
 * prefill and decode kernels support (§Belangrijkste Bijdragen, item 4:
 * MHA, GQA, MQA and MLA), without giving its shapes.  Read as the absorbed decode
 * form: each sequence caches one latent row per token, d_latent latent
 * entries followed by d_rope rotary entries; the keys are the whole rows
 * (width dk = d_latent + d_rope), the values their first d_latent entries,
 * and every query head attends to that one latent head.  All Hq heads of a
 * sequence are therefore the voting group of a tile: a tile is skipped only
 * if exp(tile_max - running_max) < lambda holds for every head (BLASST
 * summary, §Methodologie; "Skip-Softmax" §What this bounds: one decision
 * per tile).  The split of
 * the nT = ceil(Lk/128) tiles into num_kv_splits contiguous ranges and the
 * log-sum-exp merge are those of ss_attn_decode.  The values are read from
 * the key rows already on chip, so a skipped tile saves the exponentials and
 * the P.V products, not memory traffic.
 *   q:  [B][Hq][dk] bf16 (the absorbed queries), 16-byte aligned.
 *   kv: [B][Lk][dk] bf16 latent cache, contiguous, 16-byte aligned.
 *   o:  [B][Hq][d_latent] bf16.
 *   Only d_latent = 512, d_rope = 64 and 1 <= Hq <= 64 are supported (up to
 *   16 heads take one softmax warpgroup, 17..32 heads two; 33..64 heads run
 *   with the heads as the rows of the MMAs and the latent entries of O split
 *   over two CTAs per (sequence, split)).
 *   skip_counts: nullable device buffer [B*num_kv_splits]; overwritten.
 *   workspace: device buffer of at least
 *     ss_attn_mla_decode_workspace_size(B, Hq, d_latent, num_kv_splits)
 *     bytes, 16-byte aligned (may be NULL when that size is 0).
 *   dbg (the _ex form): skip_mask / vote_margin are [B][nT]; count_only as
 *     elsewhere.
 * Returns SS_OK, SS_ERR_INVALID_ARG (null or misaligned pointer, B, Hq, Lk or
 * num_kv_splits < 1, lambda outside [0, 1], scale <= 0), SS_ERR_UNSUPPORTED,
 * SS_ERR_WORKSPACE or SS_ERR_CUDA.  Asynchronous on `stream`.
 */
size_t ss_attn_mla_decode_workspace_size(int B, int Hq, int d_latent, int num_kv_splits);

ss_status ss_attn_mla_decode(const void* q, const void* kv, void* o, int B, int Hq, int Lk,
                             int d_latent, int d_rope, float scale, float lambda,
                             int num_kv_splits, uint32_t* skip_counts, void* workspace,
                             size_t workspace_bytes, void* stream);

ss_status ss_attn_mla_decode_ex(const void* q, const void* kv, void* o, int B, int Hq, int Lk,
                                int d_latent, int d_rope, float scale, float lambda,
                                int num_kv_splits, uint32_t* skip_counts, void* workspace,
                                size_t workspace_bytes, const ss_debug_opts* dbg, void* stream);

/*
 * Latent-attention decode over a paged, variable-length latent cache: the
 * computation of ss_attn_mla_decode per sequence, with the layout and the
 * per-sequence rules of ss_attn_decode_paged.
 *   kv_pages:   [num_pages][128][d_latent + d_rope] bf16, one 128-key tile per
 *               page (rows past a sequence's end in its last page are ignored).
 *   page_table: [B][max_pages] int32 device array; entry j of sequence b is the
 *               page of its keys [128 j, 128 j + 128).  Only the first
 *               ceil(seq_lens[b] / 128) entries of a row are read.
 *   seq_lens:   [B] int32 device array, keys per sequence (0 <= L_b <=
 *               128 * max_pages; a zero-length sequence gives zeros).
 *   lambda_a:   the a of lambda_b = min(1, a / L_b) ("Skip-Softmax" §The
 *               threshold: threshold = factor / seqlen), per sequence; 0 =
 *               dense.
 *   num_kv_splits: each sequence's tiles in that many contiguous ranges of
 *               ceil(tiles_b / num_kv_splits) tiles.
 *   skip_counts: nullable, [B*num_kv_splits]; workspace as in
 *               ss_attn_mla_decode.
 *   dbg:        nullable; skip_mask / vote_margin are [B][max_pages] (tiles past
 *               a sequence's end are marked not evaluated).
 * Returns SS_OK, SS_ERR_INVALID_ARG (null pointer, misalignment, B, Hq,
 * num_pages, max_pages or num_kv_splits < 1, scale <= 0, lambda_a < 0 or not
 * finite), SS_ERR_UNSUPPORTED, SS_ERR_WORKSPACE or SS_ERR_CUDA.
 */
ss_status ss_attn_mla_decode_paged(const void* q, const void* kv_pages, const int32_t* page_table,
                                   const int32_t* seq_lens, void* o, int B, int Hq, int num_pages,
                                   int max_pages, int d_latent, int d_rope, float scale,
                                   float lambda_a, int num_kv_splits, uint32_t* skip_counts,
                                   void* workspace, size_t workspace_bytes,
                                   const ss_debug_opts* dbg, void* stream);

/* A calibration problem: the inputs the threshold is fitted on. */
typedef enum { SS_PREFILL = 0, SS_DECODE = 1, SS_MLA_DECODE = 2, SS_MLA_PREFILL = 3 } ss_kind;
typedef struct {
  ss_kind kind;
  const void* q;
  const void* k;
  const void* v;
  int B, Hq, Hkv;
  int Lq;          /* prefill only */
  int Lk;          /* also the L in lambda = a / L */
  int d;
  float scale;
  int causal;      /* prefill only */
  int num_kv_splits; /* decode only */
  /* SS_MLA_DECODE: k is the latent cache [B][Lk][d], v is ignored, Hkv is 1
     and d is the key width d_latent + d_rope (576, of which 512 latent).
     SS_MLA_PREFILL: the tensors of ss_attn_mla_prefill, d = d_qk = 192 (the
     values, 128 wide, are not read by the counting launches). */
  /* Device buffer for the per-unit counters, sized as the matching call's
     skip_counts (prefill: B*Hq*ceil(Lq/128); decode: B*Hkv*num_kv_splits;
     latent decode: B*num_kv_splits). */
  uint32_t* skip_counts;
  void* stream;
  /* Test only, SS_DECODE only (0 otherwise): passed to every count-only
     launch as ss_debug_opts.fault_inject, so that a bounded wait expires and
     the calibration's handling of it can be tested. */
  int fault_inject;
} ss_problem;

/*
 * Automated calibration (BLASST summary, §Calibratie): finds a with
 * lambda = a / Lk such that the fraction of skipped tiles over all evaluated
 * (unit, tile) pairs of `p` is round(target*N)/N, N the number of evaluated
 * tiles.  It bisects on ln a with count-only launches, reading the skipped-
 * tile counters back after each, and returns the log-midpoint of the
 * interval of a that hits the target count (the widest margin), clamped to
 * lambda <= 1.  When the target is not reachable under lambda <= 1 it
 * returns the a closest to it.  Synchronises p->stream.  After each count-only
 * launch it reads and clears the device status word (that of
 * ss_stream_status): if a kernel gave up a bounded wait, the counters are not
 * used and the call returns SS_ERR_TIMEOUT.
 *   a_out: the fitted a (0 when the target rounds to zero skipped tiles).
 *   achieved_out (nullable): skipped / evaluated at the returned a.
 */
ss_status ss_calibrate(const ss_problem* p, float target_sparsity, float* a_out,
                       float* achieved_out);

/*
 * Least-squares fit of ln a = ln A + B * s over n >= 2 points with a > 0
 * ("Skip-Softmax", §The threshold: factor = a * exp(b * target_sparsity);
 * the fitted pair is returned as (A, B)).  Host only.
 */
ss_status ss_fit_factor(const float* s, const float* a, int n, float* A_out, float* B_out);

/* lambda = A * exp(B * s) / L (§The threshold: threshold = factor / seqlen). */
float ss_lambda(float A, float B, float s, int L);

/* Static description of a status code. */
const char* ss_status_string(ss_status st);

/*
 * Synchronise `stream`, then return and clear the device status word:
 * SS_ERR_TIMEOUT if any kernel since the last call gave up a bounded wait,
 * SS_ERR_CUDA if the synchronisation failed, SS_OK otherwise.
 */
ss_status ss_stream_status(void* stream);

#ifdef __cplusplus
}
#endif
#endif /* SSATTN_H */
