// Internal declarations of the latent-attention (MLA) decode kernel.
#pragma once
#include "common.cuh"

namespace ssattn {

// Absorbed multi-head latent attention: one latent head per sequence, rows
// of kMlaLatent latent entries followed by kMlaRope rotary entries.  The keys
// are the whole rows, the values their latent part.
constexpr int kMlaLatent = 512;
constexpr int kMlaRope = 64;
constexpr int kMlaDk = kMlaLatent + kMlaRope;
constexpr int kMlaMaxHeads = 16;  // voting group = MMA N of at most 16 rows

struct MlaParams {
  int B, Hq, Lk;
  int nT, S, T;  // tiles, splits, tiles per split
  float scale_log2;
  float scale;
  float thr_raw;           // ln(lambda) / scale: skip iff tile_max - m < thr_raw
  const __nv_bfloat16* q;  // [B][Hq][kMlaDk]; the cache is read through a tensor map
  __nv_bfloat16* o;        // [B][Hq][kMlaLatent] when S == 1
  float* part;             // [B*Hq][S][kMlaLatent + 2] partial (O..., m, l) when S > 1
  uint32_t* counts;        // [B][S]
  uint8_t* mask;           // [B][nT]
  float* margin;           // [B][nT]
  uint32_t* status;
  // Paged latent cache (nullptr: contiguous [B][Lk][kMlaDk]).  Pages of one
  // 128-key tile, [num_pages][128][kMlaDk]; page_table[b][j] is the page of
  // sequence b's tile j, seq_lens[b] its length; each sequence has its own
  // threshold lambda_b = min(1, lambda_a / seq_len) and its own split of its
  // ceil(seq_len / 128) tiles.
  const int32_t* page_table;
  const int32_t* seq_lens;
  int max_pages;
  float lambda_a;
};

cudaError_t launch_mla_decode(const CUtensorMap& tkv, const MlaParams& p, Mode mode,
                              cudaStream_t st);

}  // namespace ssattn
