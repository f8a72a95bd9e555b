// Internal declarations of the latent-attention (MLA) decode kernel.
#pragma once
#include "common.cuh"
#include "ptx_sm103.cuh"

namespace ssattn {

// Absorbed multi-head latent attention: one latent head per sequence, rows
// of kMlaLatent latent entries followed by kMlaRope rotary entries.  The keys
// are the whole rows, the values their latent part.
constexpr int kMlaLatent = 512;
constexpr int kMlaRope = 64;
constexpr int kMlaDk = kMlaLatent + kMlaRope;
constexpr int kMlaNarrowHeads = 16;  // one softmax warpgroup (MMA N = 16) up to here
constexpr int kMlaWideHeads = 32;    // two softmax warpgroups (MMA N = 32) up to here
constexpr int kMlaRowsMaxHeads = 64;  // heads as MMA rows, latent split over two CTAs
constexpr int kMlaMaxHeads = kMlaRowsMaxHeads;

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

// Heads 1..32: keys on the TMEM lanes (one softmax warpgroup of 16 heads up
// to 16 heads, two above).
cudaError_t launch_mla_decode(const CUtensorMap& tkv, const MlaParams& p, Mode mode,
                              cudaStream_t st);
// Heads 33..64: heads as the MMA rows, O's latent entries split over two CTAs.
cudaError_t launch_mla_decode_rows(const CUtensorMap& tkv, const MlaParams& p, Mode mode,
                                   cudaStream_t st);
// Log-sum-exp merge of the S > 1 partial states in p.part into p.o.
cudaError_t launch_mla_merge(const MlaParams& p, cudaStream_t st);

// tcgen05.ld of 16 consecutive fp32 columns of the warp's 32 lanes.
__device__ __forceinline__ void mla_tmem_ld16(uint32_t taddr, float (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=f"(r[0]), "=f"(r[1]), "=f"(r[2]), "=f"(r[3]), "=f"(r[4]), "=f"(r[5]), "=f"(r[6]),
        "=f"(r[7]), "=f"(r[8]), "=f"(r[9]), "=f"(r[10]), "=f"(r[11]), "=f"(r[12]), "=f"(r[13]),
        "=f"(r[14]), "=f"(r[15])
      : "r"(taddr));
}

// Wait (bounded, no abort flag) for the newest copy issued into each slot of
// a ring of N slots after n copies: the slot of copy i is i % N.
template <int N>
__device__ __forceinline__ void mla_drain_ring(uint64_t* full, int n) {
  for (int s = 0; s < N; ++s)
    if (n > s) mbar_wait(&full[s], ((((n - 1 - s) / N) * N + s) / N) & 1, nullptr);
}

// Maximum over the warp (every lane gets it).
__device__ __forceinline__ float mla_warp_max(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}

}  // namespace ssattn
