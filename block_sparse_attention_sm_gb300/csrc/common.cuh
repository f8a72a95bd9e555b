// Internal declarations shared by the kernels and the C-ABI layer.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include <cuda_bf16.h>

#include "ssattn.h"

namespace ssattn {

constexpr int kTile = 128;  // key tile and prefill query block
constexpr int kVoteChunkTiles = 2048;  // prefill: key tiles decided per vote/compute run

// Device status word: kernels that give up a bounded wait OR a code into the
// word whose address the launch passes them (module memory of the C-ABI
// layer, not an allocation); ss_stream_status reads and clears it.
constexpr uint32_t kDevStatusTimeout = 1u;

__device__ __forceinline__ void report_timeout(uint32_t* status) {
  if (status != nullptr) atomicOr(status, kDevStatusTimeout);
}

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Packed fp32 pairs (two IEEE fp32 operations per instruction) and a
// three-input maximum: the softmax loops are bound by instruction issue.
__device__ __forceinline__ uint64_t f32x2(float lo, float hi) {
  return static_cast<uint64_t>(__float_as_uint(lo)) |
         (static_cast<uint64_t>(__float_as_uint(hi)) << 32);
}
__device__ __forceinline__ float f32x2_lo(uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v)); }
__device__ __forceinline__ float f32x2_hi(uint64_t v) { return __uint_as_float(static_cast<uint32_t>(v >> 32)); }
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

enum class Mode : int { kDense = 0, kSparse = 1, kCount = 2 };

struct PrefillParams {
  int B, Hq, Hkv, Lq, Lk;
  int G;          // Hq / Hkv
  int nQB, nT;    // query blocks, key tiles
  int causal;
  int chunk_tiles;   // key tiles decided per vote/compute run (<= the kernel's capacity)
  float scale_log2;  // scale * log2(e): exponent factor on raw scores
  float scale;       // natural-log factor (for margins)
  float thr_raw;     // ln(lambda) / scale: skip iff tile_max - m < thr_raw (raw units)
  __nv_bfloat16* o;
  uint32_t* counts;
  uint8_t* mask;
  float* margin;
  uint32_t* status;
};

struct DecodeParams {
  int B, Hq, Hkv, Lk, d;
  int G;
  int nT, S, T;      // tiles, splits, tiles per split
  float scale_log2;
  float scale;
  float thr_raw;
  const __nv_bfloat16* q;  // [B][Hq][d]; K and V are read through tensor maps
  __nv_bfloat16* o;       // final output when S == 1
  float* part;            // [B*Hq][S][d + 2] partial (O..., m, l) when S > 1
  uint32_t* counts;
  uint8_t* mask;
  float* margin;
  uint32_t* status;
  int count_only;
  int fault_inject;  // test only: skip one K copy per split (bounded-wait expiry)
  // Paged KV cache (nullptr: contiguous [B][Hkv][Lk][d]).  K and V are pages
  // of one 128-key tile, [num_pages][Hkv][128][d]; page_table[b][j] is the
  // page of sequence b's tile j; seq_lens[b] its length.  Each sequence has
  // its own threshold lambda_b = min(1, lambda_a / seq_len) and its own
  // split of its ceil(seq_len / 128) tiles.
  const int32_t* page_table;
  const int32_t* seq_lens;
  int max_pages;
  float lambda_a;
};

// Launchers (return a CUDA error code; arguments are already validated).
cudaError_t launch_prefill(int d, Mode mode, const CUtensorMap& tq, const CUtensorMap& tk,
                           const CUtensorMap& tv, const PrefillParams& p, cudaStream_t st);
cudaError_t launch_decode(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p,
                          Mode mode, cudaStream_t st);

}  // namespace ssattn
