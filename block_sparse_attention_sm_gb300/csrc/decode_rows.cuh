// Internal declarations shared by the two split-KV decode kernels.
#pragma once
#include "common.cuh"

namespace ssattn {

// Vote groups (query heads per KV head) above this size run with the heads
// as the MMA rows (decode_rows_sm103.cu); up to it, the kernel with one
// thread per key (decode_sm103.cu).
constexpr int kDecKeyLayoutMaxG = 16;
constexpr int kDecRowsMaxG = 128;  // rows of the MMA

// Heads as MMA rows, d = 128, vote groups of kDecKeyLayoutMaxG + 1 ..
// kDecRowsMaxG rows.
cudaError_t launch_decode_rows(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p,
                               Mode mode, cudaStream_t st);
// Log-sum-exp merge of the S > 1 partial states in p.part into p.o.
cudaError_t launch_decode_merge(const DecodeParams& p, cudaStream_t st);

}  // namespace ssattn
