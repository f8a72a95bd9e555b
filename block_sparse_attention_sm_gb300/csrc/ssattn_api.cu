// C-ABI entry points of libssattn: argument validation, TMA descriptor
// encoding, kernel launches, the calibration of lambda = a / L and the
// device status word.  See include/ssattn.h for the contract of each call.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "decode_rows.cuh"
#include "mla.cuh"

namespace ssattn {

// Prefill on CTA pairs (two-SM MMAs, prefill_pair_sm103.cu); dqk = key width
// (128, or 192 with 128-wide values).  tk must have 64-row boxes (each CTA
// loads half of a key tile).
cudaError_t launch_prefill_pair(int dqk, Mode mode, const CUtensorMap& tq, const CUtensorMap& tk,
                                const CUtensorMap& tv, const PrefillParams& p, cudaStream_t st);

namespace {

__device__ uint32_t g_device_status = 0;

// Device address of the status word for the current device (cached).
uint32_t* status_ptr() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return nullptr;
  static std::mutex mu;
  static std::vector<uint32_t*> ptrs;
  std::lock_guard<std::mutex> lock(mu);
  if (static_cast<int>(ptrs.size()) <= dev) ptrs.resize(dev + 1, nullptr);
  if (ptrs[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_device_status) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<uint32_t*>(ptr);
  }
  return ptrs[dev];
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

// The current device must be sm_103 (GB300); cached per device ordinal.
ss_status check_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return SS_ERR_CUDA;
  static std::mutex mu;
  static std::vector<int> verdict;  // 0 unknown, 1 ok, 2 unsupported
  std::lock_guard<std::mutex> lock(mu);
  if (static_cast<int>(verdict.size()) <= dev) verdict.resize(dev + 1, 0);
  if (verdict[dev] == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return SS_ERR_CUDA;
    verdict[dev] = (major == 10 && minor == 3) ? 1 : 2;
  }
  return verdict[dev] == 1 ? SS_OK : SS_ERR_UNSUPPORTED;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// 3-D view [BH][L][d] of a bf16 tensor, 64 x box_rows boxes, 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, int d, int L, long BH, int box_rows = kTile) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(L),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(L) * d * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

long ceil_div(long a, long b) { return (a + b - 1) / b; }

bool lambda_ok(float lambda) { return lambda >= 0.f && lambda <= 1.f; }  // NaN fails
bool scale_ok(float scale) { return scale > 0.f && std::isfinite(scale); }

// Raw-score threshold: skip iff tile_max - m < ln(lambda) / scale.
float threshold_raw(double ln_lambda, float scale) {
  return static_cast<float>(ln_lambda / static_cast<double>(scale));
}

// d: width of q and k rows; dv: width of v and o rows (0: d).  Supported:
// d = dv in {64, 128}, and d = 192 with dv = 128 (latent-attention prefill).
ss_status prefill_impl(const void* q, const void* k, const void* v, void* o, int B, int Hq,
                       int Hkv, int Lq, int Lk, int d, float scale, int causal, bool dense,
                       float thr_raw, uint32_t* counts, const ss_debug_opts* dbg, void* stream,
                       int dv = 0) {
  if (dv == 0) dv = d;
  const bool count_only = dbg != nullptr && dbg->count_only != 0;
  if (q == nullptr || k == nullptr || v == nullptr || (o == nullptr && !count_only))
    return SS_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || (o != nullptr && !aligned16(o)))
    return SS_ERR_INVALID_ARG;
  if (B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || Lq < 1 || Lk < 1 || !scale_ok(scale))
    return SS_ERR_INVALID_ARG;
  if (!((d == dv && (d == 64 || d == 128)) || (d == 192 && dv == 128))) return SS_ERR_UNSUPPORTED;
  const long nQB = ceil_div(Lq, kTile), nT = ceil_div(Lk, kTile);
  const long units = static_cast<long>(B) * Hq * nQB;
  if (units > 0x7fffffffL || static_cast<long>(B) * Hq > 0x7fffffffL) return SS_ERR_INVALID_ARG;
  ss_status st = check_device();
  if (st != SS_OK) return st;

  // lambda = 0 with skip masks or margins requested runs the voting kernel with a
  // threshold no tile passes (every tile kept, margins reported).
  const bool debug_out = dbg != nullptr && (dbg->skip_mask != nullptr || dbg->vote_margin != nullptr);
  const Mode mode =
      count_only ? Mode::kCount : ((dense && !debug_out) ? Mode::kDense : Mode::kSparse);
  // Which prefill kernel (both compute the one-pass definition):
  //  - the CTA-pair kernel (two-SM MMAs, one pass) for the dense and voting
  //    paths at d = 128 and for every mode at d_qk = 192 / d_v = 128;
  //  - the one-CTA kernel (two query blocks per CTA; decisions of a run of
  //    tiles first, kept tiles second) for counting (calibration) at d = 128
  //    and for every mode at d = 64.  Measured on GB300 (DiT 32K, Llama 16K
  //    causal, chunked 2K on 32K, 128K): at d = 128 the pair kernel is ahead
  //    from dense up to ~70% skipped tiles (by 10-20% at 50%), the one-CTA
  //    kernel ahead at ~90% (by ~25%), where its vote pass runs the score
  //    MMAs near the tensor peak.  At d = 64 (value tiles padded to 128
  //    columns in the pair kernel) the two tie dense, the pair kernel leads
  //    at 50% and the one-CTA kernel at 70% (DiT 32K: 6.46 against 5.97 ms).
  //    The kernel can be chosen explicitly through ss_debug_opts.
  bool pair = (d == 192) || (d == 128 && mode != Mode::kCount);
  // A shortened vote run (test only) exercises the one-CTA kernel's multi-run path.
  if (d != 192 && dbg != nullptr && dbg->vote_chunk_tiles != 0) pair = false;
  const int which = dbg != nullptr ? dbg->prefill_kernel : 0;
  if (which < 0 || which > 2) return SS_ERR_INVALID_ARG;
  if (which != 0) {
    if (which == 1 && d == 192) return SS_ERR_UNSUPPORTED;
    pair = (which == 2);
  }
  CUtensorMap tq, tk, tv;
  if (!make_map(&tq, q, d, Lq, static_cast<long>(B) * Hq) ||
      !make_map(&tk, k, d, Lk, static_cast<long>(B) * Hkv, pair ? kTile / 2 : kTile) ||
      !make_map(&tv, v, dv, Lk, static_cast<long>(B) * Hkv))
    return SS_ERR_CUDA;

  PrefillParams p{};
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.Lq = Lq;
  p.Lk = Lk;
  p.G = Hq / Hkv;
  p.nQB = static_cast<int>(nQB);
  p.nT = static_cast<int>(nT);
  p.causal = causal ? 1 : 0;
  p.chunk_tiles = kVoteChunkTiles;
  if (dbg != nullptr && dbg->vote_chunk_tiles != 0) {
    if (dbg->vote_chunk_tiles < 1 || dbg->vote_chunk_tiles > kVoteChunkTiles) return SS_ERR_INVALID_ARG;
    p.chunk_tiles = dbg->vote_chunk_tiles;
  }
  p.scale = scale;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.thr_raw = thr_raw;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.counts = counts;
  p.mask = dbg ? dbg->skip_mask : nullptr;
  p.margin = dbg ? dbg->vote_margin : nullptr;
  p.status = status_ptr();
  cudaError_t e = pair ? launch_prefill_pair(d, mode, tq, tk, tv, p, static_cast<cudaStream_t>(stream))
                       : launch_prefill(d, mode, tq, tk, tv, p, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SS_OK : SS_ERR_CUDA;
}

size_t decode_ws(int B, int Hq, int d, int S) {
  if (S <= 1 || B < 1 || Hq < 1 || d < 1) return 0;
  return static_cast<size_t>(B) * Hq * S * (d + 2) * sizeof(float);
}

ss_status decode_impl(const void* q, const void* k, const void* v, void* o, int B, int Hq, int Hkv,
                      int Lk, int d, float scale, bool dense, float thr_raw, int S,
                      uint32_t* counts, void* ws, size_t ws_bytes, const ss_debug_opts* dbg,
                      void* stream) {
  const bool count_only = dbg != nullptr && dbg->count_only != 0;
  if (q == nullptr || k == nullptr || v == nullptr || (o == nullptr && !count_only))
    return SS_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || (o != nullptr && !aligned16(o)))
    return SS_ERR_INVALID_ARG;
  if (B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || Lk < 1 || S < 1 || !scale_ok(scale))
    return SS_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return SS_ERR_UNSUPPORTED;
  // voting group: up to 32 rows (MMA N) with keys on the TMEM lanes, up to
  // 128 (MMA M) with the heads as rows at d = 128
  if (Hq / Hkv > (d == 128 ? kDecRowsMaxG : 32)) return SS_ERR_UNSUPPORTED;
  const long nT = ceil_div(Lk, kTile);
  const long ctas = static_cast<long>(B) * Hkv * S;
  if (ctas > 0x7fffffffL) return SS_ERR_INVALID_ARG;
  if (!count_only && S > 1) {
    if (ws == nullptr || !aligned16(ws) || ws_bytes < decode_ws(B, Hq, d, S)) return SS_ERR_WORKSPACE;
  }
  ss_status st = check_device();
  if (st != SS_OK) return st;
  CUtensorMap tk, tv;
  if (!make_map(&tk, k, d, Lk, static_cast<long>(B) * Hkv) ||
      !make_map(&tv, v, d, Lk, static_cast<long>(B) * Hkv))
    return SS_ERR_CUDA;

  DecodeParams p{};
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.Lk = Lk;
  p.d = d;
  p.G = Hq / Hkv;
  p.nT = static_cast<int>(nT);
  p.S = S;
  p.T = static_cast<int>(ceil_div(nT, S));
  p.scale = scale;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.thr_raw = thr_raw;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.o = static_cast<__nv_bfloat16*>(o);
  p.part = static_cast<float*>(ws);
  p.counts = counts;
  p.mask = dbg ? dbg->skip_mask : nullptr;
  p.margin = dbg ? dbg->vote_margin : nullptr;
  p.status = status_ptr();
  p.count_only = count_only ? 1 : 0;
  p.fault_inject = dbg ? dbg->fault_inject : 0;
  const Mode mode = count_only ? Mode::kCount : (dense ? Mode::kDense : Mode::kSparse);
  cudaError_t e = launch_decode(tk, tv, p, mode, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SS_OK : SS_ERR_CUDA;
}

// The latent-attention decode kernel for the number of heads.
cudaError_t launch_mla_any(const CUtensorMap& tkv, const MlaParams& p, Mode mode, cudaStream_t st) {
  if (p.Hq > kMlaWideHeads) return launch_mla_decode_rows(tkv, p, mode, st);
  return launch_mla_decode(tkv, p, mode, st);
}

size_t mla_ws(int B, int Hq, int d_latent, int S) {
  if (S <= 1 || B < 1 || Hq < 1 || d_latent < 1) return 0;
  return static_cast<size_t>(B) * Hq * S * (d_latent + 2) * sizeof(float);
}

ss_status mla_impl(const void* q, const void* kv, void* o, int B, int Hq, int Lk, int d_latent,
                   int d_rope, float scale, bool dense, float thr_raw, int S, uint32_t* counts,
                   void* ws, size_t ws_bytes, const ss_debug_opts* dbg, void* stream) {
  const bool count_only = dbg != nullptr && dbg->count_only != 0;
  if (q == nullptr || kv == nullptr || (o == nullptr && !count_only)) return SS_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kv) || (o != nullptr && !aligned16(o))) return SS_ERR_INVALID_ARG;
  if (B < 1 || Hq < 1 || Lk < 1 || S < 1 || !scale_ok(scale)) return SS_ERR_INVALID_ARG;
  if (d_latent != kMlaLatent || d_rope != kMlaRope || Hq > kMlaMaxHeads) return SS_ERR_UNSUPPORTED;
  const long nT = ceil_div(Lk, kTile);
  if (static_cast<long>(B) * S > 0x7fffffffL) return SS_ERR_INVALID_ARG;
  if (!count_only && S > 1) {
    if (ws == nullptr || !aligned16(ws) || ws_bytes < mla_ws(B, Hq, d_latent, S))
      return SS_ERR_WORKSPACE;
  }
  ss_status st = check_device();
  if (st != SS_OK) return st;
  // [B][Lk][576] viewed as B rows of Lk keys: 64 x 128 boxes, 128-byte swizzle.
  CUtensorMap tkv;
  if (!make_map(&tkv, kv, kMlaDk, Lk, B)) return SS_ERR_CUDA;

  MlaParams p{};
  p.B = B;
  p.Hq = Hq;
  p.Lk = Lk;
  p.nT = static_cast<int>(nT);
  p.S = S;
  p.T = static_cast<int>(ceil_div(nT, S));
  p.scale = scale;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.thr_raw = thr_raw;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.o = static_cast<__nv_bfloat16*>(o);
  p.part = static_cast<float*>(ws);
  p.counts = counts;
  p.mask = dbg ? dbg->skip_mask : nullptr;
  p.margin = dbg ? dbg->vote_margin : nullptr;
  p.status = status_ptr();
  const Mode mode = count_only ? Mode::kCount : (dense ? Mode::kDense : Mode::kSparse);
  cudaError_t e = launch_mla_any(tkv, p, mode, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SS_OK : SS_ERR_CUDA;
}

// Evaluated (unit, tile) pairs of a problem (tiles a causal row block never
// reaches are not evaluated).
long evaluated_tiles(const ss_problem& p) {
  const long nT = ceil_div(p.Lk, kTile);  // prefill kinds: SS_PREFILL, SS_MLA_PREFILL
  if (p.kind == SS_DECODE) return static_cast<long>(p.B) * p.Hkv * nT;
  if (p.kind == SS_MLA_DECODE) return static_cast<long>(p.B) * nT;
  const long nQB = ceil_div(p.Lq, kTile);
  long per_head = 0;
  for (long qb = 0; qb < nQB; ++qb) {
    if (!p.causal) {
      per_head += nT;
      continue;
    }
    const long rows = std::min<long>(kTile, p.Lq - qb * kTile);
    const long last = qb * kTile + rows - 1 + (static_cast<long>(p.Lk) - p.Lq);
    per_head += last < 0 ? 0 : std::min(nT, last / kTile + 1);
  }
  return per_head * p.B * p.Hq;
}

long counter_len(const ss_problem& p) {
  if (p.kind == SS_DECODE) return static_cast<long>(p.B) * p.Hkv * p.num_kv_splits;
  if (p.kind == SS_MLA_DECODE) return static_cast<long>(p.B) * p.num_kv_splits;
  return static_cast<long>(p.B) * p.Hq * ceil_div(p.Lq, kTile);
}

}  // namespace
}  // namespace ssattn

// Partial states of ss_attn_decode_noalloc: module memory of this library,
// present on every device that loads it, never allocated at run time.
static __device__ __align__(256) unsigned char g_decode_scratch[SS_DECODE_STATIC_SCRATCH_BYTES];

namespace ssattn {
namespace {

// Device address of g_decode_scratch on the current device.  Host code only
// holds a stand-in for the array, so the address is looked up once per
// device (with that device current) and cached.
void* decode_scratch_ptr() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return nullptr;
  static std::mutex mu;
  static std::vector<void*> ptrs;
  std::lock_guard<std::mutex> lock(mu);
  if (static_cast<int>(ptrs.size()) <= dev) ptrs.resize(dev + 1, nullptr);
  if (ptrs[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_decode_scratch) != cudaSuccess || ptr == nullptr)
      return nullptr;
    ptrs[dev] = ptr;
  }
  return ptrs[dev];
}

}  // namespace
}  // namespace ssattn

using namespace ssattn;

extern "C" {

ss_status ss_attn_prefill_ex(const void* q, const void* k, const void* v, void* o, int B, int Hq,
                             int Hkv, int Lq, int Lk, int d, float scale, int causal, float lambda,
                             uint32_t* skip_counts, const ss_debug_opts* dbg, void* stream) {
  if (!lambda_ok(lambda)) return SS_ERR_INVALID_ARG;
  const bool dense = lambda == 0.f;
  const float thr = dense ? -INFINITY : threshold_raw(std::log(static_cast<double>(lambda)), scale);
  return prefill_impl(q, k, v, o, B, Hq, Hkv, Lq, Lk, d, scale, causal, dense, thr, skip_counts,
                      dbg, stream);
}

ss_status ss_attn_prefill(const void* q, const void* k, const void* v, void* o, int B, int Hq,
                          int Hkv, int Lq, int Lk, int d, float scale, int causal, float lambda,
                          uint32_t* skip_counts, void* stream) {
  return ss_attn_prefill_ex(q, k, v, o, B, Hq, Hkv, Lq, Lk, d, scale, causal, lambda, skip_counts,
                            nullptr, stream);
}

ss_status ss_attn_mla_prefill_ex(const void* q, const void* k, const void* v, void* o, int B,
                                 int Hq, int Hkv, int Lq, int Lk, int d_qk, int d_v, float scale,
                                 int causal, float lambda, uint32_t* skip_counts,
                                 const ss_debug_opts* dbg, void* stream) {
  if (!lambda_ok(lambda)) return SS_ERR_INVALID_ARG;
  if (d_qk != 192 || d_v != 128) return SS_ERR_UNSUPPORTED;
  const bool dense = lambda == 0.f;
  const float thr = dense ? -INFINITY : threshold_raw(std::log(static_cast<double>(lambda)), scale);
  return prefill_impl(q, k, v, o, B, Hq, Hkv, Lq, Lk, d_qk, scale, causal, dense, thr,
                      skip_counts, dbg, stream, d_v);
}

ss_status ss_attn_mla_prefill(const void* q, const void* k, const void* v, void* o, int B, int Hq,
                              int Hkv, int Lq, int Lk, int d_qk, int d_v, float scale, int causal,
                              float lambda, uint32_t* skip_counts, void* stream) {
  return ss_attn_mla_prefill_ex(q, k, v, o, B, Hq, Hkv, Lq, Lk, d_qk, d_v, scale, causal, lambda,
                                skip_counts, nullptr, stream);
}

size_t ss_attn_decode_workspace_size(int B, int Hq, int d, int num_kv_splits) {
  return decode_ws(B, Hq, d, num_kv_splits);
}

ss_status ss_attn_decode_ex(const void* q, const void* k_cache, const void* v_cache, void* o,
                            int B, int Hq, int Hkv, int Lk, int d, float scale, float lambda,
                            int num_kv_splits, uint32_t* skip_counts, void* workspace,
                            size_t workspace_bytes, const ss_debug_opts* dbg, void* stream) {
  if (!lambda_ok(lambda)) return SS_ERR_INVALID_ARG;
  const bool dense = lambda == 0.f;
  const float thr = dense ? -INFINITY : threshold_raw(std::log(static_cast<double>(lambda)), scale);
  return decode_impl(q, k_cache, v_cache, o, B, Hq, Hkv, Lk, d, scale, dense, thr, num_kv_splits,
                     skip_counts, workspace, workspace_bytes, dbg, stream);
}

ss_status ss_attn_decode(const void* q, const void* k_cache, const void* v_cache, void* o, int B,
                         int Hq, int Hkv, int Lk, int d, float scale, float lambda,
                         int num_kv_splits, uint32_t* skip_counts, void* workspace,
                         size_t workspace_bytes, void* stream) {
  return ss_attn_decode_ex(q, k_cache, v_cache, o, B, Hq, Hkv, Lk, d, scale, lambda,
                           num_kv_splits, skip_counts, workspace, workspace_bytes, nullptr, stream);
}

ss_status ss_attn_mla_decode_paged(const void* q, const void* kv_pages, const int32_t* page_table,
                                   const int32_t* seq_lens, void* o, int B, int Hq, int num_pages,
                                   int max_pages, int d_latent, int d_rope, float scale,
                                   float lambda_a, int num_kv_splits, uint32_t* skip_counts,
                                   void* workspace, size_t workspace_bytes,
                                   const ss_debug_opts* dbg, void* stream) {
  const bool count_only = dbg != nullptr && dbg->count_only != 0;
  if (q == nullptr || kv_pages == nullptr || page_table == nullptr || seq_lens == nullptr ||
      (o == nullptr && !count_only))
    return SS_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kv_pages) || (o != nullptr && !aligned16(o)))
    return SS_ERR_INVALID_ARG;
  if (B < 1 || Hq < 1 || num_pages < 1 || max_pages < 1 || num_kv_splits < 1 || !scale_ok(scale) ||
      !(lambda_a >= 0.f) || !std::isfinite(lambda_a))
    return SS_ERR_INVALID_ARG;
  if (d_latent != kMlaLatent || d_rope != kMlaRope || Hq > kMlaMaxHeads) return SS_ERR_UNSUPPORTED;
  const int S = num_kv_splits;
  if (static_cast<long>(B) * S > 0x7fffffffL) return SS_ERR_INVALID_ARG;
  if (!count_only && S > 1) {
    if (workspace == nullptr || !aligned16(workspace) ||
        workspace_bytes < mla_ws(B, Hq, d_latent, S))
      return SS_ERR_WORKSPACE;
  }
  ss_status st = check_device();
  if (st != SS_OK) return st;
  // [num_pages][128][576]: page p is "row block" p of the map; a page index
  // outside the pool reads zeros (TMA out-of-bounds fill), never faults.
  CUtensorMap tkv;
  if (!make_map(&tkv, kv_pages, kMlaDk, kTile, num_pages)) return SS_ERR_CUDA;
  MlaParams p{};
  p.B = B;
  p.Hq = Hq;
  p.Lk = max_pages * kTile;
  p.nT = max_pages;
  p.S = S;
  p.T = static_cast<int>(ceil_div(max_pages, S));
  p.scale = scale;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.thr_raw = -INFINITY;  // per sequence from lambda_a (in the kernel)
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.o = static_cast<__nv_bfloat16*>(o);
  p.part = static_cast<float*>(workspace);
  p.counts = skip_counts;
  p.mask = dbg ? dbg->skip_mask : nullptr;
  p.margin = dbg ? dbg->vote_margin : nullptr;
  p.status = status_ptr();
  p.page_table = page_table;
  p.seq_lens = seq_lens;
  p.max_pages = max_pages;
  p.lambda_a = lambda_a;
  const Mode mode = count_only ? Mode::kCount : (lambda_a == 0.f ? Mode::kDense : Mode::kSparse);
  cudaError_t e = launch_mla_any(tkv, p, mode, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SS_OK : SS_ERR_CUDA;
}

size_t ss_attn_mla_decode_workspace_size(int B, int Hq, int d_latent, int num_kv_splits) {
  return mla_ws(B, Hq, d_latent, num_kv_splits);
}

ss_status ss_attn_mla_decode_ex(const void* q, const void* kv, void* o, int B, int Hq, int Lk,
                                int d_latent, int d_rope, float scale, float lambda,
                                int num_kv_splits, uint32_t* skip_counts, void* workspace,
                                size_t workspace_bytes, const ss_debug_opts* dbg, void* stream) {
  if (!lambda_ok(lambda)) return SS_ERR_INVALID_ARG;
  const bool dense = lambda == 0.f;
  const float thr = dense ? -INFINITY : threshold_raw(std::log(static_cast<double>(lambda)), scale);
  // Debug outputs need the vote: with lambda = 0 it runs with a threshold
  // no tile passes (every tile kept, margins reported).
  const bool debug_out = dbg != nullptr && (dbg->skip_mask != nullptr || dbg->vote_margin != nullptr);
  return mla_impl(q, kv, o, B, Hq, Lk, d_latent, d_rope, scale, dense && !debug_out, thr,
                  num_kv_splits, skip_counts, workspace, workspace_bytes, dbg, stream);
}

ss_status ss_attn_mla_decode(const void* q, const void* kv, void* o, int B, int Hq, int Lk,
                             int d_latent, int d_rope, float scale, float lambda,
                             int num_kv_splits, uint32_t* skip_counts, void* workspace,
                             size_t workspace_bytes, void* stream) {
  return ss_attn_mla_decode_ex(q, kv, o, B, Hq, Lk, d_latent, d_rope, scale, lambda,
                               num_kv_splits, skip_counts, workspace, workspace_bytes, nullptr,
                               stream);
}

ss_status ss_attn_decode_paged(const void* q, const void* k_pages, const void* v_pages,
                               const int32_t* page_table, const int32_t* seq_lens, void* o,
                               int B, int Hq, int Hkv, int num_pages, int max_pages, int d,
                               float scale, float lambda_a, int num_kv_splits,
                               uint32_t* skip_counts, void* workspace, size_t workspace_bytes,
                               const ss_debug_opts* dbg, void* stream) {
  const bool count_only = dbg != nullptr && dbg->count_only != 0;
  if (q == nullptr || k_pages == nullptr || v_pages == nullptr || page_table == nullptr ||
      seq_lens == nullptr || (o == nullptr && !count_only))
    return SS_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) ||
      (o != nullptr && !aligned16(o)))
    return SS_ERR_INVALID_ARG;
  if (B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv != 0 || num_pages < 1 || max_pages < 1 ||
      num_kv_splits < 1 || !scale_ok(scale) || !(lambda_a >= 0.f) || !std::isfinite(lambda_a))
    return SS_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return SS_ERR_UNSUPPORTED;
  if (Hq / Hkv > (d == 128 ? kDecRowsMaxG : 32)) return SS_ERR_UNSUPPORTED;
  const int S = num_kv_splits;
  if (static_cast<long>(B) * Hkv * S > 0x7fffffffL ||
      static_cast<long>(num_pages) * Hkv > 0x7fffffffL ||
      static_cast<long>(B) * max_pages > 0x7fffffffL || static_cast<long>(max_pages) * kTile > 0x7fffffffL)
    return SS_ERR_INVALID_ARG;
  if (!count_only && S > 1) {
    if (workspace == nullptr || !aligned16(workspace) || workspace_bytes < decode_ws(B, Hq, d, S))
      return SS_ERR_WORKSPACE;
  }
  ss_status st = check_device();
  if (st != SS_OK) return st;
  CUtensorMap tk, tv;
  const long pages_x_heads = static_cast<long>(num_pages) * Hkv;
  if (!make_map(&tk, k_pages, d, kTile, pages_x_heads) || !make_map(&tv, v_pages, d, kTile, pages_x_heads))
    return SS_ERR_CUDA;

  DecodeParams p{};
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.Lk = 0;  // per sequence
  p.d = d;
  p.G = Hq / Hkv;
  p.nT = max_pages;
  p.S = S;
  p.T = 0;
  p.scale = scale;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.thr_raw = -INFINITY;  // per sequence from lambda_a
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.o = static_cast<__nv_bfloat16*>(o);
  p.part = static_cast<float*>(workspace);
  p.counts = skip_counts;
  p.mask = dbg ? dbg->skip_mask : nullptr;
  p.margin = dbg ? dbg->vote_margin : nullptr;
  p.status = status_ptr();
  p.count_only = count_only ? 1 : 0;
  p.fault_inject = 0;
  p.page_table = page_table;
  p.seq_lens = seq_lens;
  p.max_pages = max_pages;
  p.lambda_a = lambda_a;
  const Mode mode = count_only ? Mode::kCount : (lambda_a == 0.f ? Mode::kDense : Mode::kSparse);
  cudaError_t e = launch_decode(tk, tv, p, mode, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SS_OK : SS_ERR_CUDA;
}

ss_status ss_attn_decode_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                 void* o, int B, int Hq, int Hkv, int Lk, int d, float scale,
                                 float lambda, int num_kv_splits, uint32_t* skip_counts,
                                 void* stream) {
  if (!lambda_ok(lambda)) return SS_ERR_INVALID_ARG;
  const size_t need = decode_ws(B, Hq, d, num_kv_splits);
  if (need > SS_DECODE_STATIC_SCRATCH_BYTES) return SS_ERR_WORKSPACE;
  void* ws = nullptr;
  if (need > 0 && (ws = decode_scratch_ptr()) == nullptr) return SS_ERR_CUDA;
  const bool dense = lambda == 0.f;
  const float thr = dense ? -INFINITY : threshold_raw(std::log(static_cast<double>(lambda)), scale);
  return decode_impl(q, k_cache, v_cache, o, B, Hq, Hkv, Lk, d, scale, dense, thr, num_kv_splits,
                     skip_counts, ws, SS_DECODE_STATIC_SCRATCH_BYTES, nullptr, stream);
}

size_t ss_decode_static_scratch_bytes(void) { return SS_DECODE_STATIC_SCRATCH_BYTES; }

ss_status ss_calibrate(const ss_problem* p, float target_sparsity, float* a_out,
                       float* achieved_out) {
  if (p == nullptr || a_out == nullptr || p->skip_counts == nullptr || !aligned16(p->q) ||
      !(target_sparsity >= 0.f && target_sparsity <= 1.f) || p->Lk < 1)
    return SS_ERR_INVALID_ARG;
  if (p->kind != SS_PREFILL && p->kind != SS_DECODE && p->kind != SS_MLA_DECODE &&
      p->kind != SS_MLA_PREFILL)
    return SS_ERR_INVALID_ARG;
  if (p->kind == SS_MLA_DECODE && (p->Hkv != 1 || p->d != kMlaDk)) return SS_ERR_UNSUPPORTED;
  if (p->kind == SS_MLA_PREFILL && p->d != 192) return SS_ERR_UNSUPPORTED;
  const long N = evaluated_tiles(*p);
  const long ncnt = counter_len(*p);
  if (N <= 0 || ncnt <= 0) return SS_ERR_INVALID_ARG;
  const long k = static_cast<long>(std::floor(static_cast<double>(target_sparsity) * N + 0.5));
  const double lnL = std::log(static_cast<double>(p->Lk));
  cudaStream_t stream = static_cast<cudaStream_t>(p->stream);
  std::vector<uint32_t> host(ncnt);
  ss_debug_opts dbg{};
  dbg.count_only = 1;
  dbg.fault_inject = (p->kind == SS_DECODE) ? p->fault_inject : 0;

  // Skipped tiles at lambda = exp(ln_lambda), from one count-only launch.
  auto count_at = [&](double ln_lambda, long* out) -> ss_status {
    const float thr = threshold_raw(ln_lambda, p->scale);
    ss_status st;
    if (p->kind == SS_PREFILL || p->kind == SS_MLA_PREFILL)
      st = prefill_impl(p->q, p->k, p->v, nullptr, p->B, p->Hq, p->Hkv, p->Lq, p->Lk, p->d,
                        p->scale, p->causal, false, thr, p->skip_counts, &dbg, p->stream,
                        p->kind == SS_MLA_PREFILL ? 128 : 0);
    else if (p->kind == SS_MLA_DECODE)
      st = mla_impl(p->q, p->k, nullptr, p->B, p->Hq, p->Lk, kMlaLatent, kMlaRope, p->scale,
                    false, thr, p->num_kv_splits, p->skip_counts, nullptr, 0, &dbg, p->stream);
    else
      st = decode_impl(p->q, p->k, p->v, nullptr, p->B, p->Hq, p->Hkv, p->Lk, p->d, p->scale,
                       false, thr, p->num_kv_splits, p->skip_counts, nullptr, 0, &dbg, p->stream);
    if (st != SS_OK) return st;
    if (cudaMemcpyAsync(host.data(), p->skip_counts, ncnt * sizeof(uint32_t),
                        cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess)
      return SS_ERR_CUDA;
    // Counters of a launch that gave up a bounded wait are not trustworthy:
    // read (and clear) the device status word before using them.
    uint32_t dev_status = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&dev_status, g_device_status, sizeof dev_status) != cudaSuccess)
      return SS_ERR_CUDA;
    if (dev_status != 0) {
      if (cudaMemcpyToSymbol(g_device_status, &zero, sizeof zero) != cudaSuccess)
        return SS_ERR_CUDA;
      if (dev_status & kDevStatusTimeout) return SS_ERR_TIMEOUT;
    }
    long s = 0;
    for (uint32_t c : host) s += c;
    *out = s;
    return SS_OK;
  };

  if (k == 0) {
    *a_out = 0.f;
    if (achieved_out) *achieved_out = 0.f;
    return SS_OK;
  }
  // x = ln a = ln lambda + ln L; count(x) is non-decreasing in x.
  const double x_hi = lnL;  // lambda = 1
  long c_hi = 0;
  ss_status st = count_at(x_hi - lnL, &c_hi);
  if (st != SS_OK) return st;
  if (c_hi < k) {  // not reachable with lambda <= 1: the closest is lambda = 1
    *a_out = static_cast<float>(p->Lk);
    if (achieved_out) *achieved_out = static_cast<float>(static_cast<double>(c_hi) / N);
    return SS_OK;
  }
  double x_lo = lnL - 64.0;
  long c_lo = 0;
  for (int i = 0; i < 8; ++i) {
    if ((st = count_at(x_lo - lnL, &c_lo)) != SS_OK) return st;
    if (c_lo < k) break;
    x_lo -= 64.0;
  }
  if (c_lo >= k) return SS_ERR_INVALID_ARG;  // degenerate scores

  // Smallest x with count(x) >= target, by bisection on [lo, hi].
  auto first_reaching = [&](long target, double lo, double hi, double* out) -> ss_status {
    for (int it = 0; it < 48 && hi - lo > 1e-7 * std::max(1.0, std::fabs(hi)); ++it) {
      const double mid = 0.5 * (lo + hi);
      long c = 0;
      ss_status s2 = count_at(mid - lnL, &c);
      if (s2 != SS_OK) return s2;
      (c >= target ? hi : lo) = mid;
    }
    *out = hi;
    return SS_OK;
  };
  double x1 = x_hi, x2 = x_hi;
  if ((st = first_reaching(k, x_lo, x_hi, &x1)) != SS_OK) return st;
  if (c_hi >= k + 1) {
    if ((st = first_reaching(k + 1, x1, x_hi, &x2)) != SS_OK) return st;
  }
  // Middle of [x1, x2): the widest margin on both sides of the k-th tile.
  double a = std::exp(0.5 * (x1 + x2));
  a = std::min(a, static_cast<double>(p->Lk));
  *a_out = static_cast<float>(a);
  if (achieved_out) {
    const double lam = std::min(1.0, static_cast<double>(*a_out) / p->Lk);
    long c = 0;
    if ((st = count_at(std::log(static_cast<double>(static_cast<float>(lam))), &c)) != SS_OK)
      return st;
    *achieved_out = static_cast<float>(static_cast<double>(c) / N);
  }
  return SS_OK;
}

ss_status ss_fit_factor(const float* s, const float* a, int n, float* A_out, float* B_out) {
  if (s == nullptr || a == nullptr || A_out == nullptr || B_out == nullptr || n < 2)
    return SS_ERR_INVALID_ARG;
  double sx = 0, sy = 0, sxx = 0, sxy = 0;
  for (int i = 0; i < n; ++i) {
    if (!(a[i] > 0.f) || !std::isfinite(s[i])) return SS_ERR_INVALID_ARG;
    const double x = s[i], y = std::log(static_cast<double>(a[i]));
    sx += x;
    sy += y;
    sxx += x * x;
    sxy += x * y;
  }
  const double den = n * sxx - sx * sx;
  if (!(std::fabs(den) > 0.0)) return SS_ERR_INVALID_ARG;
  const double slope = (n * sxy - sx * sy) / den;
  const double icpt = (sy - slope * sx) / n;
  *A_out = static_cast<float>(std::exp(icpt));
  *B_out = static_cast<float>(slope);
  return SS_OK;
}

float ss_lambda(float A, float B, float s, int L) {
  if (L < 1) return 0.f;
  return static_cast<float>(static_cast<double>(A) * std::exp(static_cast<double>(B) * s) / L);
}

const char* ss_status_string(ss_status st) {
  switch (st) {
    case SS_OK: return "ok";
    case SS_ERR_INVALID_ARG: return "invalid argument";
    case SS_ERR_UNSUPPORTED: return "unsupported configuration or device";
    case SS_ERR_CUDA: return "CUDA runtime error";
    case SS_ERR_TIMEOUT: return "a kernel gave up a bounded wait";
    case SS_ERR_WORKSPACE: return "decode workspace missing or too small";
  }
  return "unknown status";
}

ss_status ss_stream_status(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return SS_ERR_CUDA;
  uint32_t v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_status, sizeof v) != cudaSuccess) return SS_ERR_CUDA;
  if (v != 0 && cudaMemcpyToSymbol(g_device_status, &zero, sizeof zero) != cudaSuccess)
    return SS_ERR_CUDA;
  return (v & kDevStatusTimeout) ? SS_ERR_TIMEOUT : SS_OK;
}

}  // extern "C"
