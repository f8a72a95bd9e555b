// Skip-softmax (BLASST) split-KV decode forward for sm_103a, plus the
// log-sum-exp merge of the splits.
//
// Method (BLASST summary, §Methodologie and §Kernel-ontwerp; "Skip-Softmax"
// design doc, §The skip test): decode is bound by HBM traffic.  Every K tile
// of a split is streamed (the scores decide the skip), but a skipped tile's
// V block is never loaded; the V tiles of kept tiles are fetched as soon as
// the vote has decided, while the following K tiles keep streaming.
//
// One CTA = one (sequence b, KV head, split); WG softmax warpgroups (one for
// vote groups of up to 16 query rows, two above) and four role warps:
//   warps 0-3  vote / softmax: thread i = TMEM lane i, which is key i of the
//              tile for the scores and dimension i for the P.V result.  With
//              two warpgroups, warps 0-3 keep rows 0-15 and warps 4-7 rows
//              16-31, and each tile's vote takes two exchanges: the warp
//              maxima of the rows, then each warpgroup's vote statistic.
//   warp 4*WG  TMA producer of the K ring (NK stages, 128-byte swizzle).
//   +1         TMA producer of the V slots (kept tiles only, in kept order).
//   +2         TMEM allocator + issuer of the score MMAs
//              S^T = K_tile . Q^T  (M = 128 keys, N = 16/32 query rows
//              padded with zero rows, K = d), fp32 in TMEM.
//   +3         issuer of the value MMAs  O_i^T = V_i^T . P_i^T
//              (M = 128 = d, N = query rows, K = 128 keys), one fresh TMEM
//              accumulator per kept tile.
// The G query heads that share the KV head (one token each) are the voting
// group: a tile is skipped only if every one of them passes the test.  The
// contraction has only G rows, but putting it on the tensor cores takes it
// off the issue slots, which bound the CUDA-core version of this kernel.
//
// Online softmax: the vote and the exponentials use the exact running
// maximum m.  P_i = exp2((s - m_i) * scale * log2e) with m_i the maximum after
// kept tile i; each thread (dimension) folds the kept tiles' P.V results into
// registers in kept order, acc = acc * exp2(m_prev - m_i) + O_i, and keeps a
// per-key partial row sum l rescaled the same way.
#include <cuda_bf16.h>

#include "common.cuh"
#include "decode_rows.cuh"
#include "ptx_sm103.cuh"

namespace ssattn {

namespace {

// Softmax warpgroups for a vote group padded to GP rows: one thread keeps the
// state of GP / WG rows (with one warpgroup, 32 rows would sit at the
// register cap and spill).
template <int GP>
constexpr int kDecWG = (GP > 16) ? 2 : 1;
template <int GP>
constexpr int kDecThreads = 128 * kDecWG<GP> + 128;

template <int D, int GP>
struct DecCfg {
  static constexpr int NQ = (GP <= 16) ? 16 : 32;  // MMA N (rows padded with zeros)
  static constexpr int NK = (D == 128) ? 4 : 8;    // K ring stages
  static constexpr int NV = (D == 128 || GP > 16) ? 2 : 4;  // V / P / O slots
  static constexpr int NS = 4;                      // score buffers in TMEM
  static constexpr int kChunks = D / 64;            // 128-byte swizzle chunks per row
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kQBytes = NQ * D * 2;
  static constexpr int kPBytes = NQ * kTile * 2;
  // V slots first: for d = 64 the value MMA (M = 128) reads a second,
  // unused 64-row atom 16 KB past its slot, which must stay inside the block.
  static constexpr int kVOff = 0;
  static constexpr int kKOff = kVOff + NV * kTileBytes;
  static constexpr int kQOff = kKOff + NK * kTileBytes;
  static constexpr int kPOff = kQOff + kQBytes;
  static constexpr int kRedOff = kPOff + NV * kPBytes;            // float [2][GP][4]
  static constexpr int kLRedOff = kRedOff + 2 * GP * 4 * 4;       // float [GP][4]
  static constexpr int kMsOff = kLRedOff + GP * 4 * 4;            // float [2 NV][GP]
  static constexpr int kPartOff = kMsOff + 2 * NV * GP * 4;       // float [2][2]
  static constexpr int kCtlOff = (kPartOff + 16 + 15) / 16 * 16;
  static constexpr int kCtlBytes = 512;
  static constexpr int kSmemBytes = kCtlOff + kCtlBytes + 1024;  // + alignment slack
  static constexpr uint32_t kColS = 0;              // S buffer b at kColS + NQ b
  static constexpr uint32_t kColO = NS * NQ;        // O slot s at kColO + NQ s
  static constexpr uint32_t kTmemCols = ((NS + NV) * NQ <= 128) ? 128 : 256;
  static_assert((NS + NV) * NQ <= kTmemCols, "TMEM columns");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
  static_assert(D != 64 || NV * kTileBytes + 16384 <= kKOff + NK * kTileBytes, "d=64 atom");
};

template <int NK, int NV, int NS>
struct DecCtl {
  uint64_t k_full[NK], k_empty[NK];
  uint64_t s_full[NS], s_empty[NS];
  uint64_t v_full[NV], slot_free[NV], vq_full[NV], p_full[NV];
  uint64_t s_done, pv_done;
  int kq[NV];    // kept tile for the V producer (-1: no more)
  int prec[NV];  // 1: P written, 0: no more (value-MMA issuer)
  uint32_t tmem_base;
  int abort_flag;
};

// tcgen05.ld of N consecutive fp32 columns of the warp's 32 lanes.
template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float (&r)[N]);
template <>
__device__ __forceinline__ void tmem_ld_cols<1>(uint32_t taddr, float (&r)[1]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=f"(r[0]) : "r"(taddr));
}
template <>
__device__ __forceinline__ void tmem_ld_cols<2>(uint32_t taddr, float (&r)[2]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x2.b32 {%0, %1}, [%2];"
               : "=f"(r[0]), "=f"(r[1])
               : "r"(taddr));
}
template <>
__device__ __forceinline__ void tmem_ld_cols<4>(uint32_t taddr, float (&r)[4]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
               : "=f"(r[0]), "=f"(r[1]), "=f"(r[2]), "=f"(r[3])
               : "r"(taddr));
}
template <>
__device__ __forceinline__ void tmem_ld_cols<8>(uint32_t taddr, float (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=f"(r[0]), "=f"(r[1]), "=f"(r[2]), "=f"(r[3]), "=f"(r[4]), "=f"(r[5]),
                 "=f"(r[6]), "=f"(r[7])
               : "r"(taddr));
}
template <>
__device__ __forceinline__ void tmem_ld_cols<16>(uint32_t taddr, float (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=f"(r[0]), "=f"(r[1]), "=f"(r[2]), "=f"(r[3]), "=f"(r[4]), "=f"(r[5]), "=f"(r[6]),
        "=f"(r[7]), "=f"(r[8]), "=f"(r[9]), "=f"(r[10]), "=f"(r[11]), "=f"(r[12]), "=f"(r[13]),
        "=f"(r[14]), "=f"(r[15])
      : "r"(taddr));
}

// Maximum over the warp (every lane gets it).
__device__ __forceinline__ float warp_max(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}

template <int D, int GP, Mode MODE>
__global__ void __launch_bounds__(kDecThreads<GP>, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const DecodeParams p) {
  using C = DecCfg<D, GP>;
  constexpr int NK = C::NK, NV = C::NV, NS = C::NS, NQ = C::NQ;
  constexpr int WG = kDecWG<GP>, HG = GP / WG;  // softmax warpgroups, rows per warpgroup
  constexpr int kWarpK = 4 * WG, kWarpV = kWarpK + 1, kWarpS = kWarpK + 2;  // +3: value MMAs
  constexpr bool kPV = (MODE != Mode::kCount);
  constexpr bool kVote = (MODE != Mode::kDense);
  constexpr bool kDenseV = (MODE == Mode::kDense);  // every tile kept: V needs no decision
  using Ctl = DecCtl<NK, NV, NS>;
  static_assert(sizeof(Ctl) <= C::kCtlBytes, "control block overflow");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sV = smem + C::kVOff;
  uint8_t* sK = smem + C::kKOff;
  uint8_t* sQ = smem + C::kQOff;
  uint8_t* sP = smem + C::kPOff;
  float* sRed = reinterpret_cast<float*>(smem + C::kRedOff);
  float* sLRed = reinterpret_cast<float*>(smem + C::kLRedOff);
  float* sMs = reinterpret_cast<float*>(smem + C::kMsOff);
  float* sPart = reinterpret_cast<float*>(smem + C::kPartOff);
  auto* ctl = reinterpret_cast<Ctl*>(smem + C::kCtlOff);
  volatile int* abort_flag = &ctl->abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = p.G;
  const int split = blockIdx.x % p.S;
  const int bk = blockIdx.x / p.S;  // b * Hkv + kvh
  const int b = bk / p.Hkv, kvh = bk - (bk / p.Hkv) * p.Hkv;
  // Sequence geometry: one length for the batch, or per sequence (paged).
  const bool paged = p.page_table != nullptr;
  int len = p.Lk, nT_b = p.nT, T_b = p.T, row_stride = p.nT;
  float thr_raw = p.thr_raw;
  if (paged) {
    len = max(0, min(p.seq_lens[b], p.max_pages * kTile));
    nT_b = (len + kTile - 1) / kTile;
    T_b = (nT_b + p.S - 1) / p.S;
    row_stride = p.max_pages;
    // lambda_b = min(1, a / L_b) ("Skip-Softmax" §The threshold); a = 0: dense
    thr_raw = (p.lambda_a > 0.f && len > 0)
                  ? logf(fminf(1.f, p.lambda_a / static_cast<float>(len))) / p.scale
                  : -INFINITY;
  }
  const int j0 = split * T_b;
  const int nt = max(0, min(nT_b, j0 + T_b) - j0);
  auto tile_rows = [&](int t) { return min(kTile, len - (j0 + t) * kTile); };
  // Tensor-map coordinates (row, outer) of the split's tile t.
  auto tile_y = [&](int t) { return paged ? 0 : (j0 + t) * kTile; };
  auto tile_z = [&](int t) {
    return paged ? p.page_table[static_cast<long>(b) * p.max_pages + j0 + t] * p.Hkv + kvh : bk;
  };

  // ------------------------------------------------------------------ setup
  int n_k_issued = 0;  // K producer bookkeeping (teardown)
  auto issue_k = [&](int t) {
    const int st = t % NK;
    if (p.fault_inject == 1 && t == 1) return;  // test only: this copy never comes
    mbar_arrive_expect_tx(&ctl->k_full[st], C::kTileBytes);
#pragma unroll
    for (int c = 0; c < C::kChunks; ++c)
      tma_load_3d(sK + st * C::kTileBytes + c * 16384, &tmK, &ctl->k_full[st], c * 64,
                  tile_y(t), tile_z(t));
    n_k_issued = t + 1;
  };
  if (warp == kWarpK && lane == 0) {
    for (int s = 0; s < NK; ++s) {
      mbar_init(&ctl->k_full[s], 1);
      mbar_init(&ctl->k_empty[s], 1);
    }
    for (int s = 0; s < NS; ++s) {
      mbar_init(&ctl->s_full[s], 1);
      mbar_init(&ctl->s_empty[s], 4 * WG);
    }
    for (int s = 0; s < NV; ++s) {
      mbar_init(&ctl->v_full[s], 1);
      mbar_init(&ctl->slot_free[s], 1);
      mbar_init(&ctl->vq_full[s], 1);
      mbar_init(&ctl->p_full[s], 4 * WG);
    }
    mbar_init(&ctl->s_done, 1);
    mbar_init(&ctl->pv_done, 1);
    ctl->abort_flag = 0;
    fence_mbar_init();
    // The first K tiles go out before anything else is set up.
    tma_prefetch_desc(&tmK);
    for (int t = 0; t < min(nt, NK); ++t) issue_k(t);
  }
  if (warp == kWarpS) {
    tmem_alloc(&ctl->tmem_base, C::kTmemCols);
    tmem_relinquish();
  }
  if (warp < 4) {
    // Q of the voting group as the score MMA's B operand: NQ rows x D,
    // K-major, 128-byte swizzle (16-byte granule j of row g lands at
    // j ^ (g & 7)); rows >= G are zero.  P slots: zero, so that their rows
    // >= G stay zero for good.
    for (int idx = tid; idx < NQ * (D / 8); idx += 128) {
      const int g = idx / (D / 8), e8 = idx - (idx / (D / 8)) * (D / 8);
      uint4 val = make_uint4(0u, 0u, 0u, 0u);
      if (g < G)
        val = *reinterpret_cast<const uint4*>(
            p.q + (static_cast<size_t>(b) * p.Hq + kvh * G + g) * D + e8 * 8);
      *reinterpret_cast<uint4*>(sQ + (e8 >> 3) * NQ * 128 + g * 128 + (((e8 & 7) ^ (g & 7)) << 4)) =
          val;
    }
    if (kPV)
      for (int idx = tid; idx < NV * C::kPBytes / 16; idx += 128)
        reinterpret_cast<uint4*>(sP)[idx] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;

  if (warp >= 4 * WG) {
    int n_v_issued = 0;
    if (warp == kWarpK) {
      // ---------------------------------------------------------- K producer
      if (lane == 0) {
        for (int t = NK; t < nt; ++t) {
          if (!mbar_wait(&ctl->k_empty[t % NK], ((t / NK) & 1) ^ 1, abort_flag)) break;
          issue_k(t);
        }
      }
    } else if (warp == kWarpV) {
      // ---------------------------------------------------------- V producer
      if (kPV && lane == 0 && nt > 0) {
        tma_prefetch_desc(&tmV);
        for (int i = 0; i < nt; ++i) {
          const int s = i % NV;
          int t = i;
          if (!kDenseV) {
            if (!mbar_wait(&ctl->vq_full[s], (i / NV) & 1, abort_flag)) break;
            t = *reinterpret_cast<volatile int*>(&ctl->kq[s]);
            if (t < 0) break;
          }
          if (!mbar_wait(&ctl->slot_free[s], ((i / NV) & 1) ^ 1, abort_flag)) break;
          mbar_arrive_expect_tx(&ctl->v_full[s], C::kTileBytes);
#pragma unroll
          for (int c = 0; c < C::kChunks; ++c)
            tma_load_3d(sV + s * C::kTileBytes + c * 16384, &tmV, &ctl->v_full[s], c * 64,
                        tile_y(t), tile_z(t));
          n_v_issued = i + 1;
        }
      }
    } else if (warp == kWarpS) {
      // ---------------------------------------------------------- score MMAs
      if (lane == 0 && nt > 0) {
        constexpr uint32_t idS = idesc_bf16_f32(128, NQ, false, false);
        const uint64_t dq = smem_desc(smem_u32(sQ), 16, 1024);
        const uint32_t sKa = smem_u32(sK);
        for (int t = 0; t < nt; ++t) {
          const int st = t % NK, sb = t % NS;
          if (!mbar_wait(&ctl->k_full[st], (t / NK) & 1, abort_flag)) break;
          if (!mbar_wait(&ctl->s_empty[sb], ((t / NS) & 1) ^ 1, abort_flag)) break;
          tc_fence_after();
          const uint64_t dk = smem_desc(sKa + st * C::kTileBytes, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t ka = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
            const uint32_t qa = ((kk >> 2) * NQ * 128 + (kk & 3) * 32) >> 4;
            mma_bf16_ss(tmem + C::kColS + NQ * sb, dk + ka, dq + qa, idS, kk > 0 ? 1u : 0u);
          }
          mma_commit(&ctl->s_full[sb]);
          mma_commit(&ctl->k_empty[st]);
        }
        mma_commit(&ctl->s_done);
        mbar_wait(&ctl->s_done, 0, nullptr);  // all score MMAs done before TMEM is freed
      }
    } else {
      // ---------------------------------------------------------- value MMAs
      if (kPV && lane == 0 && nt > 0) {
        constexpr uint32_t idO = idesc_bf16_f32(128, NQ, true, false);
        const uint32_t sVa = smem_u32(sV), sPa = smem_u32(sP);
        for (int i = 0;; ++i) {
          const int s = i % NV;
          if (!mbar_wait(&ctl->p_full[s], (i / NV) & 1, abort_flag)) break;
          if (*reinterpret_cast<volatile int*>(&ctl->prec[s]) == 0) break;
          if (!mbar_wait(&ctl->v_full[s], (i / NV) & 1, abort_flag)) break;
          tc_fence_after();
          const uint64_t dv = smem_desc(sVa + s * C::kTileBytes, 16384, 1024);
          const uint64_t dp = smem_desc(sPa + s * C::kPBytes, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < kTile / 16; ++kk) {
            const uint32_t va = (kk * 2048) >> 4;
            const uint32_t pa = ((kk >> 2) * NQ * 128 + (kk & 3) * 32) >> 4;
            mma_bf16_ss(tmem + C::kColO + NQ * s, dv + va, dp + pa, idO, kk > 0 ? 1u : 0u);
          }
          mma_commit(&ctl->slot_free[s]);
        }
        mma_commit(&ctl->pv_done);
        mbar_wait(&ctl->pv_done, 0, nullptr);
      }
    }
    if (lane == 0 && *abort_flag) {
      // Let in-flight copies land before shared memory is released: the
      // newest copy into stage s is the largest index < n with index % N == s.
      // (With the test-only missing copy, stage 1 never received one.)
      if (warp == kWarpK)
        for (int s = 0; s < NK; ++s)
          if (n_k_issued > s && !(p.fault_inject == 1 && s == 1))
            mbar_wait(&ctl->k_full[s], ((s + ((n_k_issued - 1 - s) / NK) * NK) / NK) & 1, nullptr);
      if (warp == kWarpV)
        for (int s = 0; s < NV; ++s)
          if (n_v_issued > s)
            mbar_wait(&ctl->v_full[s], ((s + ((n_v_issued - 1 - s) / NV) * NV) / NV) & 1, nullptr);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ vote / softmax
    const int wg = warp >> 2;   // softmax warpgroup: rows hg .. hg + HG - 1
    const int hg = HG * wg;
    const int wq = warp & 3;    // warp within the warpgroup
    const int key = tid & 127;  // TMEM lane: key of the tile (scores), dimension (P.V)
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(wq * 32) << 16) + hg;
    constexpr int kSoftmaxThreads = 128 * WG;
    const float sl2 = p.scale_log2;
    auto wwait = [&](uint64_t* bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag));
    };
    float m[HG], l[HG], acc[HG], macc[HG];
#pragma unroll
    for (int g = 0; g < HG; ++g) {
      m[g] = -INFINITY;
      l[g] = 0.f;
      acc[g] = 0.f;
      macc[g] = -INFINITY;
    }
    uint32_t skipped = 0;
    int kept = 0;
    bool ok = true;

    // Fold the P.V result of kept tile j (slot j % NV) into acc (own rows).
    auto accumulate = [&](int j) {
      float o[HG];
      tmem_ld_cols<HG>(lane_base + C::kColO + NQ * (j % NV), o);
      tmem_wait_ld();
      const float* ms = sMs + (j % (2 * NV)) * GP + hg;
#pragma unroll
      for (int g = 0; g < HG; ++g) {
        const float mj = ms[g];
        const float f = (macc[g] == -INFINITY) ? 0.f : ex2_approx((macc[g] - mj) * sl2);
        acc[g] = fmaf(acc[g], f, o[g]);
        macc[g] = mj;
      }
    };

    for (int t = 0; t < nt; ++t) {
      const int sb = t % NS;
      const bool got = wwait(&ctl->s_full[sb], (t / NS) & 1);
      ok = ok && got;
      tc_fence_after();
      float s[HG];
      if (got) {
        tmem_ld_cols<HG>(lane_base + C::kColS + NQ * sb, s);
        tmem_wait_ld();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->s_empty[sb]);
      const bool valid_key = got && key < tile_rows(t);
#pragma unroll
      for (int g = 0; g < HG; ++g)
        if (!valid_key) s[g] = -INFINITY;

      // Tile maximum of each row: warp maxima, exchanged through shared
      // memory at one barrier of the softmax threads per tile (double-
      // buffered by tile parity, so a warp that runs ahead cannot overwrite
      // unread values).
      float mine = -INFINITY;
#pragma unroll
      for (int g = 0; g < HG; ++g) {
        const float wm = warp_max(s[g]);
        if (lane == g) mine = wm;
      }
      if (lane < HG) sRed[((t & 1) * GP + hg + lane) * 4 + wq] = mine;
      named_bar_sync(1, kSoftmaxThreads);
      float tm[HG];
#pragma unroll
      for (int g = 0; g < HG; ++g) {
        const float4 r = *reinterpret_cast<const float4*>(sRed + ((t & 1) * GP + hg + g) * 4);
        tm[g] = fmaxf(fmaxf(r.x, r.y), fmaxf(r.z, r.w));
      }

      // Vote: skip iff every row r has tile_max_r - m_r < ln(lambda)/scale;
      // with two warpgroups, each one's statistic over its rows, then the
      // maximum of both (second barrier).
      float cval = -INFINITY;
#pragma unroll
      for (int g = 0; g < HG; ++g)
        if (hg + g < G && tm[g] != -INFINITY)
          cval = fmaxf(cval, (m[g] == -INFINITY) ? INFINITY : tm[g] - m[g]);
      if constexpr (WG == 2) {
        if (key == 0) sPart[(t & 1) * 2 + wg] = cval;
        named_bar_sync(1, kSoftmaxThreads);
        cval = fmaxf(sPart[(t & 1) * 2], sPart[(t & 1) * 2 + 1]);
      }
      const bool skip = kVote && cval < thr_raw;
      if (tid == 0) {
        const long gi = static_cast<long>(bk) * row_stride + j0 + t;
        if (p.mask != nullptr) p.mask[gi] = skip ? 1 : 0;
        if (p.margin != nullptr) p.margin[gi] = (cval == INFINITY) ? INFINITY : cval * p.scale;
        skipped += skip ? 1u : 0u;
      }
      if (skip) continue;  // skipped tiles never raise m (lambda <= 1)

      float mn[HG];
#pragma unroll
      for (int g = 0; g < HG; ++g) mn[g] = fmaxf(m[g], tm[g]);
      if (kPV) {
        const int sl = kept % NV;
        // The slot's previous tile (kept - NV) must be through its P.V MMA
        // before its V, P and O space is reused.
        if (kept >= NV) ok = wwait(&ctl->slot_free[sl], ((kept / NV) - 1) & 1) && ok;
        if (!kDenseV && tid == 0) {
          ctl->kq[sl] = t;
          mbar_arrive(&ctl->vq_full[sl]);
        }
        if (kept >= NV) {
          tc_fence_after();
          accumulate(kept - NV);
        }
        // P for this tile as the value MMA's B operand: NQ rows x 128 keys,
        // K-major, 128-byte swizzle; this thread writes column `key` of its
        // warpgroup's rows.
        uint8_t* ps = sP + sl * C::kPBytes + (key >> 6) * NQ * 128 + (key & 7) * 2;
        const int j8 = (key & 63) >> 3;
#pragma unroll
        for (int g = 0; g < HG; ++g) {
          const float alpha = (m[g] == -INFINITY) ? 0.f : ex2_approx((m[g] - mn[g]) * sl2);
          const float mb = (mn[g] == -INFINITY) ? 0.f : mn[g] * sl2;
          const float pv = ex2_approx(fmaf(s[g], sl2, -mb));
          l[g] = fmaf(l[g], alpha, pv);
          const int row = hg + g;
          if (row < G)
            *reinterpret_cast<__nv_bfloat16*>(ps + row * 128 + ((j8 ^ (row & 7)) << 4)) =
                __float2bfloat16_rn(pv);
        }
        if (paged && tile_rows(t) < kTile) {
          // A page's rows past the sequence end hold whatever the cache
          // holds (TMA fills only rows outside the tensor map with zeros):
          // zero them so that P = 0 there cannot meet a non-finite V.
          ok = wwait(&ctl->v_full[sl], (kept / NV) & 1) && ok;
          if (wg == 0 && key >= tile_rows(t)) {
#pragma unroll
            for (int c = 0; c < C::kChunks; ++c) {
              uint4* row = reinterpret_cast<uint4*>(sV + sl * C::kTileBytes + c * 16384 + key * 128);
#pragma unroll
              for (int e = 0; e < 8; ++e) row[e] = make_uint4(0u, 0u, 0u, 0u);
            }
          }
        }
        float mine_m = 0.f;
#pragma unroll
        for (int g = 0; g < HG; ++g)
          if (key == g) mine_m = mn[g];
        if (key < HG) sMs[(kept % (2 * NV)) * GP + hg + key] = mine_m;
        if (tid == 0) ctl->prec[sl] = 1;
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->p_full[sl]);
        ++kept;
      }
#pragma unroll
      for (int g = 0; g < HG; ++g) m[g] = mn[g];
    }

    if (kPV) {
      // End of the kept stream for the V producer and the value-MMA issuer.
      const int sl = kept % NV;
      if (kept >= NV) ok = wwait(&ctl->slot_free[sl], ((kept / NV) - 1) & 1) && ok;
      if (tid == 0) {
        if (!kDenseV) {
          ctl->kq[sl] = -1;
          mbar_arrive(&ctl->vq_full[sl]);
        }
        ctl->prec[sl] = 0;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->p_full[sl]);
      named_bar_sync(1, kSoftmaxThreads);  // the last tile's maxima (sMs) are visible
      for (int j = max(0, kept - NV); j < kept; ++j) {
        ok = wwait(&ctl->slot_free[j % NV], (j / NV) & 1) && ok;
        tc_fence_after();
        accumulate(j);
      }
      // Row sums: per-key partials over the warpgroup's 128 threads.
#pragma unroll
      for (int g = 0; g < HG; ++g) {
        float v = l[g];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) sLRed[(hg + g) * 4 + wq] = v;
      }
      named_bar_sync(1, kSoftmaxThreads);
      if (ok && !*abort_flag && key < D) {
        const int e = key;
#pragma unroll
        for (int g = 0; g < HG; ++g) {
          if (hg + g >= G) break;
          const float4 r = *reinterpret_cast<const float4*>(sLRed + (hg + g) * 4);
          const float lt = (r.x + r.y) + (r.z + r.w);
          const size_t row = static_cast<size_t>(b) * p.Hq + kvh * G + hg + g;
          if (p.S == 1) {
            p.o[row * D + e] = __float2bfloat16_rn(lt > 0.f ? acc[g] / lt : 0.f);
          } else {
            float* pr = p.part + (row * p.S + split) * (D + 2);
            pr[e] = acc[g];
            if (e == 0) {
              pr[D] = (m[g] == -INFINITY) ? -INFINITY : m[g] * sl2;
              pr[D + 1] = lt;
            }
          }
        }
      }
    }
    if (tid == 0 && p.counts != nullptr) p.counts[static_cast<long>(bk) * p.S + split] = skipped;
    if (paged && split == 0 && tid < 32)
      for (int j = nT_b + tid; j < p.max_pages; j += 32) {
        const long gi = static_cast<long>(bk) * row_stride + j;
        if (p.mask != nullptr) p.mask[gi] = 2;
        if (p.margin != nullptr) p.margin[gi] = NAN;
      }
    tc_fence_before();
    __syncwarp();
  }

  // ------------------------------------------------------------------ teardown
  barrier_sync(2, kDecThreads<GP>);
  if (warp == kWarpS) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  if (tid == 0 && *abort_flag) report_timeout(p.status);
}

// Log-sum-exp merge of the per-split partial states: one warp per (b, h_q).
template <int D>
__global__ void __launch_bounds__(256) decode_merge_kernel(const float* __restrict__ part,
                                                           __nv_bfloat16* __restrict__ o, int rows,
                                                           int S) {
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const float* pr = part + static_cast<size_t>(row) * S * (D + 2);
  float mstar = -INFINITY;
  for (int s = 0; s < S; ++s) {
    const float l = pr[s * (D + 2) + D + 1];
    if (l > 0.f) mstar = fmaxf(mstar, pr[s * (D + 2) + D]);
  }
  constexpr int E = D / 32;
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  float L = 0.f;
  for (int s = 0; s < S; ++s) {
    const float l = pr[s * (D + 2) + D + 1];
    if (!(l > 0.f)) continue;
    const float w = ex2_approx(pr[s * (D + 2) + D] - mstar);
    L = fmaf(l, w, L);
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = fmaf(pr[s * (D + 2) + lane + 32 * e], w, acc[e]);
  }
  const float inv = (L > 0.f) ? 1.f / L : 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) o[static_cast<size_t>(row) * D + lane + 32 * e] = __float2bfloat16_rn(acc[e] * inv);
}

template <int D, int GP, Mode MODE>
cudaError_t launch_dec(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p,
                       cudaStream_t st) {
  using C = DecCfg<D, GP>;
  auto* fn = decode_kernel<D, GP, MODE>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  const long ctas = static_cast<long>(p.B) * p.Hkv * p.S;
  fn<<<dim3(static_cast<unsigned>(ctas)), dim3(kDecThreads<GP>), C::kSmemBytes, st>>>(tk, tv, p);
  e = cudaGetLastError();
  if (e != cudaSuccess || MODE == Mode::kCount || p.S == 1) return e;
  const int rows = p.B * p.Hq;
  decode_merge_kernel<D><<<dim3((rows + 7) / 8), dim3(256), 0, st>>>(p.part, p.o, rows, p.S);
  return cudaGetLastError();
}

template <int D, int GP>
cudaError_t launch_dec_mode(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p,
                            Mode mode, cudaStream_t st) {
  switch (mode) {
    case Mode::kDense: return launch_dec<D, GP, Mode::kDense>(tk, tv, p, st);
    case Mode::kSparse: return launch_dec<D, GP, Mode::kSparse>(tk, tv, p, st);
    default: return launch_dec<D, GP, Mode::kCount>(tk, tv, p, st);
  }
}

template <int D>
cudaError_t launch_dec_g(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p,
                         Mode mode, cudaStream_t st) {
  if (p.G <= 1) return launch_dec_mode<D, 1>(tk, tv, p, mode, st);
  if (p.G <= 2) return launch_dec_mode<D, 2>(tk, tv, p, mode, st);
  if (p.G <= 4) return launch_dec_mode<D, 4>(tk, tv, p, mode, st);
  if (p.G <= 8) return launch_dec_mode<D, 8>(tk, tv, p, mode, st);
  if (p.G <= 16) return launch_dec_mode<D, 16>(tk, tv, p, mode, st);
  return launch_dec_mode<D, 32>(tk, tv, p, mode, st);
}

}  // namespace

cudaError_t launch_decode(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p,
                          Mode mode, cudaStream_t st) {
  if (p.d == 128 && p.G > kDecKeyLayoutMaxG) return launch_decode_rows(tk, tv, p, mode, st);
  return (p.d == 128) ? launch_dec_g<128>(tk, tv, p, mode, st)
                      : launch_dec_g<64>(tk, tv, p, mode, st);
}

cudaError_t launch_decode_merge(const DecodeParams& p, cudaStream_t st) {
  const int rows = p.B * p.Hq;
  if (p.d == 128)
    decode_merge_kernel<128><<<dim3((rows + 7) / 8), dim3(256), 0, st>>>(p.part, p.o, rows, p.S);
  else
    decode_merge_kernel<64><<<dim3((rows + 7) / 8), dim3(256), 0, st>>>(p.part, p.o, rows, p.S);
  return cudaGetLastError();
}

}  // namespace ssattn
