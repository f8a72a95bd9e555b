// Skip-softmax (BLASST) split-KV decode for sm_103a with the vote group's
// query heads as the rows of the MMAs: GQA / MQA groups of 17..128 heads on
// one KV head, d = 128.
//
// Method (BLASST summary, §Methodologie and §Kernel-ontwerp; "Skip-Softmax"
// design doc, §The skip test): every K tile of a split is streamed; a tile is
// skipped when every query head of the group passes exp(scale * (tile_max -
// m)) < lambda against its exact running maximum m, and then its V tile is
// never loaded; splits are merged by log-sum-exp.
//
// One CTA = (sequence b, KV head, split).  Per tile j:
//   S_j = Q K_j^T: M = 128 rows (the G heads, zero rows past them), N = 128
//   keys, K = d, both operands K-major from shared memory, into one of three
//   TMEM score buffers (so score MMAs run up to three tiles ahead);
//   softmax warps 0-3, thread = TMEM lane = head: the row's 128 scores in two
//   halves of 64, its maximum, the vote (one bar.red.and over the 128
//   threads), P = exp2((S - m_ref) * scale * log2e) as bf16 over the first
//   32 columns of each half (the P.V MMA's A operand, from TMEM);
//   the V tile of a kept tile is requested right after the vote (dense:
//   every tile, in order, without waiting for a vote), and
//   O += P_j V_j (M = 128, N = d, K = 128 keys; V MN-major) accumulates in
//   TMEM across tiles.
// m_ref trails the exact maximum lazily (moved only when the maximum has grown
// by more than 2^8 in exp2 units; the warp then has the P.V issuer drain the
// P.V MMAs issued so far, rescales its rows of O and l, and signals back).
// Compared with the kernel that puts keys on the TMEM lanes, the per-head
// state sits in one thread (no cross-thread row reductions, no register fold
// of a fresh accumulator per tile), so the tile's work does not grow with the
// group beyond the exponentials.
//
// Roles (256 threads, 8 warps):
//   warps 0-3  softmax / vote, one thread per head (a warp with no head only
//              meets the barriers);
//   warp 4     barrier setup, TMA producer of the K ring;
//   warp 5     TMA producer of the V ring;
//   warp 6     TMEM allocation, issuer of the score MMAs;
//   warp 7     issuer of the P.V MMAs (the whole warp zeroes the rows of a
//              partial page past the sequence end).
#include <cuda_bf16.h>

#include "decode_rows.cuh"
#include "ptx_sm103.cuh"

namespace ssattn {

namespace {

constexpr int kRDThreads = 256;
constexpr int kRDWarpK = 4, kRDWarpV = 5, kRDWarpS = 6, kRDWarpPV = 7;
constexpr int kRDD = 128;  // head width
constexpr int kRDNB = 3;   // score buffers
constexpr float kRDRescaleLog2 = 8.0f;
constexpr uint32_t kRDFlagKept = 1u, kRDFlagRescale = 2u;

struct RDCfg {
  static constexpr int NK = 3;   // K ring slots
  static constexpr int NV = 3;   // V ring slots
  static constexpr int NVQ = 4;  // kept-tile queue entries
  static constexpr int kTileBytes = kTile * kRDD * 2;  // one K or V tile: two 64-column boxes
  static constexpr int kQBytes = kTile * kRDD * 2;     // 128 rows x d
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + kQBytes;
  static constexpr int kVOff = kKOff + NK * kTileBytes;
  static constexpr int kCtlOff = kVOff + NV * kTileBytes;
  static constexpr int kCtlBytes = 1024;
  static constexpr int kSmemBytes = kCtlOff + kCtlBytes + 1024;  // + alignment slack
  static constexpr uint32_t kColO = 128u * kRDNB;                // O: columns 384 .. 511
  static constexpr uint32_t kTmemCols = 512;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
};

struct RDCtl {
  uint64_t k_full[RDCfg::NK], k_empty[RDCfg::NK];
  uint64_t v_full[RDCfg::NV], v_empty[RDCfg::NV];
  uint64_t vq_full[RDCfg::NVQ], vq_empty[RDCfg::NVQ];
  uint64_t s_full[kRDNB];  // scores of the buffer's tile are in TMEM
  uint64_t s_free[kRDNB];  // the buffer's P.V is issued (or not needed)
  uint64_t dec[kRDNB];     // the 4 softmax warps have decided the buffer's tile
  uint64_t drain[4];       // per softmax warp: the P.V MMAs issued so far are done
  uint64_t rescaled[4];    // per softmax warp: its rows of O are rescaled
  uint64_t o_full;         // the last P.V is done
  uint64_t mma_done[2];    // teardown, per issuer
  alignas(16) uint32_t flags[kRDNB][4];  // per buffer and softmax warp: kept | rescale
  int kq[RDCfg::NVQ];      // kept tiles for the V producer (-1: no more)
  uint32_t tmem_base;
  int abort_flag;
  float red[4];
};

template <Mode MODE>
__global__ void __launch_bounds__(kRDThreads, 1)
    decode_rows_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                       const DecodeParams p) {
  using C = RDCfg;
  constexpr int NK = C::NK, NV = C::NV, NVQ = C::NVQ;
  constexpr bool kPV = (MODE != Mode::kCount);
  constexpr bool kVote = (MODE != Mode::kDense);
  constexpr bool kDenseV = (MODE == Mode::kDense);  // every tile kept: V needs no decision
  static_assert(sizeof(RDCtl) <= C::kCtlBytes, "control block overflow");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem + C::kQOff;
  uint8_t* sK = smem + C::kKOff;
  uint8_t* sV = smem + C::kVOff;
  auto* ctl = reinterpret_cast<RDCtl*>(smem + C::kCtlOff);
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
  int n_k = 0;  // K copies issued (teardown bookkeeping)
  auto issue_k = [&](int t) {
    const int st = t % NK;
    if (p.fault_inject == 1 && t == 1) return;  // test only: this copy never comes
    mbar_arrive_expect_tx(&ctl->k_full[st], C::kTileBytes);
    tma_load_3d(sK + st * C::kTileBytes, &tmK, &ctl->k_full[st], 0, tile_y(t), tile_z(t));
    tma_load_3d(sK + st * C::kTileBytes + 16384, &tmK, &ctl->k_full[st], 64, tile_y(t), tile_z(t));
    n_k = t + 1;
  };
  if (warp == kRDWarpK && lane == 0) {
    for (int s = 0; s < NK; ++s) {
      mbar_init(&ctl->k_full[s], 1);
      mbar_init(&ctl->k_empty[s], 1);
    }
    for (int s = 0; s < NV; ++s) {
      mbar_init(&ctl->v_full[s], 1);
      mbar_init(&ctl->v_empty[s], 1);
    }
    for (int s = 0; s < NVQ; ++s) {
      mbar_init(&ctl->vq_full[s], 1);
      mbar_init(&ctl->vq_empty[s], 1);
    }
    for (int s = 0; s < kRDNB; ++s) {
      mbar_init(&ctl->s_full[s], 1);
      mbar_init(&ctl->s_free[s], 1);
      mbar_init(&ctl->dec[s], 4);
    }
    for (int w = 0; w < 4; ++w) {
      mbar_init(&ctl->drain[w], 1);
      mbar_init(&ctl->rescaled[w], 1);
    }
    mbar_init(&ctl->o_full, 1);
    mbar_init(&ctl->mma_done[0], 1);
    mbar_init(&ctl->mma_done[1], 1);
    ctl->abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    for (int t = 0; t < min(nt, NK); ++t) issue_k(t);
  }
  if (warp == kRDWarpS) {
    tmem_alloc(&ctl->tmem_base, C::kTmemCols);
    tmem_relinquish();
  }
  if (warp < 4) {
    // Queries as the score MMA's A operand: 128 rows x d, K-major, two
    // 64-column chunks, 128-byte swizzle; rows >= G are zero.
    constexpr int kGran = kRDD / 8;
    for (int idx = tid; idx < kTile * kGran; idx += 128) {
      const int g = idx / kGran, e8 = idx - (idx / kGran) * kGran;
      uint4 val = make_uint4(0u, 0u, 0u, 0u);
      if (g < G)
        val = *reinterpret_cast<const uint4*>(
            p.q + (static_cast<size_t>(b) * p.Hq + static_cast<size_t>(kvh) * G + g) * kRDD + e8 * 8);
      *reinterpret_cast<uint4*>(sQ + (e8 >> 3) * (kTile * 128) + g * 128 +
                                (((e8 & 7) ^ (g & 7)) << 4)) = val;
    }
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;

  if (warp == kRDWarpK) {
    // ------------------------------------------------------------ K producer
    if (lane == 0)
      for (int t = NK; t < nt; ++t) {
        if (!mbar_wait(&ctl->k_empty[t % NK], ((t / NK) & 1) ^ 1, abort_flag)) break;
        issue_k(t);
      }
    if (lane == 0 && *abort_flag) {
      // Let the copies in flight land before shared memory is released.
      for (int s = 0; s < NK; ++s)
        if (n_k > s && !(p.fault_inject == 1 && s == 1))
          mbar_wait(&ctl->k_full[s], ((((n_k - 1 - s) / NK) * NK + s) / NK) & 1, nullptr);
    }
    __syncwarp();
  } else if (warp == kRDWarpV) {
    // ------------------------------------------------------------ V producer
    int n_v = 0;
    if (kPV && lane == 0 && nt > 0) {
      for (int i = 0;; ++i) {
        int t = i;
        if (!kDenseV) {
          const int s = i % NVQ;
          if (!mbar_wait(&ctl->vq_full[s], (i / NVQ) & 1, abort_flag)) break;
          t = *reinterpret_cast<volatile int*>(&ctl->kq[s]);
          mbar_arrive(&ctl->vq_empty[s]);
        }
        if (t < 0 || t >= nt) break;
        const int vs = i % NV;
        if (!mbar_wait(&ctl->v_empty[vs], ((i / NV) & 1) ^ 1, abort_flag)) break;
        mbar_arrive_expect_tx(&ctl->v_full[vs], C::kTileBytes);
        tma_load_3d(sV + vs * C::kTileBytes, &tmV, &ctl->v_full[vs], 0, tile_y(t), tile_z(t));
        tma_load_3d(sV + vs * C::kTileBytes + 16384, &tmV, &ctl->v_full[vs], 64, tile_y(t),
                    tile_z(t));
        n_v = i + 1;
      }
    }
    if (lane == 0 && *abort_flag)
      for (int s = 0; s < NV; ++s)
        if (n_v > s) mbar_wait(&ctl->v_full[s], ((((n_v - 1 - s) / NV) * NV + s) / NV) & 1, nullptr);
    __syncwarp();
  } else if (warp == kRDWarpS) {
    // ------------------------------------------------------------ score MMAs
    if (lane == 0 && nt > 0) {
      constexpr uint32_t idS = idesc_bf16_f32(128, 128, false, false);
      const uint64_t dq = smem_desc(smem_u32(sQ), 16, 1024);
      const uint32_t sKa = smem_u32(sK);
      for (int t = 0; t < nt; ++t) {
        const int sb = t % kRDNB, st = t % NK;
        // The buffer's previous tile was decided and its P.V issued (P lives
        // in the score buffer): the P.V issuer's fence + barrier order this
        // MMA after it.
        if (t >= kRDNB && !mbar_wait(&ctl->s_free[sb], ((t / kRDNB) - 1) & 1, abort_flag)) break;
        if (!mbar_wait(&ctl->k_full[st], (t / NK) & 1, abort_flag)) break;
        tc_fence_after();
        const uint64_t dk = smem_desc(sKa + st * C::kTileBytes, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < kRDD / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * (kTile * 128) + (kk & 3) * 32) >> 4;
          mma_bf16_ss(tmem + 128u * sb, dq + off, dk + off, idS, kk > 0 ? 1u : 0u);
        }
        mma_commit(&ctl->k_empty[st]);
        mma_commit(&ctl->s_full[sb]);
      }
      mma_commit(&ctl->mma_done[0]);
      mbar_wait(&ctl->mma_done[0], 0, nullptr);  // all MMAs done before TMEM is freed
    }
    __syncwarp();
  } else if (warp == kRDWarpPV) {
    // ------------------------------------------------------------ P.V MMAs
    if (nt > 0) {
      constexpr uint32_t idO = idesc_bf16_f32(128, kRDD, false, true);
      const uint32_t sVa = smem_u32(sV);
      bool fine = true;
      uint32_t o_acc = 0u, nresc = 0u;
      int nk = 0;  // V tiles consumed (kept tiles; every tile when dense)
      for (int t = 0; t < nt && fine; ++t) {
        const int sb = t % kRDNB;
        if (!__all_sync(0xffffffffu, mbar_wait(&ctl->dec[sb], (t / kRDNB) & 1, abort_flag))) break;
        const uint4 f4 = *reinterpret_cast<const uint4*>(ctl->flags[sb]);
        const uint32_t f[4] = {f4.x, f4.y, f4.z, f4.w};
        const bool kept = (f[0] & kRDFlagKept) != 0;
        uint32_t resc = 0u;
#pragma unroll
        for (int w = 0; w < 4; ++w) resc |= ((f[w] >> 1) & 1u) << w;
        if (kPV && resc) {
          // Warps that move their reference maximum rescale their rows of O
          // once every P.V issued so far has finished.
          if (lane == 0)
            for (int w = 0; w < 4; ++w)
              if (resc & (1u << w)) mma_commit(&ctl->drain[w]);
          for (int w = 0; w < 4 && fine; ++w)
            if (resc & (1u << w)) {
              fine = __all_sync(0xffffffffu,
                                mbar_wait(&ctl->rescaled[w], (nresc >> w) & 1u, abort_flag));
              nresc ^= 1u << w;
            }
          if (!fine) break;
        }
        if (kPV && kept) {
          const int vs = nk % NV;
          if (!__all_sync(0xffffffffu, mbar_wait(&ctl->v_full[vs], (nk / NV) & 1, abort_flag))) {
            fine = false;
            break;
          }
          const int rows = tile_rows(t);
          if (paged && rows < kTile) {
            // Rows of a page past the sequence end hold whatever the cache
            // holds: zero them so that P = 0 there cannot meet a non-finite value.
            uint4* base = reinterpret_cast<uint4*>(sV + vs * C::kTileBytes);
            for (int idx = rows * 8 + lane; idx < kTile * 8; idx += 32) {
              base[idx] = make_uint4(0u, 0u, 0u, 0u);
              base[1024 + idx] = make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();
          }
          __syncwarp();
          if (lane == 0) {
            tc_fence_after();
            const uint64_t dv = smem_desc(sVa + vs * C::kTileBytes, 16384, 1024);
#pragma unroll
            for (int kk = 0; kk < kTile / 16; ++kk)  // P of keys 16kk..: column 64 (kk / 4) + 8 (kk % 4)
              mma_bf16_ts(tmem + C::kColO, tmem + 128u * sb + 64 * (kk >> 2) + 8 * (kk & 3),
                          dv + ((kk * 2048) >> 4), idO, (o_acc | kk) ? 1u : 0u);
            mma_commit(&ctl->v_empty[vs]);
          }
          __syncwarp();
          o_acc = 1u;
          ++nk;
        }
        if (lane == 0) {
          tc_fence_before();
          mbar_arrive(&ctl->s_free[sb]);
        }
        __syncwarp();
      }
      if (lane == 0) {
        if (kPV && fine) mma_commit(&ctl->o_full);
        mma_commit(&ctl->mma_done[1]);
        mbar_wait(&ctl->mma_done[1], 0, nullptr);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ vote / softmax
    // Thread = head row = TMEM lane.  After a failed wait a thread carries on
    // to the end of the loop (every later wait gives up at once), so all 128
    // threads take the same sequence of barriers.  The tcgen05 loads and
    // stores are warp-collective (.sync.aligned): a warp with any head runs
    // them on all 32 lanes, and rows past the last head are masked instead.
    const int row = tid;
    const bool active = row < G;
    const bool warp_active = warp * 32 < G;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const uint32_t colO = lane_base + C::kColO;
    const float sl2 = p.scale_log2;
    float m_true = -INFINITY, m_ref = -INFINITY, l = 0.f;
    uint32_t skipped = 0, n_drain = 0;
    int n_vq = 0;  // kept tiles pushed to the V producer (thread 0)
    bool ok = true;
    auto wwait = [&](uint64_t* bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag));
    };
    // Scores of keys 64 hf .. + 63, masked past the tile's last key, into
    // sr; returns their maximum.
    auto load_half = [&](uint32_t colS, int hf, int rows_t, uint32_t* sr) -> float {
      tmem_ld32p(colS + 64 * hf, sr);
      tmem_ld32p(colS + 64 * hf + 32, sr + 32);
      tmem_wait_ld();
      const int vis = rows_t - 1 - 64 * hf;  // last visible key of the half
      if (vis < 63) {
#pragma unroll
        for (int e = 0; e < 64; ++e)
          if (e > vis) sr[e] = __float_as_uint(-INFINITY);
      }
      float mx[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) mx[e] = -INFINITY;
#pragma unroll
      for (int e = 0; e < 32; ++e)
        mx[e & 3] = fmax3(mx[e & 3], __uint_as_float(sr[2 * e]), __uint_as_float(sr[2 * e + 1]));
      return fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
    };
    // P of the 64 scores in sr as bf16 pairs into sr[0..31]; returns their sum.
    auto exp_half = [&](uint32_t* sr) -> float {
      const float mb = (m_ref == -INFINITY) ? 0.f : m_ref * sl2;
      const uint64_t sl2x2 = f32x2(sl2, sl2), nmb = f32x2(-mb, -mb);
      uint64_t ls[2] = {0ull, 0ull};
#pragma unroll
      for (int cc = 0; cc < 32; ++cc) {
        const uint64_t xp = fma_f32x2(
            f32x2(__uint_as_float(sr[2 * cc]), __uint_as_float(sr[2 * cc + 1])), sl2x2, nmb);
        const float p0 = ex2_approx(f32x2_lo(xp));
        const float p1 = ex2_approx(f32x2_hi(xp));
        ls[cc & 1] = add_f32x2(ls[cc & 1], f32x2(p0, p1));
        sr[cc] = pack_bf16x2(p0, p1);
      }
      const uint64_t lsum = add_f32x2(ls[0], ls[1]);
      return f32x2_lo(lsum) + f32x2_hi(lsum);
    };

    for (int t = 0; t < nt; ++t) {
      const int sb = t % kRDNB;
      const uint32_t colS = lane_base + 128u * sb;
      if (!wwait(&ctl->s_full[sb], (t / kRDNB) & 1)) ok = false;
      tc_fence_after();
      const int rows_t = tile_rows(t);
      uint32_t sr[64];
      float tmax = -INFINITY;
      if (warp_active) {
        tmax = load_half(colS, 0, rows_t, sr);
        asm volatile("" : "+f"(tmax));  // one half of the scores in registers at a time
        tmax = fmaxf(tmax, load_half(colS, 1, rows_t, sr));  // sr keeps the second half
        if (!active) tmax = -INFINITY;  // no head on this row: never votes, never moves m
      }
      // Skip vote: every head must pass exp(scale*(tile_max - m)) < lambda.
      float c = -INFINITY;
      if (tmax != -INFINITY) c = (m_true == -INFINITY) ? INFINITY : tmax - m_true;
      bool kept = true;
      if constexpr (kVote) kept = !named_bar_and(1, 128, c < thr_raw);
      // Debug outputs (also on the dense path): the largest statistic over
      // the group, and the decision.
      if (p.margin != nullptr) {
        float cm = c;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, o));
        if (lane == 0) *reinterpret_cast<volatile float*>(&ctl->red[warp]) = cm;
        named_bar_sync(1, 128);
        if (tid == 0) {
          const volatile float* rr = ctl->red;
          const float cmax = fmaxf(fmaxf(rr[0], rr[1]), fmaxf(rr[2], rr[3]));
          p.margin[static_cast<long>(bk) * row_stride + j0 + t] =
              (cmax == INFINITY) ? INFINITY : cmax * p.scale;
        }
        named_bar_sync(1, 128);  // red[] is read before the next tile writes it
      }
      if (tid == 0) {
        skipped += kept ? 0u : 1u;
        if (p.mask != nullptr) p.mask[static_cast<long>(bk) * row_stride + j0 + t] = kept ? 0 : 1;
      }
      m_true = fmaxf(m_true, tmax);
      bool resc = false;
      float alpha = 1.f;
      if (kPV && kept) {
        if (!kDenseV && tid == 0) {
          // The V tile of this tile may be fetched now.
          const int s = n_vq % NVQ;
          if (!mbar_wait(&ctl->vq_empty[s], ((n_vq / NVQ) & 1) ^ 1, abort_flag)) ok = false;
          ctl->kq[s] = t;
          mbar_arrive(&ctl->vq_full[s]);
          ++n_vq;
        }
        bool need = false;
        if (m_ref == -INFINITY) {
          m_ref = m_true;  // no key of this row counted yet: its O row and l are zero
        } else if ((m_true - m_ref) * sl2 > kRDRescaleLog2) {
          need = true;
        }
        resc = __any_sync(0xffffffffu, need);
        if (resc && m_ref != -INFINITY) {
          alpha = ex2_approx((m_ref - m_true) * sl2);
          l *= alpha;
          m_ref = m_true;
        }
        // P as bf16 pairs over the first 32 columns of each half: the
        // second half from the registers, then the first half loaded again.
        // (A row past the last head writes values nobody reads.)
        if (warp_active) {
          float ls = exp_half(sr);
          tmem_st32p(colS + 64, sr);
          load_half(colS, 0, rows_t, sr);
          ls += exp_half(sr);
          tmem_st32p(colS, sr);
          l += ls;
          tmem_wait_st();
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        ctl->flags[sb][warp] = (kept ? kRDFlagKept : 0u) | (resc ? kRDFlagRescale : 0u);
        mbar_arrive(&ctl->dec[sb]);
      }
      if (kPV && resc) {
        // The P.V issuer drains the P.V MMAs issued so far; then this warp's
        // rows of O are rescaled before this tile's P.V.
        if (!wwait(&ctl->drain[warp], n_drain & 1)) ok = false;
        ++n_drain;
        if (__all_sync(0xffffffffu, ok)) {
          tc_fence_after();
#pragma unroll 1
          for (int cc = 0; cc < kRDD / 32; ++cc) {
            uint32_t orr[32];
            tmem_ld32p(colO + cc * 32, orr);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) orr[e] = __float_as_uint(__uint_as_float(orr[e]) * alpha);
            tmem_st32p(colO + cc * 32, orr);
          }
          tmem_wait_st();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->rescaled[warp]);
      }
    }

    if (kPV && !kDenseV && tid == 0) {
      // End of the kept stream for the V producer.
      const int s = n_vq % NVQ;
      if (!mbar_wait(&ctl->vq_empty[s], ((n_vq / NVQ) & 1) ^ 1, abort_flag)) ok = false;
      ctl->kq[s] = -1;
      mbar_arrive(&ctl->vq_full[s]);
    }
    ok = !named_bar_or(1, 128, !ok);
    if (kPV && ok && nt > 0) {
      ok = wwait(&ctl->o_full, 0);
      tc_fence_after();
    }
    if (kPV && ok && warp_active) {  // (ok is the same on all 128 threads here)
      const size_t hrow = static_cast<size_t>(b) * p.Hq + static_cast<size_t>(kvh) * G +
                          static_cast<size_t>(min(row, G - 1));
      if (p.S == 1) {
        // O / l -> bf16 (a head that saw no key writes zeros).
        const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
        __nv_bfloat16* orow = p.o + hrow * kRDD;
#pragma unroll 1
        for (int cc = 0; cc < kRDD / 32; ++cc) {
          uint32_t orr[32];
          if (nt > 0) {
            tmem_ld32p(colO + cc * 32, orr);
            tmem_wait_ld();
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) orr[e] = 0u;
          }
          uint32_t w[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            w[e] = pack_bf16x2(__uint_as_float(orr[2 * e]) * inv_l,
                               __uint_as_float(orr[2 * e + 1]) * inv_l);
          if (active) {
            uint4* dst = reinterpret_cast<uint4*>(orow + cc * 32);
#pragma unroll
            for (int e = 0; e < 4; ++e)
              dst[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
          }
        }
      } else {
        // Partial state of this split: O against m_ref, m_ref * scale * log2e, l.
        // (a partial row is d + 2 floats: 8-byte aligned, not 16)
        float* pr = p.part + (hrow * p.S + split) * (kRDD + 2);
#pragma unroll 1
        for (int cc = 0; cc < kRDD / 32; ++cc) {
          uint32_t orr[32];
          if (nt > 0) {
            tmem_ld32p(colO + cc * 32, orr);
            tmem_wait_ld();
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) orr[e] = 0u;
          }
          if (active) {
            float2* dst = reinterpret_cast<float2*>(pr + cc * 32);
#pragma unroll
            for (int e = 0; e < 16; ++e)
              dst[e] = make_float2(__uint_as_float(orr[2 * e]), __uint_as_float(orr[2 * e + 1]));
          }
        }
        if (active) {
          pr[kRDD] = (m_ref == -INFINITY) ? -INFINITY : m_ref * sl2;
          pr[kRDD + 1] = l;
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
  __syncthreads();
  if (warp == kRDWarpS) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  if (tid == 0 && *abort_flag) report_timeout(p.status);
}

template <Mode MODE>
cudaError_t launch_rows(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p,
                        cudaStream_t st) {
  auto* fn = decode_rows_kernel<MODE>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       RDCfg::kSmemBytes);
  if (e != cudaSuccess) return e;
  const long ctas = static_cast<long>(p.B) * p.Hkv * p.S;
  fn<<<dim3(static_cast<unsigned>(ctas)), dim3(kRDThreads), RDCfg::kSmemBytes, st>>>(tk, tv, p);
  e = cudaGetLastError();
  if (e != cudaSuccess || MODE == Mode::kCount || p.S == 1) return e;
  return launch_decode_merge(p, st);
}

}  // namespace

cudaError_t launch_decode_rows(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p,
                               Mode mode, cudaStream_t st) {
  switch (mode) {
    case Mode::kDense: return launch_rows<Mode::kDense>(tk, tv, p, st);
    case Mode::kSparse: return launch_rows<Mode::kSparse>(tk, tv, p, st);
    default: return launch_rows<Mode::kCount>(tk, tv, p, st);
  }
}

}  // namespace ssattn
