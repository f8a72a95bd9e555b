// Latent-attention (MLA) skip-softmax decode on sm_103a with the query heads
// as the rows of the MMAs: up to 64 heads, the 512 latent entries of O split
// over two CTAs.
//
// Method (BLASST summary, §Methodologie and §Kernel-ontwerp; the MLA reading
// of §Belangrijkste Bijdragen item 4): per sequence one latent head shared by
// all query heads (rows of 512 latent + 64 rotary entries); the keys are the
// whole rows, the values their latent part.  A 128-key tile is skipped when
// every query head passes exp(scale * (tile_max - m)) < lambda against its
// exact running maximum m; splits of the tiles are merged by log-sum-exp.
//
// One CTA = (sequence b, split, latent half h): it computes the scores of
// all heads and O[:, 256 h .. 256 h + 255].  The two halves take the same
// decisions (same scores, same arithmetic); half 0 writes the counters and
// debug outputs.  Per tile j:
//   S_j = Q K_j^T: M = 128 rows (the heads; see the note on rows 64..127
//   below), N = 128 keys, K = 576, both operands K-major from shared memory,
//   into one of two TMEM score buffers;
//   softmax warps 0-3, thread = TMEM lane = head: the row's 128 scores in two
//   halves of 64, its maximum, the vote (one bar.red.and over the 128
//   threads), P = exp2((S - m_ref) * scale * log2e) as bf16 over the first
//   32 columns of each half (the P.V MMA's A operand, from TMEM);
//   O[:, half] += P_j V_j (M = 128, N = 128 per 128-entry value block, K =
//   128 keys; V MN-major) for kept tiles, O accumulated in TMEM across tiles.
// m_ref, the maximum P is referenced to, trails the exact maximum lazily: a
// row moves it only when the exact maximum has grown by more than 2^8 in
// exp2 units; its warp then asks the P.V issuer to drain the P.V MMAs issued
// so far, rescales its rows of O (and l) and signals back.  The values of a
// kept tile are loaded (by TMA, from L2 as a rule: the key stream just read
// them) only once the vote has kept it.
//
// Rows 64..127 of the score MMA: only 64 query rows are staged (72 KB); the
// A descriptor of the last 64-entry chunk runs into the first key slot for
// rows 64..127.  Those rows' scores, P and O are never read.
//
// Roles (256 threads, 8 warps):
//   warps 0-3  softmax / vote, one thread per head;
//   warp 4     barrier setup, TMA producer of the key stream (64-entry
//              chunks of 128 keys);
//   warp 5     TMA producer of the values of kept tiles (this CTA's half);
//   warp 6     TMEM allocation, issuer of the score MMAs;
//   warp 7     issuer of the P.V MMAs (the whole warp zeroes the rows of a
//              partial page past the sequence end).
#include <cuda_bf16.h>

#include "mla.cuh"
#include "ptx_sm103.cuh"

namespace ssattn {

namespace {

constexpr int kRThreads = 256;
constexpr int kRWarpK = 4, kRWarpV = 5, kRWarpS = 6, kRWarpPV = 7;
constexpr int kRHalf = kMlaLatent / 2;  // latent entries of O per CTA
constexpr float kRRescaleLog2 = 8.0f;
constexpr uint32_t kRFlagKept = 1u, kRFlagRescale = 2u;

struct RCfg {
  static constexpr int kChunks = kMlaDk / 64;              // 64-entry chunks of a key row
  static constexpr int NKB = 5;                             // key-chunk slots
  static constexpr int NVP = 2;                             // value slots (128 latent entries)
  static constexpr int NVQ = 4;                             // kept-tile queue entries
  static constexpr int kChunkBytes = kTile * 64 * 2;        // 128 keys x 64 entries
  static constexpr int kQChunkBytes = kMlaRowsMaxHeads * 128;  // 64 rows x 64 entries
  static constexpr int kPairBytes = kTile * 128 * 2;        // 128 keys x 128 latent entries
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + kChunks * kQChunkBytes;
  static constexpr int kVOff = kKOff + NKB * kChunkBytes;
  static constexpr int kCtlOff = kVOff + NVP * kPairBytes;
  static constexpr int kCtlBytes = 1024;
  static constexpr int kSmemBytes = kCtlOff + kCtlBytes + 1024;  // + alignment slack
  static constexpr uint32_t kColO = 256;                    // O: columns 256 .. 511
  static constexpr uint32_t kTmemCols = 512;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
  // rows 64..127 of the last query chunk are read from the first key slot
  static_assert(kKOff == kQOff + kChunks * kQChunkBytes && NKB * kChunkBytes >= kQChunkBytes,
                "query rows 64..127 stay inside shared memory");
};

struct RCtl {
  uint64_t kb_full[RCfg::NKB], kb_empty[RCfg::NKB];
  uint64_t vp_full[RCfg::NVP], vp_empty[RCfg::NVP];
  uint64_t vq_full[RCfg::NVQ], vq_empty[RCfg::NVQ];
  uint64_t s_full[2];    // scores of the buffer's tile are in TMEM
  uint64_t s_free[2];    // the buffer's P.V is issued (or not needed)
  uint64_t dec[2];       // the 4 softmax warps have decided the buffer's tile
  uint64_t drain[4];     // per softmax warp: the P.V MMAs issued so far are done
  uint64_t rescaled[4];  // per softmax warp: its rows of O are rescaled
  uint64_t o_full;       // the last P.V is done
  uint64_t mma_done[2];  // teardown, per issuer
  alignas(16) uint32_t flags[2][4];  // per buffer and softmax warp: kept | rescale
  int kq[RCfg::NVQ];     // kept tiles for the value producer (-1: no more)
  uint32_t tmem_base;
  int abort_flag;
  float red[4];
};

template <Mode MODE>
__global__ void __launch_bounds__(kRThreads, 1)
    mla_decode_rows_kernel(const __grid_constant__ CUtensorMap tmKV, const MlaParams p) {
  using C = RCfg;
  constexpr int NKB = C::NKB, NVP = C::NVP, NVQ = C::NVQ, kChunks = C::kChunks;
  constexpr bool kPV = (MODE != Mode::kCount);
  constexpr bool kVote = (MODE != Mode::kDense);
  static_assert(sizeof(RCtl) <= C::kCtlBytes, "control block overflow");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem + C::kQOff;
  uint8_t* sK = smem + C::kKOff;
  uint8_t* sV = smem + C::kVOff;
  auto* ctl = reinterpret_cast<RCtl*>(smem + C::kCtlOff);
  volatile int* abort_flag = &ctl->abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = p.Hq;
  const int half = blockIdx.x & 1;
  const int split = (blockIdx.x >> 1) % p.S;
  const int b = (blockIdx.x >> 1) / p.S;
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
  auto tile_y = [&](int t) { return paged ? 0 : (j0 + t) * kTile; };
  auto tile_z = [&](int t) {
    return paged ? p.page_table[static_cast<long>(b) * p.max_pages + j0 + t] : b;
  };

  // ------------------------------------------------------------------ setup
  int n_k = 0;  // key-chunk copies issued (teardown bookkeeping)
  auto issue_chunk = [&](int e) {
    const int t = e / kChunks, c = e - (e / kChunks) * kChunks, st = e % NKB;
    mbar_arrive_expect_tx(&ctl->kb_full[st], C::kChunkBytes);
    tma_load_3d(sK + st * C::kChunkBytes, &tmKV, &ctl->kb_full[st], 64 * c, tile_y(t), tile_z(t));
    n_k = e + 1;
  };
  if (warp == kRWarpK && lane == 0) {
    for (int s = 0; s < NKB; ++s) {
      mbar_init(&ctl->kb_full[s], 1);
      mbar_init(&ctl->kb_empty[s], 1);
    }
    for (int s = 0; s < NVP; ++s) {
      mbar_init(&ctl->vp_full[s], 1);
      mbar_init(&ctl->vp_empty[s], 1);
    }
    for (int s = 0; s < NVQ; ++s) {
      mbar_init(&ctl->vq_full[s], 1);
      mbar_init(&ctl->vq_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
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
    tma_prefetch_desc(&tmKV);
    for (int e = 0; e < min(nt * kChunks, NKB); ++e) issue_chunk(e);
  }
  if (warp == kRWarpS) {
    tmem_alloc(&ctl->tmem_base, C::kTmemCols);
    tmem_relinquish();
  }
  if (warp < 4) {
    // Queries as the score MMA's A operand: 64 rows x 576, K-major, one
    // 64-entry chunk after another, 128-byte swizzle; rows >= G are zero.
    constexpr int kGran = kMlaDk / 8;
    for (int idx = tid; idx < kMlaRowsMaxHeads * kGran; idx += 128) {
      const int g = idx / kGran, e8 = idx - (idx / kGran) * kGran;
      uint4 val = make_uint4(0u, 0u, 0u, 0u);
      if (g < G)
        val = *reinterpret_cast<const uint4*>(p.q + (static_cast<size_t>(b) * p.Hq + g) * kMlaDk +
                                              e8 * 8);
      *reinterpret_cast<uint4*>(sQ + (e8 >> 3) * C::kQChunkBytes + g * 128 +
                                (((e8 & 7) ^ (g & 7)) << 4)) = val;
    }
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;

  if (warp == kRWarpK) {
    // ---------------------------------------------------------- key producer
    if (lane == 0)
      for (int e = NKB; e < nt * kChunks; ++e) {
        if (!mbar_wait(&ctl->kb_empty[e % NKB], ((e / NKB) & 1) ^ 1, abort_flag)) break;
        issue_chunk(e);
      }
    if (lane == 0 && *abort_flag) mla_drain_ring<NKB>(ctl->kb_full, n_k);
    __syncwarp();
  } else if (warp == kRWarpV) {
    // -------------------------------------------------------- value producer
    int n_v = 0;
    if (kPV && lane == 0 && nt > 0) {
      bool fine = true;
      for (int i = 0; fine; ++i) {
        const int s = i % NVQ;
        if (!mbar_wait(&ctl->vq_full[s], (i / NVQ) & 1, abort_flag)) break;
        const int t = *reinterpret_cast<volatile int*>(&ctl->kq[s]);
        mbar_arrive(&ctl->vq_empty[s]);
        if (t < 0) break;
        for (int c = 0; c < 2; ++c) {
          const int f = 2 * i + c, vs = f % NVP;
          if (!mbar_wait(&ctl->vp_empty[vs], ((f / NVP) & 1) ^ 1, abort_flag)) {
            fine = false;
            break;
          }
          mbar_arrive_expect_tx(&ctl->vp_full[vs], C::kPairBytes);
          uint8_t* dst = sV + vs * C::kPairBytes;
          const int x = kRHalf * half + 128 * c;
          tma_load_3d(dst, &tmKV, &ctl->vp_full[vs], x, tile_y(t), tile_z(t));
          tma_load_3d(dst + 16384, &tmKV, &ctl->vp_full[vs], x + 64, tile_y(t), tile_z(t));
          n_v = f + 1;
        }
      }
    }
    if (lane == 0 && *abort_flag) mla_drain_ring<NVP>(ctl->vp_full, n_v);
    __syncwarp();
  } else if (warp == kRWarpS) {
    // ---------------------------------------------------------- score MMAs
    if (lane == 0 && nt > 0) {
      constexpr uint32_t idS = idesc_bf16_f32(128, 128, false, false);
      const uint64_t dq = smem_desc(smem_u32(sQ), 16, 1024);
      const uint32_t sKa = smem_u32(sK);
      bool fine = true;
      for (int t = 0; t < nt && fine; ++t) {
        const int sb = t & 1;
        // The buffer's previous tile was decided and its P.V issued (P lives
        // in the score buffer): the P.V issuer's fence + barrier order this
        // MMA after it.
        if (t >= 2 && !mbar_wait(&ctl->s_free[sb], ((t >> 1) - 1) & 1, abort_flag)) break;
        for (int c = 0; c < kChunks; ++c) {
          const int e = kChunks * t + c, st = e % NKB;
          if (!mbar_wait(&ctl->kb_full[st], (e / NKB) & 1, abort_flag)) {
            fine = false;
            break;
          }
          tc_fence_after();
          const uint64_t dk = smem_desc(sKa + st * C::kChunkBytes, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint32_t qa = (c * C::kQChunkBytes + kk * 32) >> 4;
            mma_bf16_ss(tmem + 128u * sb, dq + qa, dk + ((kk * 32) >> 4), idS, (c | kk) ? 1u : 0u);
          }
          mma_commit(&ctl->kb_empty[st]);
        }
        if (fine) mma_commit(&ctl->s_full[sb]);
      }
      mma_commit(&ctl->mma_done[0]);
      mbar_wait(&ctl->mma_done[0], 0, nullptr);  // all MMAs done before TMEM is freed
    }
    __syncwarp();
  } else if (warp == kRWarpPV) {
    // ------------------------------------------------------------ P.V MMAs
    if (nt > 0) {
      constexpr uint32_t idO = idesc_bf16_f32(128, 128, false, true);
      const uint32_t sVa = smem_u32(sV);
      bool fine = true;
      uint32_t o_acc = 0u, nresc = 0u;
      int nk = 0;  // kept tiles so far
      for (int t = 0; t < nt && fine; ++t) {
        const int sb = t & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(&ctl->dec[sb], (t >> 1) & 1, abort_flag))) break;
        const uint4 f4 = *reinterpret_cast<const uint4*>(ctl->flags[sb]);
        const uint32_t f[4] = {f4.x, f4.y, f4.z, f4.w};
        const bool kept = (f[0] & kRFlagKept) != 0;
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
          const int rows = tile_rows(t);
          for (int c = 0; c < 2; ++c) {
            const int fidx = 2 * nk + c, vs = fidx % NVP;
            if (!__all_sync(0xffffffffu,
                            mbar_wait(&ctl->vp_full[vs], (fidx / NVP) & 1, abort_flag))) {
              fine = false;
              break;
            }
            if (paged && rows < kTile) {
              // Rows of a page past the sequence end hold whatever the cache
              // holds: zero them so that P = 0 there cannot meet a non-finite value.
              uint4* base = reinterpret_cast<uint4*>(sV + vs * C::kPairBytes);
              for (int idx = rows * 8 + lane; idx < kTile * 8; idx += 32) {
                base[idx] = make_uint4(0u, 0u, 0u, 0u);
                base[1024 + idx] = make_uint4(0u, 0u, 0u, 0u);
              }
              fence_proxy_async_smem();
            }
            __syncwarp();
            if (lane == 0) {
              tc_fence_after();
              const uint64_t dv = smem_desc(sVa + vs * C::kPairBytes, 16384, 1024);
#pragma unroll
              for (int kk = 0; kk < kTile / 16; ++kk)  // P of keys 16kk..: column 64 (kk / 4) + 8 (kk % 4)
                mma_bf16_ts(tmem + C::kColO + 128u * c,
                            tmem + 128u * sb + 64 * (kk >> 2) + 8 * (kk & 3),
                            dv + ((kk * 2048) >> 4), idO, (o_acc | kk) ? 1u : 0u);
              mma_commit(&ctl->vp_empty[vs]);
            }
            __syncwarp();
          }
          if (!fine) break;
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
    // to the end of the loop (every later wait gives up at once), so all
    // 128 threads take the same sequence of barriers.  The tcgen05 loads and
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
    int n_vq = 0;  // kept tiles pushed to the value producer (thread 0)
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
      const int sb = t & 1;
      const uint32_t colS = lane_base + 128u * sb;
      if (!wwait(&ctl->s_full[sb], (t >> 1) & 1)) ok = false;
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
      // the heads, and the decision.
      if (p.margin != nullptr) {
        float cm = c;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, o));
        if (lane == 0) *reinterpret_cast<volatile float*>(&ctl->red[warp]) = cm;
        named_bar_sync(1, 128);
        if (tid == 0 && half == 0) {
          const volatile float* rr = ctl->red;
          const float cmax = fmaxf(fmaxf(rr[0], rr[1]), fmaxf(rr[2], rr[3]));
          p.margin[static_cast<long>(b) * row_stride + j0 + t] =
              (cmax == INFINITY) ? INFINITY : cmax * p.scale;
        }
        named_bar_sync(1, 128);  // red[] is read before the next tile writes it
      }
      if (tid == 0) {
        skipped += kept ? 0u : 1u;
        if (half == 0 && p.mask != nullptr)
          p.mask[static_cast<long>(b) * row_stride + j0 + t] = kept ? 0 : 1;
      }
      m_true = fmaxf(m_true, tmax);
      bool resc = false;
      float alpha = 1.f;
      if (kPV && kept) {
        if (tid == 0) {
          // The values of this tile may be fetched now.
          const int s = n_vq % NVQ;
          if (!mbar_wait(&ctl->vq_empty[s], ((n_vq / NVQ) & 1) ^ 1, abort_flag)) ok = false;
          ctl->kq[s] = t;
          mbar_arrive(&ctl->vq_full[s]);
          ++n_vq;
        }
        bool need = false;
        if (m_ref == -INFINITY) {
          m_ref = m_true;  // no key of this row counted yet: its O row and l are zero
        } else if ((m_true - m_ref) * sl2 > kRRescaleLog2) {
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
        ctl->flags[sb][warp] = (kept ? kRFlagKept : 0u) | (resc ? kRFlagRescale : 0u);
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
          for (int cc = 0; cc < kRHalf / 32; ++cc) {
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

    if (kPV && tid == 0) {
      // End of the kept stream for the value producer.
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
      const size_t hrow = static_cast<size_t>(b) * p.Hq + min(row, G - 1);
      if (p.S == 1) {
        // O / l -> bf16 (a head that saw no key writes zeros).
        const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
        __nv_bfloat16* orow = p.o + hrow * kMlaLatent + kRHalf * half;
#pragma unroll 1
        for (int cc = 0; cc < kRHalf / 32; ++cc) {
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
        float* pr = p.part + (hrow * p.S + split) * (kMlaLatent + 2);
#pragma unroll 1
        for (int cc = 0; cc < kRHalf / 32; ++cc) {
          uint32_t orr[32];
          if (nt > 0) {
            tmem_ld32p(colO + cc * 32, orr);
            tmem_wait_ld();
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) orr[e] = 0u;
          }
          // (a partial row is 514 floats: 8-byte aligned, not 16)
          if (active) {
            float2* dst = reinterpret_cast<float2*>(pr + kRHalf * half + cc * 32);
#pragma unroll
            for (int e = 0; e < 16; ++e)
              dst[e] = make_float2(__uint_as_float(orr[2 * e]), __uint_as_float(orr[2 * e + 1]));
          }
        }
        if (half == 0 && active) {
          pr[kMlaLatent] = (m_ref == -INFINITY) ? -INFINITY : m_ref * sl2;
          pr[kMlaLatent + 1] = l;
        }
      }
    }
    if (tid == 0 && half == 0 && p.counts != nullptr)
      p.counts[static_cast<long>(b) * p.S + split] = skipped;
    if (paged && split == 0 && half == 0 && tid < 32)
      for (int j = nT_b + tid; j < p.max_pages; j += 32) {
        const long gi = static_cast<long>(b) * row_stride + j;
        if (p.mask != nullptr) p.mask[gi] = 2;
        if (p.margin != nullptr) p.margin[gi] = NAN;
      }
    tc_fence_before();
    __syncwarp();
  }

  // ------------------------------------------------------------------ teardown
  __syncthreads();
  if (warp == kRWarpS) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  if (tid == 0 && *abort_flag) report_timeout(p.status);
}

template <Mode MODE>
cudaError_t launch_rows(const CUtensorMap& tkv, const MlaParams& p, cudaStream_t st) {
  auto* fn = mla_decode_rows_kernel<MODE>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       RCfg::kSmemBytes);
  if (e != cudaSuccess) return e;
  const long ctas = 2L * p.B * p.S;  // two latent halves per (sequence, split)
  fn<<<dim3(static_cast<unsigned>(ctas)), dim3(kRThreads), RCfg::kSmemBytes, st>>>(tkv, p);
  e = cudaGetLastError();
  if (e != cudaSuccess || MODE == Mode::kCount || p.S == 1) return e;
  return launch_mla_merge(p, st);
}

}  // namespace

cudaError_t launch_mla_decode_rows(const CUtensorMap& tkv, const MlaParams& p, Mode mode,
                                   cudaStream_t st) {
  switch (mode) {
    case Mode::kDense: return launch_rows<Mode::kDense>(tkv, p, st);
    case Mode::kSparse: return launch_rows<Mode::kSparse>(tkv, p, st);
    default: return launch_rows<Mode::kCount>(tkv, p, st);
  }
}

}  // namespace ssattn
