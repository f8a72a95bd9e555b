// Skip-softmax (BLASST) prefill forward for sm_103a on CTA pairs.
//
// Method ("Skip-Softmax" design doc, §The online-softmax pass and §The skip
// test; BLASST summary, §Methodologie and §Kernel-ontwerp): one streaming
// pass over 128-key tiles keeping per query row m, l and O; the scores
// S_j = Q K_j^T * scale always run on the tensor cores; when every row of a
// 128-row query block has exp(scale * (tile_max - m)) < lambda, the tile's
// exponentials and its P.V are skipped and it adds nothing to l or O.
//
// Head widths: d_qk = d_v = 128; d_qk = 192 with d_v = 128 (latent
// attention); d = 64 with the value tiles padded to 128 columns (the second
// SM's half of each value tile is a fully out-of-range TMA box, read as zeros).
//
// One cluster of two CTAs = query blocks 2p and 2p + 1 of one (b, h_q); the
// CTAs run on two SMs and share every K/V tile through two-SM MMAs
// (tcgen05.mma.cta_group::2, M = 256: each SM computes its own block's 128
// rows).  Each SM stages half of every operand tile: 64 of the tile's 128
// keys of K and 64 of the d_v columns of V, next to its own Q block.  TMEM
// per SM: three score buffers S_0..S_2 (columns 0, 128, 256) and O (384 ..
// 384 + d_v), so the score MMAs of the next tiles run while the softmax of a
// tile decides and exponentiates.
//
// One pass, every tile once.  Per tile j, in each CTA:
//   the softmax warpgroup j % 2 (warps 4 (j % 2) .. + 3, one thread per
//   query row: warp w has TMEM lanes 32 (w % 4) .. + 31) loads S_j in two
//   halves of 64 columns, masks it and takes each row's maximum; receives
//   the rows' running state (exact maximum m, reference maximum m_ref) from
//   the warpgroup that did tile j - 1; votes with one bar.red.and over its
//   128 threads against m (every row must pass); hands the updated state on;
//   and for a kept tile computes P = exp2((S - m_ref) * scale * log2e), for a
//   skipped one zeros (the pair's P.V covers both blocks and the other block
//   may keep the tile), as bf16 pairs over the first 32 columns of each
//   half.  So the two warpgroups' work overlaps: one exponentiates while the
//   other loads and votes, and only the short state hand-over is serial
//   from tile to tile.  Each of the warpgroup's warps then publishes its
//   decision: in CTA 0 by a store and an arrival on a local barrier, in CTA
//   1 by an asynchronous store into CTA 0 that completes 4 bytes on CTA 0's
//   barrier (a plain remote store followed by a cluster-scope release would
//   cost the warp a memory barrier, ~1400 cycles, on every tile).
//   In CTA 0 two threads issue the pair's MMAs: the P.V issuer waits for both
//   blocks' decisions on tile j and, if either keeps it, issues O += P_j V_j
//   (A = P from TMEM); then it frees the tile's score buffer for the score
//   issuer, which issues S_{j+3} into it.  The P.V issuer passes a tcgen05
//   fence before that barrier, which orders S_{j+3} after PV_j.
// What bounds it (measured on sm_103a): one thread issues two-SM M256 N128
// K16 MMAs at the pipe's rate, 64 cycles each, in any operand form; two
// threads issuing at once interleave at ~88 cycles per step, and TMEM loads
// and stores by other warps slow concurrent MMAs further.  Here the steps
// average ~85-95 cycles: with every softmax operation removed the dense
// kernel still takes 93% of its time.  One issuer thread is slower (an MMA
// issue waits for the pipe, so the thread cannot wait for decisions while
// the pipe is busy), and so is P in shared memory (shared-memory bandwidth).
// m_ref, the maximum P is referenced to, trails the exact maximum lazily: a
// row moves it only when the exact maximum has grown by more than 2^8 in
// exp2 units (so P stays below 256); the warps on such rows then ask the
// P.V issuer to drain the P.V MMAs issued so far, rescale their part of O
// and l, and signal back before that tile's P.V is issued.  With the tile order
// fixed, kept tiles, counters and O are those of the one-pass definition.
//
// Roles (384 threads, 12 warps, in each CTA):
//   warps 0-7  softmax and vote of this CTA's query block, as two
//              warpgroups taking alternate tiles;
//   warp 8     TMA producer of Q (once) and of this CTA's halves of K;
//   warp 9     TMA producer of this CTA's halves of V;
//   warp 10    TMEM allocation (both CTAs, two-SM form); in CTA 0 the issuer
//              of the score MMAs;
//   warp 11    in CTA 0 the issuer of the P.V MMAs; idle in CTA 1.
// Both halves of a K or V tile complete one mbarrier of CTA 0 (the peer's
// TMA signals CTA 0's barrier); CTA 0's commits arrive on the barriers of
// both CTAs (multicast).
#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx_pair_sm103.cuh"
#include "ptx_sm103.cuh"

namespace ssattn {

namespace {

constexpr float kRescaleLog2 = 8.0f;  // lazy-rescale slack (exp2 domain)
constexpr int kSoftWarps = 8;                 // two warpgroups of 4: alternate tiles
constexpr int kGroupWarps = 4;                // one thread per query row
constexpr int kSoftThreads = 32 * kSoftWarps;
constexpr int kThreads = kSoftThreads + 128;  // + producers and issuers
constexpr int kWarpK = 8, kWarpV = 9, kWarpMma = 10, kWarpPV = 11;
constexpr int kNB = 3;  // score buffers
constexpr uint32_t kFlagKept = 1u, kFlagRescale = 2u;

// Scheduling fence for registers: the 8 values `done` are complete before,
// and the 16 values `next` are read only after, this point (a compiler hint
// that bounds how far exponentials are hoisted ahead, and so the registers
// they hold; no instruction is emitted).
__device__ __forceinline__ void order_after(uint32_t* done, uint32_t* next) {
  asm volatile(""
               : "+r"(done[0]), "+r"(done[1]), "+r"(done[2]), "+r"(done[3]), "+r"(done[4]),
                 "+r"(done[5]), "+r"(done[6]), "+r"(done[7]), "+r"(next[0]), "+r"(next[1]),
                 "+r"(next[2]), "+r"(next[3]), "+r"(next[4]), "+r"(next[5]), "+r"(next[6]),
                 "+r"(next[7]), "+r"(next[8]), "+r"(next[9]), "+r"(next[10]), "+r"(next[11]),
                 "+r"(next[12]), "+r"(next[13]), "+r"(next[14]), "+r"(next[15]));
}

template <int DQK, int DV>
struct PairCfg {
  static_assert(DQK % 64 == 0 && DQK >= 64 && DQK <= 192, "key width");
  static_assert(DV == 128, "value width: O occupies TMEM columns 384..511");
  static constexpr int kChunksQ = DQK / 64;             // 128-byte swizzle chunks per row
  static constexpr int kQBytes = kTile * DQK * 2;        // this CTA's query block
  static constexpr int kKHalfBytes = 64 * DQK * 2;      // 64 keys of a tile
  static constexpr int kKChunk = 64 * 128;               // one 64-column chunk of 64 keys
  static constexpr int kVHalfBytes = kTile * 64 * 2;    // 64 value columns of a tile
  static constexpr int kNK = (DQK <= 128) ? 6 : 4;       // K ring slots
  static constexpr int kNV = (DQK <= 128) ? 5 : 4;       // V ring slots
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + kQBytes;
  static constexpr int kVOff = kKOff + kNK * kKHalfBytes;
  static constexpr int kCtlOff = kVOff + kNV * kVHalfBytes;
  static constexpr int kCtlBytes = 5120;
  static constexpr int kSmemBytes = kCtlOff + kCtlBytes + 1024;  // + alignment slack
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
  static constexpr uint32_t kColO = 384;
  static constexpr uint32_t kTmemCols = 512;
};

template <int NK, int NV>
struct PairCtl {
  uint64_t q_full;             // leader: both Q blocks landed
  uint64_t k_full[NK];         // leader: both K halves of a ring entry landed
  uint64_t v_full[NV];         // leader: both V halves landed
  uint64_t k_empty[NK];        // each CTA: its K slot may be refilled
  uint64_t v_empty[NV];        // each CTA: its V slot may be refilled
  uint64_t s_full[kNB];        // each CTA: scores of the buffer's tile are in TMEM
  uint64_t dec[kNB];           // leader: both CTAs' 4 warps on the buffer's tile have decided
                               // it (CTA 0's by arrivals, CTA 1's as 16 bytes of stores)
  uint64_t drain[kSoftWarps];  // each CTA, per softmax warp: the P.V MMAs issued so far are done
  uint64_t rescaled[2][kSoftWarps];  // leader: (CTA, warp) has rescaled its part of O
  uint64_t s_free[kNB];        // leader: the buffer's P.V is issued (or not needed)
  uint64_t o_full;             // each CTA: the last P.V is done
  uint64_t mma_done[2];        // leader: teardown, per issuer
  alignas(16) uint32_t flags[kNB][kGroupWarps];       // leader: per buffer and warp of the
                                                      // tile's warpgroup, kFlagKept | kFlagRescale
  alignas(16) uint32_t peer_flags[kNB][kGroupWarps];  // leader: the same for CTA 1's warps
  uint32_t tmem_base;
  int abort_flag;
  uint32_t skipped[2];         // per warpgroup: tiles it skipped
  float red[2][kGroupWarps];   // per warpgroup and warp: largest vote statistic of a tile
  float2 hand[kTile];          // per row: (m, m_ref) after the last tile, passed between warpgroups
  float2 fin[2][kTile];        // per warpgroup and row: (m_ref, l) at the end
};

// DVO: the value (and output) width in memory.  DVO = 64 runs as DV = 128
// with the second SM's half of every value tile a fully out-of-range TMA box
// (read as zeros): O's columns 64.. stay zero and are not written.
template <int DQK, int DV, int DVO, Mode MODE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    prefill_pair_kernel(const __grid_constant__ CUtensorMap tmQ,
                        const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const PrefillParams p) {
  using C = PairCfg<DQK, DV>;
  static_assert(DVO == DV || (DVO == 64 && DV == 128), "value width");
  constexpr int NK = C::kNK, NV = C::kNV;
  using Ctl = PairCtl<NK, NV>;
  static_assert(sizeof(Ctl) <= C::kCtlBytes, "control block overflow");
  constexpr bool kPV = (MODE != Mode::kCount);
  constexpr bool kVote = (MODE != Mode::kDense);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem + C::kQOff;
  uint8_t* sK = smem + C::kKOff;
  uint8_t* sV = smem + C::kVOff;
  auto* ctl = reinterpret_cast<Ctl*>(smem + C::kCtlOff);
  volatile int* abort_flag = &ctl->abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = (rank == 0);
  const uint32_t peer_abort = map_shared(smem_u32(&ctl->abort_flag), rank ^ 1u);
  // shared::cluster address of a barrier of the leader
  auto lead = [&](uint64_t* bar) { return map_shared(smem_u32(bar), 0u); };

  // Work: query blocks 2*pr and 2*pr + 1 of head (b, h); causal: heaviest first.
  const int nP = (p.nQB + 1) / 2;
  const int x = blockIdx.x >> 1;
  const int bh = x / nP;
  const int ip = x - bh * nP;
  const int pr = p.causal ? (nP - 1 - ip) : ip;
  const int b = bh / p.Hq, h = bh - (bh / p.Hq) * p.Hq;
  const int kvh = h / p.G;
  const int zk = b * p.Hkv + kvh;
  const long off = static_cast<long>(p.Lk) - p.Lq;
  // tiles evaluated by either block of the pair (every CTA computes both)
  int n_pair = 0, n_mine = 0, rows_mine = 0;
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int r0 = (2 * pr + t) * kTile;
    const int rows = max(0, min(kTile, p.Lq - r0));
    int n = (rows > 0) ? p.nT : 0;
    if (p.causal && rows > 0) {
      const long last = static_cast<long>(r0) + rows - 1 + off;
      n = last < 0 ? 0 : min(p.nT, static_cast<int>(last / kTile) + 1);
    }
    n_pair = max(n_pair, n);
    if (t == static_cast<int>(rank)) {
      n_mine = n;
      rows_mine = rows;
    }
  }
  const int qb = 2 * pr + static_cast<int>(rank);
  const int r0_mine = qb * kTile;

  if (tid == 0) {
    mbar_init(&ctl->q_full, 1);
    for (int s = 0; s < NK; ++s) {
      mbar_init(&ctl->k_full[s], 1);
      mbar_init(&ctl->k_empty[s], 1);
    }
    for (int s = 0; s < NV; ++s) {
      mbar_init(&ctl->v_full[s], 1);
      mbar_init(&ctl->v_empty[s], 1);
    }
    for (int s = 0; s < kNB; ++s) {
      mbar_init(&ctl->s_full[s], 1);
      // this CTA's 4 warps + the score issuer's arrival (which sets the 16
      // bytes that CTA 1's 4 warps complete)
      mbar_init(&ctl->dec[s], kGroupWarps + 1);

    }
    for (int w = 0; w < kSoftWarps; ++w) {
      mbar_init(&ctl->drain[w], 1);
      mbar_init(&ctl->rescaled[0][w], 1);
      mbar_init(&ctl->rescaled[1][w], 1);
    }
    for (int b = 0; b < kNB; ++b) mbar_init(&ctl->s_free[b], 1);
    mbar_init(&ctl->o_full, 1);
    mbar_init(&ctl->mma_done[0], 1);
    mbar_init(&ctl->mma_done[1], 1);
    ctl->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc_pair(&ctl->tmem_base, C::kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();  // barriers of both CTAs initialised, TMEM allocated
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;

  if (warp == kWarpK) {
    // ------------------------------------------------------------ Q, K producer
    if (lane == 0 && n_pair > 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      if (leader) mbar_arrive_expect_tx(&ctl->q_full, 2 * C::kQBytes);
      const uint32_t qbar = lead(&ctl->q_full);
#pragma unroll
      for (int c = 0; c < C::kChunksQ; ++c)
        tma_load_3d_pair(sQ + c * (kTile * 128), &tmQ, qbar, c * 64, r0_mine, bh);
      for (int j = 0; j < n_pair; ++j) {
        const int s = j % NK;
        if (!mbar_wait_pair(&ctl->k_empty[s], ((j / NK) & 1) ^ 1, abort_flag, peer_abort)) break;
        if (leader) mbar_arrive_expect_tx(&ctl->k_full[s], 2 * C::kKHalfBytes);
        const uint32_t kbar = lead(&ctl->k_full[s]);
#pragma unroll
        for (int c = 0; c < C::kChunksQ; ++c)
          tma_load_3d_pair(sK + s * C::kKHalfBytes + c * C::kKChunk, &tmK, kbar, c * 64,
                           j * kTile + 64 * static_cast<int>(rank), zk);
      }
    }
    __syncwarp();
  } else if (warp == kWarpV) {
    // ------------------------------------------------------------ V producer
    if (kPV && lane == 0 && n_pair > 0) {
      tma_prefetch_desc(&tmV);
      for (int j = 0; j < n_pair; ++j) {
        const int s = j % NV;
        if (!mbar_wait_pair(&ctl->v_empty[s], ((j / NV) & 1) ^ 1, abort_flag, peer_abort)) break;
        if (leader) mbar_arrive_expect_tx(&ctl->v_full[s], 2 * C::kVHalfBytes);
        tma_load_3d_pair(sV + s * C::kVHalfBytes, &tmV, lead(&ctl->v_full[s]),
                         64 * static_cast<int>(rank), j * kTile, zk);
      }
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ score issuer (leader)
    if (leader && lane == 0 && n_pair > 0) {
      constexpr uint32_t idS = idesc_bf16_f32(256, 128, false, false);
      const uint64_t dq = smem_desc(smem_u32(sQ), 16, 1024);
      const uint32_t sKa = smem_u32(sK);
      bool ok = mbar_wait_pair(&ctl->q_full, 0, abort_flag, peer_abort);
      for (int t = 0; ok && t < n_pair; ++t) {
        const int bsel = t % kNB;
        // The buffer's previous tile has been decided by both blocks and its
        // P.V (if any) issued: S_t is ordered after it (tcgen05 fence + barrier).
        if (t >= kNB && !(ok = mbar_wait_pair(&ctl->s_free[bsel], ((t / kNB) - 1) & 1, abort_flag,
                                              peer_abort)))
          break;
        const int s = t % NK;
        if (!(ok = mbar_wait_pair(&ctl->k_full[s], (t / NK) & 1, abort_flag, peer_abort))) break;
        tc_fence_after();
        const uint64_t dk = smem_desc(sKa + s * C::kKHalfBytes, 16, 1024);
        const uint32_t col = 128u * static_cast<uint32_t>(bsel);
#pragma unroll
        for (int kk = 0; kk < DQK / 16; ++kk) {
          const uint32_t qoff = ((kk >> 2) * (kTile * 128) + (kk & 3) * 32) >> 4;
          const uint32_t koff = ((kk >> 2) * C::kKChunk + (kk & 3) * 32) >> 4;
          mma2_bf16_ss(tmem + col, dq + qoff, dk + koff, idS, kk > 0 ? 1u : 0u);
        }
        mma2_commit_mc(&ctl->s_full[bsel], 3);
        mma2_commit_mc(&ctl->k_empty[s], 3);
        // CTA 1's four warps on this tile complete 4 bytes each on dec; this
        // arrival sets that count for the tile's phase.
        mbar_arrive_expect_tx(&ctl->dec[bsel], 4 * kGroupWarps);
      }
      // Every MMA issued must have finished before TMEM is freed.
      mma2_commit_mc(&ctl->mma_done[0], 1);
      mbar_wait(&ctl->mma_done[0], 0, nullptr);
    }
    __syncwarp();
  } else if (warp == kWarpPV) {
    // ------------------------------------------------------------ P.V issuer (leader)
    if (leader && lane == 0 && n_pair > 0) {
      constexpr uint32_t idO = idesc_bf16_f32(256, DV, false, true);
      const uint32_t sVa = smem_u32(sV);
      bool ok = true;
      uint32_t o_acc = 0u;
      uint32_t nresc = 0u;  // bit (kSoftWarps * r + warp): parity of (CTA r, warp)'s requests
      for (int j = 0; ok && j < n_pair; ++j) {
        const int bsel = j % kNB;
        const uint32_t ph = (j / kNB) & 1;
        // The tile's V halves do not depend on the decisions: wait for them
        // first, while the softmax is still deciding.
        const int vs = j % NV;
        if (kPV && !mbar_wait_pair(&ctl->v_full[vs], (j / NV) & 1, abort_flag, peer_abort)) {
          ok = false;
          break;
        }
        if (!mbar_wait_pair(&ctl->dec[bsel], ph, abort_flag, peer_abort)) {
          ok = false;
          break;
        }
        // Tile j's decisions come from the warps of warpgroup j % 2.
        const int wg0 = kGroupWarps * (j & 1);
        uint32_t resc = 0u, any_kept = 0u;  // resc: bit (kGroupWarps * r + w)
        {
          // (plain loads: the barrier waits above are compiler memory barriers)
          const uint4 f4 = *reinterpret_cast<const uint4*>(ctl->flags[bsel]);
          const uint4 g4 = *reinterpret_cast<const uint4*>(ctl->peer_flags[bsel]);
          const uint32_t f[4] = {f4.x, f4.y, f4.z, f4.w};
          const uint32_t g[4] = {g4.x, g4.y, g4.z, g4.w};
#pragma unroll
          for (int w = 0; w < kGroupWarps; ++w) {
            any_kept |= (f[w] | g[w]) & kFlagKept;
            resc |= ((f[w] >> 1) & 1u) << w;
            resc |= ((g[w] >> 1) & 1u) << (kGroupWarps + w);
          }
        }
        if (kPV && resc) {
          // Warps that move their reference maximum rescale O once every P.V
          // issued so far has finished.
#pragma unroll
          for (int r = 0; r < 2; ++r)
#pragma unroll
            for (int w = 0; w < kGroupWarps; ++w)
              if (resc & (1u << (kGroupWarps * r + w)))
                mma2_commit_mc(&ctl->drain[wg0 + w], static_cast<uint16_t>(1u << r));
#pragma unroll
          for (int r = 0; r < 2; ++r)
#pragma unroll
            for (int w = 0; w < kGroupWarps; ++w) {
              const uint32_t bit = 1u << (kSoftWarps * r + wg0 + w);
              if (ok && (resc & (1u << (kGroupWarps * r + w)))) {
                const uint32_t par = (nresc & bit) ? 1u : 0u;
                ok = (r == 0) ? mbar_wait_pair(&ctl->rescaled[0][wg0 + w], par, abort_flag, peer_abort)
                              : mbar_wait_pair<true>(&ctl->rescaled[1][wg0 + w], par, abort_flag,
                                                     peer_abort);
                nresc ^= bit;
              }
            }
          if (!ok) break;
        }
        if (kPV) {
          if (any_kept) {
            tc_fence_after();
            const uint64_t dv = smem_desc(sVa + vs * C::kVHalfBytes, 16384, 1024);
            const uint32_t pcol = 128u * static_cast<uint32_t>(bsel);
#pragma unroll
            for (int kk = 0; kk < kTile / 16; ++kk)  // P of keys 16kk..: column 64 (kk / 4) + 8 (kk % 4)
              mma2_bf16_ts(tmem + C::kColO, tmem + pcol + 64 * (kk >> 2) + 8 * (kk & 3),
                           dv + ((kk * 2048) >> 4), idO, (o_acc | kk) ? 1u : 0u);
            o_acc = 1u;
          }
          mma2_commit_mc(&ctl->v_empty[vs], 3);
        }
        tc_fence_before();
        mbar_arrive(&ctl->s_free[bsel]);
      }
      if (kPV && ok) mma2_commit_mc(&ctl->o_full, 3);
      mma2_commit_mc(&ctl->mma_done[1], 1);
      mbar_wait(&ctl->mma_done[1], 0, nullptr);
    }
    __syncwarp();
  } else if (warp < kSoftWarps) {
    // ------------------------------------------------------------ softmax / vote
    // Two warpgroups take alternate tiles: warpgroup g = warp / 4 handles the
    // tiles j with j % 2 == g, one thread per query row (warp w reads TMEM
    // lanes 32 (w % 4) .. + 31) over all 128 score columns, loaded as two
    // halves of 64.  A row's running state passes from one warpgroup to the
    // other once per tile: the warpgroup on tile j - 1 writes the exact running
    // maximum m (the vote's reference) and the reference maximum m_ref of P to
    // shared memory and arrives on a named barrier, and the warpgroup on tile j
    // completes that barrier before its vote (one barrier per direction, so an
    // arrival can only complete the hand-over it is meant for).  The state chain of consecutive
    // tiles is therefore short (a barrier, the vote, a store), and each
    // warpgroup's loads, maxima and exponentials overlap the other's.  Each
    // warpgroup sums its own tiles' P into l against the m_ref it last saw; a
    // moved m_ref rescales that sum when the state arrives, and the two sums
    // meet at the end.  After a failed wait a thread carries on to the end of
    // the loop (every later wait gives up at once), so all threads take the
    // same sequence of named barriers.
    const int g = warp / kGroupWarps, q4 = warp % kGroupWarps;
    const int row = q4 * 32 + lane;  // TMEM lane
    const int gtid = tid - 128 * g;  // thread index within the warpgroup
    const long grow = static_cast<long>(r0_mine) + row;
    const bool row_valid = row < rows_mine;
    long lim = static_cast<long>(p.Lk) - 1;  // last key index this row may see
    if (p.causal && grow + off < lim) lim = grow + off;
    if (!row_valid) lim = -1;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(q4 * 32) << 16);
    const uint32_t colO = lane_base + C::kColO;
    const float sl2 = p.scale_log2;
    const long unit = static_cast<long>(bh) * p.nQB + qb;
    const bool has_unit = rows_mine > 0;
    float m_true = -INFINITY, m_ref = -INFINITY, l = 0.f;
    uint32_t skipped = 0, n_drain = 0;
    bool ok = true;
    auto wwait = [&](uint64_t* bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait_pair(bar, parity, abort_flag, peer_abort));
    };
    constexpr uint32_t kBar = 2;               // named barrier of all softmax threads
    const uint32_t bar_give = 3 + g;           // hand-over from this warpgroup
    const uint32_t bar_take = 3 + (g ^ 1);     // hand-over to this warpgroup
    const uint32_t bar_vote = 5 + g;           // the 128 threads of this warpgroup

    // Scores of keys 64 hf .. + 63 of tile j, masked, into sr; returns their maximum.
    auto load_half = [&](uint32_t colS, int j, int hf, uint32_t* sr) -> float {
      tmem_ld32p(colS + 64 * hf, sr);
      tmem_ld32p(colS + 64 * hf + 32, sr + 32);
      tmem_wait_ld();
      const long k0 = static_cast<long>(j) * kTile + 64 * hf;
      if (!(k0 + 63 <= lim)) {
        const int vis = static_cast<int>(max(-1L, min(63L, lim - k0)));
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
    // P = exp2(s*scale*log2e - m_ref*scale*log2e) of the 64 scores in sr, as
    // bf16 pairs into sr[0..31]; returns their sum.
    auto exp_half = [&](uint32_t* sr) -> float {
      const float mb = (m_ref == -INFINITY) ? 0.f : m_ref * sl2;
      const uint64_t sl2x2 = f32x2(sl2, sl2), nmb = f32x2(-mb, -mb);
      uint64_t ls[2] = {0ull, 0ull};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
#pragma unroll
        for (int cc = 8 * q; cc < 8 * q + 8; ++cc) {
          const uint64_t xp = fma_f32x2(
              f32x2(__uint_as_float(sr[2 * cc]), __uint_as_float(sr[2 * cc + 1])), sl2x2, nmb);
          const float p0 = ex2_approx(f32x2_lo(xp));
          const float p1 = ex2_approx(f32x2_hi(xp));
          ls[cc & 1] = add_f32x2(ls[cc & 1], f32x2(p0, p1));
          sr[cc] = pack_bf16x2(p0, p1);
        }
        if (q < 3) order_after(sr + 8 * q, sr + 16 * (q + 1));
      }
      const uint64_t lsum = add_f32x2(ls[0], ls[1]);
      return f32x2_lo(lsum) + f32x2_hi(lsum);
    };

    for (int j = g; j < n_pair; j += 2) {
      const int bsel = j % kNB;
      const uint32_t colS = lane_base + 128u * static_cast<uint32_t>(bsel);
      if (!wwait(&ctl->s_full[bsel], (j / kNB) & 1)) ok = false;
      tc_fence_after();
      const bool mine = j < n_mine;
      uint32_t sr[64];
      float tmax = -INFINITY;
      if (mine) {
        tmax = load_half(colS, j, 0, sr);
        // (finish the first half's maximum before the second half's load, so
        // that only one half of the scores is ever held in registers)
        asm volatile("" : "+f"(tmax));
        tmax = fmaxf(tmax, load_half(colS, j, 1, sr));  // sr keeps the second half
      }
      // The state after tile j - 1, from the other warpgroup.
      if (j > 0) {
        named_bar_sync(bar_take, kSoftThreads);
        const float2 hs = ctl->hand[row];
        m_true = hs.x;
        if (hs.y != m_ref) {
          if (m_ref != -INFINITY) l *= ex2_approx((m_ref - hs.y) * sl2);
          m_ref = hs.y;
        }
      }
      bool kept = false, resc = false;
      float alpha = 1.f;
      if (mine) {
        // Skip vote: every row of the block must pass exp(scale*(tile_max - m)) < lambda.
        float c = -INFINITY;
        if (tmax != -INFINITY) c = (m_true == -INFINITY) ? INFINITY : tmax - m_true;
        if constexpr (kVote) {
          kept = !named_bar_and(bar_vote, 128, c < p.thr_raw);
          if (p.margin != nullptr) {
            float cm = c;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, o));
            if (lane == 0) *reinterpret_cast<volatile float*>(&ctl->red[g][q4]) = cm;
            named_bar_sync(bar_vote, 128);
            if (gtid == 0 && has_unit) {
              const volatile float* rr = ctl->red[g];
              const float cmax = fmaxf(fmaxf(rr[0], rr[1]), fmaxf(rr[2], rr[3]));
              p.margin[unit * p.nT + j] = (cmax == INFINITY) ? INFINITY : cmax * p.scale;
            }
          }
          if (gtid == 0 && has_unit) {
            skipped += kept ? 0u : 1u;
            if (p.mask != nullptr) p.mask[unit * p.nT + j] = kept ? 0 : 1;
          }
        } else {
          kept = true;
        }
        m_true = fmaxf(m_true, tmax);
        if (kPV && kept) {
          // m_ref trails m lazily: it moves only when m has grown by more than
          // 2^8 in exp2 units, and then the warp's rows of O are rescaled.
          bool need = false;
          if (m_ref == -INFINITY) {
            m_ref = m_true;  // no key of this row counted yet: its O row and l are zero
          } else if ((m_true - m_ref) * sl2 > kRescaleLog2) {
            need = true;
          }
          resc = __any_sync(0xffffffffu, need);
          if (resc && m_ref != -INFINITY) {
            alpha = ex2_approx((m_ref - m_true) * sl2);
            l *= alpha;
            m_ref = m_true;
          }
        }
      }
      if (j + 1 < n_pair) {
        ctl->hand[row] = make_float2(m_true, m_ref);
        named_bar_arrive(bar_give, kSoftThreads);
      }
      if constexpr (kPV) {
        // P of keys 64 hf .. as bf16 pairs over the first 32 of those keys'
        // own score columns (64 hf ..); the second half goes first, from the
        // registers, then the first half is loaded again.  A skipped or unseen
        // tile writes zeros (the pair's P.V covers both blocks; the other
        // block may keep the tile).
        if (kept) {
          float ls = exp_half(sr);
          tmem_st32p(colS + 64, sr);
          load_half(colS, j, 0, sr);
          ls += exp_half(sr);
          tmem_st32p(colS, sr);
          l += ls;
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) sr[e] = 0u;
          tmem_st32p(colS + 64, sr);
          tmem_st32p(colS, sr);
        }
        tmem_wait_st();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        const uint32_t f = (kept ? kFlagKept : 0u) | (resc ? kFlagRescale : 0u);
        if (leader) {
          *reinterpret_cast<volatile uint32_t*>(&ctl->flags[bsel][q4]) = f;
          mbar_arrive(&ctl->dec[bsel]);
        } else {
          st_async_u32(map_shared(smem_u32(&ctl->peer_flags[bsel][q4]), 0u), f,
                       lead(&ctl->dec[bsel]));
        }
      }
      if (kPV && resc) {
        // The P.V issuer drains the P.V MMAs issued so far; then this warp's
        // rows of O are rescaled before this tile's P.V.
        if (!wwait(&ctl->drain[warp], n_drain & 1)) ok = false;
        ++n_drain;
        if (ok) {
          tc_fence_after();
#pragma unroll 1
          for (int cc = 0; cc < DV / 32; ++cc) {
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
        if (lane == 0) {
          if (leader)
            mbar_arrive(&ctl->rescaled[0][warp]);
          else
            mbar_arrive_cluster(lead(&ctl->rescaled[1][warp]));
        }
      }
    }

    // The row's denominator: both warpgroups' sums against the later m_ref
    // (the one O is kept against).
    ctl->fin[g][row] = make_float2(m_ref, l);
    if (gtid == 0) ctl->skipped[g] = skipped;
    ok = !named_bar_or(kBar, kSoftThreads, !ok);
    const float2 other = ctl->fin[g ^ 1][row];
    const float m_fin = fmaxf(m_ref, other.x);
    float l_row = 0.f;
    if (m_fin != -INFINITY) {
      if (m_ref != -INFINITY) l_row += l * ex2_approx((m_ref - m_fin) * sl2);
      if (other.x != -INFINITY) l_row += other.y * ex2_approx((other.x - m_fin) * sl2);
    }
    if (kPV && ok && n_pair > 0) {
      ok = wwait(&ctl->o_full, 0);
      tc_fence_after();
    }
    if (kPV && ok && has_unit && g * (DV / 2) < DVO) {
      // Epilogue: this warpgroup's half of the row's O / l -> bf16 (a row that
      // saw no key writes zeros).
      const float inv_l = (l_row > 0.f) ? 1.f / l_row : 0.f;
      __nv_bfloat16* orow = p.o + (static_cast<size_t>(bh) * p.Lq + grow) * DVO + g * (DV / 2);
#pragma unroll 1
      for (int c = 0; c < DV / 64; ++c) {
        uint32_t orr[32];
        if (n_pair > 0) {
          tmem_ld32p(colO + g * (DV / 2) + c * 32, orr);
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
        if (row_valid) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            dst[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
        }
      }
    }
    if (tid == 0 && has_unit) {
      if (p.counts != nullptr) p.counts[unit] = ctl->skipped[0] + ctl->skipped[1];
      for (int j = n_mine; j < p.nT; ++j) {
        if (p.mask != nullptr) p.mask[unit * p.nT + j] = 2;
        if (p.margin != nullptr) p.margin[unit * p.nT + j] = NAN;
      }
    }
    __syncwarp();
  }

  // ------------------------------------------------------------ teardown
  // After an expired wait, copies may still be in flight into either CTA's
  // shared memory (the leader's barriers count both halves): give them time
  // to land before the pair's shared memory is released.
  if (*abort_flag) {
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 50000ull) {
    }
  }
  tc_fence_before();
  cluster_sync_all();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, C::kTmemCols);
  }
  if (tid == 0 && *abort_flag) report_timeout(p.status);
}

template <int DQK, int DV, int DVO, Mode MODE>
cudaError_t launch_pair(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                        const PrefillParams& p, cudaStream_t st) {
  using C = PairCfg<DQK, DV>;
  auto* fn = prefill_pair_kernel<DQK, DV, DVO, MODE>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  const long pairs = static_cast<long>(p.B) * p.Hq * ((p.nQB + 1) / 2);
  // Clusters of two CTAs (the kernel's __cluster_dims__): one per pair.
  fn<<<dim3(static_cast<unsigned>(2 * pairs)), dim3(kThreads), C::kSmemBytes, st>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_pair(int dqk, Mode mode, const CUtensorMap& tq, const CUtensorMap& tk,
                                const CUtensorMap& tv, const PrefillParams& p, cudaStream_t st) {
  if (dqk == 192) {
    switch (mode) {
      case Mode::kDense: return launch_pair<192, 128, 128, Mode::kDense>(tq, tk, tv, p, st);
      case Mode::kSparse: return launch_pair<192, 128, 128, Mode::kSparse>(tq, tk, tv, p, st);
      default: return launch_pair<192, 128, 128, Mode::kCount>(tq, tk, tv, p, st);
    }
  }
  if (dqk == 64) {
    switch (mode) {
      case Mode::kDense: return launch_pair<64, 128, 64, Mode::kDense>(tq, tk, tv, p, st);
      case Mode::kSparse: return launch_pair<64, 128, 64, Mode::kSparse>(tq, tk, tv, p, st);
      default: return launch_pair<64, 128, 64, Mode::kCount>(tq, tk, tv, p, st);
    }
  }
  switch (mode) {
    case Mode::kDense: return launch_pair<128, 128, 128, Mode::kDense>(tq, tk, tv, p, st);
    case Mode::kSparse: return launch_pair<128, 128, 128, Mode::kSparse>(tq, tk, tv, p, st);
    default: return launch_pair<128, 128, 128, Mode::kCount>(tq, tk, tv, p, st);
  }
}

}  // namespace ssattn
