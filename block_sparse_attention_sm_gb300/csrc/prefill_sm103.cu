// Skip-softmax (BLASST) prefill forward for sm_103a.
//
// Method ("Skip-Softmax" design doc, §The online-softmax pass and §The skip
// test; BLASST summary, §Methodologie and §Kernel-ontwerp): one streaming
// pass over 128-key tiles; the scores S_j = Q K_j^T * scale always run on the
// tensor cores; when every row of a 128-row query block has
// exp(scale*(tile_max - m)) < lambda, the tile's exponentials and its P.V MMA
// are skipped and it adds nothing to l or O.
//
// Decisions first, values second.  With lambda <= 1 a skipped tile never
// raises a row's maximum, so the maximum m_r before tile j is the prefix
// maximum of the row's scores over tiles < j whatever was skipped, and every
// decision depends on the scores alone.  Each CTA therefore runs
//   a vote pass:    S_j for every tile into double-buffered TMEM, row maxima,
//                   the vote against the exact running maximum; no
//                   exponentials, so the score MMAs stream back to back;
//   a compute pass: over the kept tiles only, S_j again, P = exp2((S - m) *
//                   scale * log2e) with m the row's final maximum from the
//                   vote pass (so O never needs a rescale), O += P V_j.
// The kept set, the counters and O equal those of the one-pass definition;
// kept tiles pay their QK^T twice, skipped tiles once.  Very long keys are
// handled in runs of p.chunk_tiles (at most 2048) tiles: vote pass, then
// compute pass, per run, with O rescaled once when a later run raises a row
// maximum.  The dense path (lambda = 0) has no vote pass: one online pass
// with a lazily rescaled maximum.
//
// One CTA = two 128-row query blocks (t = 0, 1) of one (b, h_q), sharing every
// K/V tile; 384 threads (3 warpgroups; registers re-split with setmaxnreg):
//   warps 0-3 / 4-7  softmax of query block 0 / 1: thread = query row = TMEM
//                    lane.  Vote pass: loads the row's 128 scores, row
//                    maximum, vote (a bar.red.and over the block's 128
//                    threads).  Compute pass: writes P as bf16 over the first
//                    64 columns of S; epilogue O / l.
//   warp 8           TMA producer: both Q blocks, then one FIFO ring of
//                    tiles: K of every tile (vote pass), then K and V of the
//                    kept tiles (compute pass).
//   warps 9, 10      tcgen05 MMA issuers (one thread each; warp 10 also
//                    allocates TMEM).  Vote pass: S_0(i), S_1(i) into score
//                    buffer i % 2, one commit for both; the first chunk's
//                    even / odd tiles come from warp 10 / 9.  Compute pass:
//                    warp 10 issues block 0's PV_0(prev), S_0(u) ..., warp 9
//                    block 1's, each as its softmax frees S, so one block's
//                    softmax overlaps the other block's MMAs.
//                    S_t = Q_t K^T: SS form, both operands K-major, 128-byte
//                    swizzle.  O_t += P_t V: TS form, P_t from TMEM, V MN-major.
// TMEM (512 columns): S_0 [0,128), S_1 [128,256), O_0 [256, 256+d),
// O_1 [384, 384+d); the vote pass's second score buffers of the first chunk
// are O_0 / O_1 (the compute pass's first P.V overwrites them).  tcgen05 MMAs
// of a CTA execute in issue order, so an MMA issued after PV_t cannot
// overwrite P_t early, and a commit covers every MMA issued before it.
#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx_sm103.cuh"

namespace ssattn {

namespace {

constexpr float kRescaleLog2 = 8.0f;  // lazy-rescale slack of the dense path, exp2 domain
constexpr int kThreads = 384;         // three warpgroups
constexpr int kWarpLoad = 8, kWarpMma = 10;  // warp 11 idles
constexpr int kWarpMma2 = 9;  // MMA issuer of query block 1
// Register split: launched at 168 per thread (384 x 168 = 64512); the
// producer/MMA warpgroup drops to kRegsIssue and the two softmax warpgroups
// rise to kRegsSoftmax, with 128 x issue + 256 x softmax = 64512, i.e.
// exactly the launch pool.  The voting kernels' issuer walks the kept-tile
// masks and needs more than the dense kernel's.
constexpr int kLaunchRegs = 168;
template <Mode MODE>
constexpr int kRegsIssue = (MODE == Mode::kDense) ? 72 : 104;
template <Mode MODE>
constexpr int kRegsSoftmax = (kThreads * kLaunchRegs - 128 * kRegsIssue<MODE>) / 256;
static_assert(128 * kRegsIssue<Mode::kDense> + 256 * kRegsSoftmax<Mode::kDense> ==
                  kThreads * kLaunchRegs &&
              128 * kRegsIssue<Mode::kSparse> + 256 * kRegsSoftmax<Mode::kSparse> ==
                  kThreads * kLaunchRegs,
              "register split must equal the launch pool");
static_assert(kRegsSoftmax<Mode::kDense> % 8 == 0 && kRegsSoftmax<Mode::kSparse> % 8 == 0,
              "setmaxnreg takes multiples of 8");
constexpr int kMaskWords = kVoteChunkTiles / 32;  // mask capacity of one chunk

template <int D>
struct PrefillCfg {
  static constexpr int kChunks = D / 64;            // 128-byte swizzle chunks per row
  static constexpr int kTileBytes = kTile * D * 2;  // one 128 x D bf16 tile
  // One FIFO ring of tile slots for K and V: the vote pass streams K tiles
  // through every slot; the compute pass loads K(u), V(u), K(u'), V(u'), ...
  // and frees them in the same order (an MMA that reads V(u) is issued
  // before the one that reads K(u'), and MMAs complete in issue order).
  static constexpr int kRingSlots = (D == 128) ? 5 : 12;
  static constexpr int kQOff = 0;  // two query blocks
  static constexpr int kRingOff = kQOff + 2 * kTileBytes;
  static constexpr int kCtlOff = kRingOff + kRingSlots * kTileBytes;
  static constexpr int kCtlBytes = 2048;
  static constexpr int kSmemBytes = kCtlOff + kCtlBytes + 1024;  // + alignment slack
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
  static constexpr uint32_t kColS = 0;    // S_t at kColS + 128 t
  static constexpr uint32_t kColO = 256;  // O_t at kColO + 128 t
  static constexpr uint32_t kTmemCols = 512;
};

template <int NR>
struct PrefillCtl {
  uint64_t q_full;
  uint64_t r_full[NR], r_empty[NR];        // tile ring
  // Vote pass, per score buffer b (both blocks' S in it): one commit after
  // S_0 and S_1, and one release by the 8 softmax warps (the issuer stands in
  // for a block that has no tile there), so the issuer pays one wait and one
  // commit per tile pair.
  uint64_t s1_full[2], s1_empty[2];
  uint64_t s_full[2], p_full[2];           // compute pass: [block]
  // Per chunk parity: the 8 softmax warps are done voting.  Two barriers, so
  // that a reader one chunk behind (the V producer, when a chunk keeps no
  // tile) never sees a phase two chunks ahead.
  uint64_t votes_done[2];
  uint64_t mask_free[2];                   // per chunk parity: its 3 readers are done
  uint64_t o_done[2];                      // per block: its last P.V is done
  uint64_t c1_done;                        // per chunk: block 1's compute MMAs are done
  uint64_t mma_done[2];                    // per issuing thread, for teardown
  uint32_t tmem_base;
  int abort_flag;
  int n_loaded;  // ring entries whose copy has been issued (monotone)
  float red[2][2][4];
  uint32_t kmask[2][2][kMaskWords];  // kept tiles: [chunk parity][block][bit]
};

template <int D, Mode MODE>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const PrefillParams p) {
  using C = PrefillCfg<D>;
  constexpr int NR = C::kRingSlots;
  constexpr bool kPV = (MODE != Mode::kCount);
  constexpr bool kVote = (MODE != Mode::kDense);
  using Ctl = PrefillCtl<NR>;
  static_assert(sizeof(Ctl) <= C::kCtlBytes, "control block overflow");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem + C::kQOff;
  uint8_t* sR = smem + C::kRingOff;
  auto* ctl = reinterpret_cast<Ctl*>(smem + C::kCtlOff);
  volatile int* abort_flag = &ctl->abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // Work: query blocks 2*pr and 2*pr + 1 of head (b, h).  Causal: heaviest first.
  const int nP = (p.nQB + 1) / 2;
  const int x = blockIdx.x;
  const int bh = x / nP;
  const int ip = x - bh * nP;
  const int pr = p.causal ? (nP - 1 - ip) : ip;
  const int b = bh / p.Hq, h = bh - (bh / p.Hq) * p.Hq;
  const int kvh = h / p.G;
  const long off = static_cast<long>(p.Lk) - p.Lq;
  int r0[2], rows[2], n_t[2];
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    r0[t] = (2 * pr + t) * kTile;
    rows[t] = max(0, min(kTile, p.Lq - r0[t]));
    n_t[t] = (rows[t] > 0) ? p.nT : 0;
    if (p.causal && rows[t] > 0) {
      const long last = static_cast<long>(r0[t]) + rows[t] - 1 + off;  // last key of the last row
      n_t[t] = last < 0 ? 0 : min(p.nT, static_cast<int>(last / kTile) + 1);
    }
  }
  const int nmax = max(n_t[0], n_t[1]);

  // Vote pass whenever decisions are wanted (the dense instantiation is
  // launched only without debug outputs); the kept-tile masks are needed
  // only when a compute pass follows.
  constexpr bool vote_pass = kVote;
  constexpr bool use_masks = vote_pass && kPV;
  const int nchunks = vote_pass ? (nmax + p.chunk_tiles - 1) / p.chunk_tiles : (nmax > 0 ? 1 : 0);
  auto chunk_begin = [&](int c) { return vote_pass ? c * p.chunk_tiles : 0; };
  auto chunk_end = [&](int c) { return vote_pass ? min(nmax, (c + 1) * p.chunk_tiles) : nmax; };
  auto mask_word = [&](int c, int t, int w) -> uint32_t {
    return *reinterpret_cast<volatile uint32_t*>(&ctl->kmask[c & 1][t][w]);
  };
  // Is tile u (in chunk c) computed for block t?
  auto kept = [&](int c, int t, int u) -> bool {
    if (!use_masks) return u < n_t[t];
    const int r = u - c * p.chunk_tiles;
    return ((mask_word(c, t, r >> 5) >> (r & 31)) & 1u) != 0;
  };
  // First tile >= from in chunk c that block `which` (0, 1; 2 = either)
  // computes; the chunk end if none.
  auto next_kept = [&](int c, int which, int from) -> int {
    const int e = chunk_end(c);
    if (!use_masks) return (which == 2) ? from : (from < n_t[which] ? from : e);
    int u = from;
    while (u < e) {
      const int r = u - c * p.chunk_tiles;
      const int w = r >> 5;
      uint32_t bits = (which == 2) ? (mask_word(c, 0, w) | mask_word(c, 1, w)) : mask_word(c, which, w);
      bits >>= (r & 31);
      if (bits != 0u) return min(e, u + __ffs(bits) - 1);
      u += 32 - (r & 31);
    }
    return e;
  };

  if (tid == 0) {
    mbar_init(&ctl->q_full, 1);
    for (int s = 0; s < NR; ++s) {
      mbar_init(&ctl->r_full[s], 1);
      mbar_init(&ctl->r_empty[s], MODE == Mode::kDense ? 1 : 2);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&ctl->s1_full[t], 1);
      mbar_init(&ctl->s1_empty[t], 8);
      mbar_init(&ctl->s_full[t], 1);
      mbar_init(&ctl->p_full[t], 128);
    }
    mbar_init(&ctl->votes_done[0], 8);
    mbar_init(&ctl->votes_done[1], 8);
    mbar_init(&ctl->mask_free[0], 3);
    mbar_init(&ctl->mask_free[1], 3);
    mbar_init(&ctl->o_done[0], 1);
    mbar_init(&ctl->o_done[1], 1);
    mbar_init(&ctl->c1_done, 1);
    mbar_init(&ctl->mma_done[0], 1);
    mbar_init(&ctl->mma_done[1], 1);
    ctl->abort_flag = 0;
    ctl->n_loaded = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(&ctl->tmem_base, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  const int zk = b * p.Hkv + kvh;

  // Each warpgroup's code below runs to the end of the kernel under its own
  // register budget; the two paths meet only at the final named barrier.
  if (warp >= 8) {
  constexpr uint32_t kRegsDown = kRegsIssue<MODE>;
  setmaxnreg_dec<kRegsDown>();
  int n_issued = 0;  // producer bookkeeping for teardown: ring entries issued
  if (warp == kWarpLoad) {
    // ---------------------------------------------------------- TMA producer
    if (lane == 0 && nmax > 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      if (kPV) tma_prefetch_desc(&tmV);
      const int nq = (rows[0] > 0 ? 1 : 0) + (rows[1] > 0 ? 1 : 0);
      mbar_arrive_expect_tx(&ctl->q_full, nq * C::kTileBytes);
#pragma unroll
      for (int t = 0; t < 2; ++t)
        if (rows[t] > 0)
#pragma unroll
          for (int c = 0; c < C::kChunks; ++c)
            tma_load_3d(sQ + t * C::kTileBytes + c * 16384, &tmQ, &ctl->q_full, c * 64, r0[t], bh);
      // Next ring entry: tile u of K or V.
      auto load_tile = [&](const CUtensorMap* map, int u) -> bool {
        const int st = n_issued % NR;
        if (!mbar_wait(&ctl->r_empty[st], ((n_issued / NR) & 1) ^ 1, abort_flag)) return false;
        mbar_arrive_expect_tx(&ctl->r_full[st], C::kTileBytes);
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_3d(sR + st * C::kTileBytes + c * 16384, map, &ctl->r_full[st], c * 64,
                      u * kTile, zk);
        ++n_issued;
        *reinterpret_cast<volatile int*>(&ctl->n_loaded) = n_issued;
        return true;
      };
      bool ok = true;
      for (int c = 0; ok && c < nchunks; ++c) {
        if (vote_pass) {
          for (int u = chunk_begin(c); ok && u < chunk_end(c); ++u) ok = load_tile(&tmK, u);
          if (!kPV) continue;
          ok = ok && mbar_wait(&ctl->votes_done[c & 1], (c >> 1) & 1, abort_flag);
        }
        for (int u = next_kept(c, 2, chunk_begin(c)); ok && u < chunk_end(c); u = next_kept(c, 2, u + 1))
          ok = load_tile(&tmK, u) && load_tile(&tmV, u);
        if (use_masks) mbar_arrive(&ctl->mask_free[c & 1]);
      }
    }
  } else if (warp == kWarpMma || warp == kWarpMma2) {
    // ---------------------------------------------------------- MMA issuers
    // Issuing blocks until the tensor pipe takes each MMA, so the pipe idles
    // while its issuer waits or commits.  Two threads issue: warp 10 the
    // MMAs of query block 0, warp 9 those of block 1 (compute pass), and in
    // the first chunk's vote pass the even / odd tiles into score buffer
    // 0 / 1; one keeps the pipe fed while the other synchronises.  Later
    // chunks' vote passes (score buffer 0 only) are issued by warp 10.
    if (lane == 0 && nmax > 0) {
      const int tb = (warp == kWarpMma) ? 0 : 1;
      constexpr uint32_t idS = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t idO = idesc_bf16_f32(128, D, false, true);
      const uint32_t sQa = smem_u32(sQ), sRa = smem_u32(sR);
      // Descriptors are built once per operand tile and advanced by adding the
      // encoded (>>4) byte offset to the start-address field; shared-memory
      // offsets here stay far below the field's 2^18-byte range, so the add
      // never carries out of it.
      auto issue_s = [&](int t, int kst, uint32_t col) {
        const uint64_t dq = smem_desc(sQa + t * C::kTileBytes, 16, 1024);
        const uint64_t dk = smem_desc(sRa + kst * C::kTileBytes, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
          mma_bf16_ss(tmem + col, dq + koff, dk + koff, idS, kk > 0 ? 1u : 0u);
        }
      };
      auto issue_pv = [&](int t, int vst, uint32_t acc) {
        const uint64_t dv = smem_desc(sRa + vst * C::kTileBytes, 16384, 1024);
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          mma_bf16_ts(tmem + C::kColO + 128 * t, tmem + C::kColS + 128 * t + kk * 8,
                      dv + ((kk * 2048) >> 4), idO, (acc | kk) ? 1u : 0u);
      };
      // Voting kernels: a ring slot is free after two arrivals, one commit
      // per block whose MMAs read it; a block that reads it alone adds the
      // second arrival itself (after its wait for the slot's data, so in the
      // right phase).  Dense kernel: one thread issues every read, one commit.
      auto release = [&](int st, bool alone) {
        mma_commit(&ctl->r_empty[st]);
        if (MODE != Mode::kDense && alone) mbar_arrive(&ctl->r_empty[st]);
      };
      bool ok = mbar_wait(&ctl->q_full, 0, abort_flag);
      // Wait for ring entry e's data.  The two issuers consume different
      // subsets of the ring, so one may ask for an entry the producer has not
      // reached; a parity wait alone could then see the slot's previous
      // phase.  Waiting first until the copy of e has been issued pins the
      // slot's barrier to e's phase (e's slot cannot be reused before this
      // thread releases e).
      int seen_loaded = 0;  // last value of n_loaded this thread read
      auto ring_wait = [&](int e) -> bool {
        if (seen_loaded <= e) {
          seen_loaded = *reinterpret_cast<volatile int*>(&ctl->n_loaded);
          if (seen_loaded <= e) {
            const uint64_t t0 = globaltimer_ns();
            while ((seen_loaded = *reinterpret_cast<volatile int*>(&ctl->n_loaded)) <= e) {
              if (*abort_flag) return false;
              if (globaltimer_ns() - t0 > kWaitTimeoutNs) {
                *abort_flag = 1;
                return false;
              }
            }
          }
        }
        return mbar_wait(&ctl->r_full[e % NR], (e / NR) & 1, abort_flag);
      };
      // One vote-pass tile: ring entry `e`, score buffer `bsel`, `n` earlier uses of it.
      auto vote_tile = [&](int u, int e, int bsel, int n) -> bool {
        const int kst = e % NR;
        if (!ring_wait(e) || !mbar_wait(&ctl->s1_empty[bsel], (n & 1) ^ 1, abort_flag))
          return false;
        tc_fence_after();
        const uint32_t col = bsel ? C::kColO : C::kColS;
        if (u < n_t[0]) issue_s(0, kst, col);
        if (u < n_t[1]) issue_s(1, kst, col + 128);
        mma_commit(&ctl->s1_full[bsel]);
        release(kst, true);
        const uint32_t absent = (u < n_t[0] ? 0u : 4u) + (u < n_t[1] ? 0u : 4u);
        if (absent != 0u) mbar_arrive_cnt(&ctl->s1_empty[bsel], absent);
        return true;
      };
      int rseq = 0;    // ring entries of the chunks before (both threads track it)
      int s1cnt = 0;   // vote-pass uses of this thread's score buffer
      int scnt = 0;    // compute-pass S MMAs of block tb
      uint32_t o_acc = 0u;
      for (int c = 0; ok && c < nchunks; ++c) {
        const int cb = chunk_begin(c), ce = chunk_end(c);
        if (vote_pass) {
          // ---- vote pass: every tile, both blocks, double-buffered scores
          // Block 1's last compute MMAs of the previous chunk read its S
          // columns, which this chunk's scores overwrite.
          if (tb == 0 && kPV && c > 0 && !mbar_wait(&ctl->c1_done, (c - 1) & 1, abort_flag)) {
            ok = false;
            break;
          }
          for (int u = cb; ok && u < ce; ++u) {
            if (c == 0 ? ((u & 1) != tb) : (tb != 0)) continue;
            ok = vote_tile(u, rseq + (u - cb), c == 0 ? tb : 0, s1cnt);
            ++s1cnt;
          }
          rseq += ce - cb;
          if (!kPV || !ok) continue;
          if (!mbar_wait(&ctl->votes_done[c & 1], (c >> 1) & 1, abort_flag)) {
            ok = false;
            break;
          }
        }
        if constexpr (MODE == Mode::kDense) {
          // ---- dense: one thread issues both blocks' MMAs in the order
          // PV_0(i-1), S_0(i), PV_1(i-1), S_1(i), which keeps the two blocks'
          // softmaxes alternating (ring entries K(i), V(i); one trailing step).
          // A single consumer takes the ring in order: plain parity waits.
          if (tb == 0) {
            bool prevk[2] = {false, false};
            int prev_ve = 0;
            uint32_t oacc[2] = {0u, 0u};
            int sc[2] = {0, 0};
            for (int u = cb;; ++u) {
              const bool last = (u >= ce);
              const int ke = rseq + 2 * (u - cb), kst = ke % NR, vst = prev_ve % NR;
              bool k_ready = false, v_ready = false, any_pv = false;
#pragma unroll
              for (int t = 0; t < 2; ++t) {
                if (prevk[t]) {
                  if (!mbar_wait(&ctl->p_full[t], (sc[t] - 1) & 1, abort_flag) ||
                      (!v_ready && !mbar_wait(&ctl->r_full[vst], (prev_ve / NR) & 1, abort_flag))) {
                    ok = false;
                    break;
                  }
                  v_ready = true;
                  tc_fence_after();
                  issue_pv(t, vst, oacc[t]);
                  oacc[t] = 1u;
                  any_pv = true;
                }
                prevk[t] = !last && u < n_t[t];
                if (prevk[t]) {
                  if (!k_ready && !mbar_wait(&ctl->r_full[kst], (ke / NR) & 1, abort_flag)) {
                    ok = false;
                    break;
                  }
                  k_ready = true;
                  tc_fence_after();
                  issue_s(t, kst, C::kColS + 128 * t);
                  mma_commit(&ctl->s_full[t]);
                  ++sc[t];
                }
              }
              if (!ok) break;
              if (any_pv) release(vst, true);  // one thread covers both blocks' reads
              if (last) break;
              release(kst, true);
              prev_ve = ke + 1;
            }
            if (ok) mma_commit(&ctl->o_done[1]);
          }
        } else {
          // ---- compute pass of block tb over the tiles kept by either block
          // (ring entries K(u), V(u) in that order).
          bool have_prev = false, prev_alone = false;
          int prev_ve = 0;  // ring entry of the previous kept tile's V
          auto pv_prev = [&]() -> bool {
            const int vst = prev_ve % NR;
            if (!mbar_wait(&ctl->p_full[tb], (scnt - 1) & 1, abort_flag) || !ring_wait(prev_ve))
              return false;
            tc_fence_after();
            issue_pv(tb, vst, o_acc);
            o_acc = 1u;
            release(vst, prev_alone);
            return true;
          };
          int k = 0;
          for (int u = next_kept(c, 2, cb); ok && u < ce; u = next_kept(c, 2, u + 1), ++k) {
            if (!kept(c, tb, u)) continue;
            const int ke = rseq + 2 * k, kst = ke % NR;
            const bool alone = !kept(c, 1 - tb, u);
            if (have_prev && !pv_prev()) {
              ok = false;
              break;
            }
            if (!ring_wait(ke)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_s(tb, kst, C::kColS + 128 * tb);
            mma_commit(&ctl->s_full[tb]);
            release(kst, alone);
            ++scnt;
            have_prev = true;
            prev_ve = ke + 1;
            prev_alone = alone;
          }
          if (ok && have_prev && !pv_prev()) ok = false;
        }
        if (!ok) break;
        // the ring entries of this chunk's compute pass (count the whole list)
        for (int u = next_kept(c, 2, cb); u < ce; u = next_kept(c, 2, u + 1)) rseq += 2;
        if (tb == 1 && kPV && vote_pass && c + 1 < nchunks) mma_commit(&ctl->c1_done);
        if (use_masks) mbar_arrive(&ctl->mask_free[c & 1]);
      }
      // (Dense: warp 10 issued block 1's MMAs too and has committed its o_done.)
      if (kPV && ok && !(MODE == Mode::kDense && tb == 1)) mma_commit(&ctl->o_done[tb]);
      // Every MMA this thread issued must have finished before TMEM is freed.
      mma_commit(&ctl->mma_done[tb]);
      mbar_wait(&ctl->mma_done[tb], 0, nullptr);
    }
    __syncwarp();
  }
  // ------------------------------------------------------------ teardown (warps 8-11)
  if (warp == kWarpLoad && lane == 0 && *abort_flag) {
    // On an abort, let in-flight TMA writes land before shared memory is released.
    // The newest entry issued into slot s is the largest e < n with e % NR == s.
    if (nmax > 0) mbar_wait(&ctl->q_full, 0, nullptr);
    for (int s = 0; s < NR; ++s)
      if (n_issued > s)
        mbar_wait(&ctl->r_full[s], ((s + ((n_issued - 1 - s) / NR) * NR) / NR) & 1, nullptr);
  }
  __syncwarp();
  tc_fence_before();
  barrier_sync(1, kThreads);
  if (warp == kWarpMma) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  } else {
    // ---------------------------------------------------------- softmax (block t)
    constexpr uint32_t kRegsUp = kRegsSoftmax<MODE>;
    setmaxnreg_inc<kRegsUp>();
    const int t = warp >> 2;
    const int tid_t = tid & 127;
    const int row = tid_t;
    // per-block scalars (selected, not indexed, to keep them in registers)
    const int r0_t = t ? r0[1] : r0[0];
    const int rows_t = t ? rows[1] : rows[0];
    const int n_mine = t ? n_t[1] : n_t[0];
    const long grow = static_cast<long>(r0_t) + row;
    const bool row_valid = row < rows_t;
    long lim = static_cast<long>(p.Lk) - 1;  // last key index this row may see
    if (p.causal && grow + off < lim) lim = grow + off;
    if (!row_valid) lim = -1;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    const uint32_t colS = lane_base + C::kColS + 128 * t;
    const uint32_t colO = lane_base + C::kColO + 128 * t;
    const float sl2 = p.scale_log2;
    const long unit = static_cast<long>(bh) * p.nQB + 2 * pr + t;
    float m_true = -INFINITY, m_used = -INFINITY, l = 0.f;
    uint32_t skipped = 0;
    bool ok = true;
    int n1[2] = {0, 0}, n2 = 0;
    // Warp-uniform waits: tcgen05.ld/st are warp-collective, so a failed wait
    // ends the loop for the whole warp; the other warps then time out too.
    auto wwait = [&](uint64_t* bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag));
    };
    // Masked scores of tile i in registers (one TMEM round trip) and the row
    // maximum (four independent partial maxima).
    auto load_scores = [&](uint32_t col, int i, uint32_t (&sr)[128], bool want_max) -> float {
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32p(col + 32 * c, sr + 32 * c);
      tmem_wait_ld();
      const long k0 = static_cast<long>(i) * kTile;
      const bool full = (k0 + kTile - 1 <= lim);
      // last visible column of this tile for this row (-1: none), 32-bit
      const int vis = static_cast<int>(max(-1L, min(static_cast<long>(kTile - 1), lim - k0)));
      if (!full) {
#pragma unroll
        for (int e = 0; e < 128; ++e)
          if (e > vis) sr[e] = __float_as_uint(-INFINITY);
      }
      if (!want_max) return 0.f;
      float mx[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) mx[e] = -INFINITY;
#pragma unroll
      for (int e = 0; e < 64; ++e)
        mx[e & 3] = fmax3(mx[e & 3], __uint_as_float(sr[2 * e]), __uint_as_float(sr[2 * e + 1]));
      return fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
    };
    const uint32_t bar_id = 2 + t;

    for (int c = 0; c < nchunks; ++c) {
      const int cb = chunk_begin(c);
      const int ce = min(chunk_end(c), n_mine);
      if (vote_pass) {
        // ---------------------------------------------- vote pass (chunk c)
        bool mf_ok = true;
        if (use_masks && tid_t == 0) {
          // the chunk parity's masks are free once chunk c-2's readers are done
          if (c >= 2) mf_ok = mbar_wait(&ctl->mask_free[c & 1], ((c >> 1) - 1) & 1, abort_flag);
          for (int w = 0; w < kMaskWords; ++w) ctl->kmask[c & 1][t][w] = 0u;
        }
        // The block's four warps meet at named barrier 2 + t once per tile
        // (bar.red), and no thread may skip it: a failed wait is carried to
        // the barrier and the warps leave the loop together.
        for (int i = cb; i < ce; ++i) {
          const int bsel = (c == 0) ? (i & 1) : 0;
          const bool got = wwait(&ctl->s1_full[bsel], (bsel ? n1[1] : n1[0]) & 1);
          if (bsel) ++n1[1]; else ++n1[0];
          tc_fence_after();
          uint32_t sr[128];
          float tmax = -INFINITY;
          if (got) tmax = load_scores(lane_base + (bsel ? C::kColO : C::kColS) + 128 * t, i, sr, true);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&ctl->s1_empty[bsel]);

          // Skip vote: every row of the block must pass exp(scale*(tmax - m)) < lambda.
          // (The dense path runs the same reduction only to report margins.)
          float c_r = -INFINITY;  // a row with no visible key does not veto
          if (tmax != -INFINITY) c_r = (m_true == -INFINITY) ? INFINITY : tmax - m_true;
          const bool all_pass = named_bar_and(bar_id, 128, got && c_r < p.thr_raw);
          if (!all_pass && named_bar_or(bar_id, 128, !got)) {
            ok = false;
            break;
          }
          const bool skip = kVote && all_pass;
          if (p.margin != nullptr) {
            float cm = c_r;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, o));
            if (lane == 0) *reinterpret_cast<volatile float*>(&ctl->red[t][i & 1][warp & 3]) = cm;
            named_bar_sync(bar_id, 128);
            if (tid_t == 0) {
              const volatile float* rr = ctl->red[t][i & 1];
              const float cmax = fmaxf(fmaxf(rr[0], rr[1]), fmaxf(rr[2], rr[3]));
              p.margin[unit * p.nT + i] = (cmax == INFINITY) ? INFINITY : cmax * p.scale;
            }
          }
          m_true = fmaxf(m_true, tmax);
          if (tid_t == 0) {
            skipped += skip ? 1u : 0u;
            if (p.mask != nullptr) p.mask[unit * p.nT + i] = skip ? 1 : 0;
            if (use_masks && !skip) {
              const int r = i - cb;
              ctl->kmask[c & 1][t][r >> 5] |= 1u << (r & 31);
            }
          }
        }
        // Masks of this chunk are complete: the producers and the MMA issuer
        // may walk them; the block's own threads read them after the barrier.
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->votes_done[c & 1]);
        if (!kPV) {
          if (!ok) break;  // block-uniform: vote-pass failures leave through bar.red.or
          continue;
        }
        // Wait until both blocks have voted: a block with fewer (or no) tiles
        // would otherwise run ahead and arrive for chunk c + 2 while chunk c's
        // phase of the same barrier is still open, completing it early.
        if (!wwait(&ctl->votes_done[c & 1], (c >> 1) & 1)) ok = false;
        // Block-uniform exit on any failure so far; also publishes the masks.
        if (named_bar_or(bar_id, 128, !(ok && mf_ok))) {
          ok = false;
          break;
        }
        // Known maxima: the compute pass uses the exact row maximum so far.
        // A later chunk that raised it rescales O and l once (every earlier
        // P.V is complete: the vote-pass scores waited on came after them).
        float alpha = 1.f;
        bool need_rescale = false;
        if (m_used != -INFINITY && m_true > m_used) {
          alpha = ex2_approx((m_used - m_true) * sl2);
          need_rescale = true;
          l *= alpha;
        }
        if (__any_sync(0xffffffffu, need_rescale)) {
#pragma unroll 1
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t orr[32];
            tmem_ld32p(colO + cc * 32, orr);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) orr[e] = __float_as_uint(__uint_as_float(orr[e]) * alpha);
            tmem_st32p(colO + cc * 32, orr);
          }
          tmem_wait_st();
        }
        m_used = m_true;
      }

      // ---------------------------------------------- compute pass (chunk c)
      for (int i = next_kept(c, t, cb); i < ce; i = next_kept(c, t, i + 1)) {
        if (!wwait(&ctl->s_full[t], n2 & 1)) {
          ok = false;
          break;
        }
        ++n2;
        tc_fence_after();
        uint32_t sr[128];
        const float tmax = load_scores(colS, i, sr, !vote_pass);
        if (!vote_pass) {
          // Dense path: online maximum with a lazy O rescale.
          m_true = fmaxf(m_true, tmax);
          float alpha = 1.f;
          bool need_rescale = false;
          if (m_used == -INFINITY) {
            m_used = m_true;  // first visible key of this row: its O row is still zero
          } else if ((m_true - m_used) * sl2 > kRescaleLog2) {
            alpha = ex2_approx((m_used - m_true) * sl2);
            need_rescale = true;
            m_used = m_true;
            l *= alpha;
          }
          if (__any_sync(0xffffffffu, need_rescale)) {
            // O_t may be touched: the commit behind s_full covers P.V of the previous tile.
#pragma unroll
            for (int cc = 0; cc < D / 32; ++cc) {
              uint32_t orr[32];
              tmem_ld32p(colO + cc * 32, orr);
              tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 32; ++e) orr[e] = __float_as_uint(__uint_as_float(orr[e]) * alpha);
              tmem_st32p(colO + cc * 32, orr);
            }
          }
        }
        // P = exp2(s*scale*log2e - m) packed in place as bf16 pairs, then
        // written over the first 64 columns of S (already read).
        const float mb = (m_used == -INFINITY) ? 0.f : m_used * sl2;
        const uint64_t sl2x2 = f32x2(sl2, sl2), nmb = f32x2(-mb, -mb);
        uint64_t ls[2] = {0ull, 0ull};  // +0.0 pairs
#pragma unroll
        for (int cc = 0; cc < 64; ++cc) {
          const uint64_t xp = fma_f32x2(f32x2(__uint_as_float(sr[2 * cc]), __uint_as_float(sr[2 * cc + 1])),
                                        sl2x2, nmb);
          const float p0 = ex2_approx(f32x2_lo(xp));
          const float p1 = ex2_approx(f32x2_hi(xp));
          ls[cc & 1] = add_f32x2(ls[cc & 1], f32x2(p0, p1));
          sr[cc] = pack_bf16x2(p0, p1);
        }
        tmem_st32p(colS, sr);
        tmem_st32p(colS + 32, sr + 32);
        tmem_wait_st();
        const uint64_t lsum = add_f32x2(ls[0], ls[1]);
        l += f32x2_lo(lsum) + f32x2_hi(lsum);
        tc_fence_before();
        mbar_arrive(&ctl->p_full[t]);
      }
      // Another chunk's vote pass meets at the named barrier again: leave
      // together if any warp of the block failed.
      if (vote_pass && c + 1 < nchunks && named_bar_or(bar_id, 128, !ok)) {
        ok = false;
        break;
      }
      if (!ok) break;
    }

    if (kPV && ok && n_mine > 0) {
      ok = wwait(&ctl->o_done[t], 0);
      tc_fence_after();
    }
    if (kPV && ok && rows_t > 0) {
      // Epilogue: O / l -> bf16 (a row that saw no key writes zeros).
      const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
      __nv_bfloat16* orow = p.o + (static_cast<size_t>(bh) * p.Lq + grow) * D;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t orr[32];
        if (n_mine > 0) {
          tmem_ld32p(colO + c * 32, orr);
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
    if (tid_t == 0 && rows_t > 0) {
      if (p.counts != nullptr) p.counts[unit] = skipped;
      for (int j = n_mine; j < p.nT; ++j) {
        if (p.mask != nullptr) p.mask[unit * p.nT + j] = 2;
        if (p.margin != nullptr) p.margin[unit * p.nT + j] = NAN;
      }
    }
    __syncwarp();
    tc_fence_before();
    barrier_sync(1, kThreads);
    if (tid == 0 && *abort_flag) report_timeout(p.status);
  }
}

template <int D, Mode MODE>
cudaError_t launch_one(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const PrefillParams& p, cudaStream_t st) {
  using C = PrefillCfg<D>;
  auto* fn = prefill_kernel<D, MODE>;
  // The setmaxnreg split assumes the kernel is launched with exactly
  // kLaunchRegs registers per thread; with fewer, the softmax warpgroups'
  // increase could never be satisfied.  Refuse to launch in that case.
  static const int launch_regs = [fn] {
    cudaFuncAttributes attr{};
    return cudaFuncGetAttributes(&attr, fn) == cudaSuccess ? attr.numRegs : -1;
  }();
  if (launch_regs != kLaunchRegs) return cudaErrorInvalidKernelImage;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  const long ctas = static_cast<long>(p.B) * p.Hq * ((p.nQB + 1) / 2);
  fn<<<dim3(static_cast<unsigned>(ctas)), dim3(kThreads), C::kSmemBytes, st>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(int d, Mode mode, const CUtensorMap& tq, const CUtensorMap& tk,
                           const CUtensorMap& tv, const PrefillParams& p, cudaStream_t st) {
  if (d == 128) {
    switch (mode) {
      case Mode::kDense: return launch_one<128, Mode::kDense>(tq, tk, tv, p, st);
      case Mode::kSparse: return launch_one<128, Mode::kSparse>(tq, tk, tv, p, st);
      default: return launch_one<128, Mode::kCount>(tq, tk, tv, p, st);
    }
  }
  switch (mode) {
    case Mode::kDense: return launch_one<64, Mode::kDense>(tq, tk, tv, p, st);
    case Mode::kSparse: return launch_one<64, Mode::kSparse>(tq, tk, tv, p, st);
    default: return launch_one<64, Mode::kCount>(tq, tk, tv, p, st);
  }
}

}  // namespace ssattn
