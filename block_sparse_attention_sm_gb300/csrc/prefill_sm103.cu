// Skip-softmax (BLASST) prefill forward for sm_103a.
//
// Method ("Skip-Softmax" design doc, §The online-softmax pass and §The skip
// test; BLASST summary, §Methodologie and §Kernel-ontwerp): one streaming
// pass over 128-key tiles; the scores S_j = Q K_j^T * scale always run on the
// tensor cores; when every row of a 128-row query block has
// exp(scale*(tile_max - m)) < lambda, the tile's exponentials and its P.V MMA
// are skipped and it adds nothing to l or O.
//
// One CTA = two 128-row query blocks (t = 0, 1) of one (b, h_q), sharing every
// K/V tile; 384 threads (3 warpgroups; registers re-split with setmaxnreg):
//   warps 0-3 / 4-7  softmax of query block 0 / 1: thread = query row = TMEM
//                    lane.  It loads its 128 scores from TMEM once, takes the
//                    row maximum, votes (a bar.red.and over the block's 128
//                    threads) and, for kept tiles, writes P as bf16 over the
//                    first 64 columns of S; lazy O rescale; epilogue O / l.
//   warp 8           TMA producer: both Q blocks, then the K ring.
//   warp 9           TMA producer: the V ring.
//   warp 10          TMEM allocator + single-thread tcgen05 MMA issuer, in the
//                    order ... PV_0(i-1), S_0(i), PV_1(i-1), S_1(i) ... so one
//                    block's softmax overlaps the other block's MMAs.
//                    S_t = Q_t K^T: SS form, both operands K-major, 128-byte
//                    swizzle.  O_t += P_t V: TS form, P_t from TMEM, V MN-major.
// TMEM (512 columns): S_0 [0,128), S_1 [128,256) (P_t in the first 64 columns
// of S_t), O_0 [256, 256+d), O_1 [384, 384+d).  tcgen05 MMAs of a CTA execute
// in issue order, so S_t(i+1) (issued after PV_t(i)) cannot overwrite P_t(i)
// early, and the commit after S_t(i+1) also covers PV_t(i).
//
// Exactness of the decisions: the vote uses the true running maximum
// (max over every earlier tile).  The exponentials use m_used, which only
// follows it when it has grown by more than 2^8 in the exp2 domain (then O and
// l are rescaled); O / l is the same either way.
#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx_sm103.cuh"

namespace ssattn {

namespace {

constexpr float kRescaleLog2 = 8.0f;  // lazy-rescale slack, exp2 domain
constexpr int kThreads = 384;         // three warpgroups
constexpr int kWarpK = 8, kWarpV = 9, kWarpMma = 10;  // warp 11 idles
// Register split: launched at 168 per thread (384 x 168 = 64512); the
// producer/MMA warpgroup drops to 56 and the two softmax warpgroups rise to
// 224: 128 x 56 + 256 x 224 = 64512, i.e. exactly the launch pool.
constexpr int kLaunchRegs = 168, kRegsIssue = 56, kRegsSoftmax = 224;
static_assert(128 * kRegsIssue + 256 * kRegsSoftmax == kThreads * kLaunchRegs,
              "register split must equal the launch pool");

template <int D>
struct PrefillCfg {
  static constexpr int kChunks = D / 64;            // 128-byte swizzle chunks per row
  static constexpr int kTileBytes = kTile * D * 2;  // one 128 x D bf16 tile
  static constexpr int kKStages = (D == 128) ? 3 : 4;
  static constexpr int kVStages = (D == 128) ? 2 : 4;
  static constexpr int kQOff = 0;  // two query blocks
  static constexpr int kKOff = kQOff + 2 * kTileBytes;
  static constexpr int kVOff = kKOff + kKStages * kTileBytes;
  static constexpr int kCtlOff = kVOff + kVStages * kTileBytes;
  static constexpr int kCtlBytes = 1024;
  static constexpr int kSmemBytes = kCtlOff + kCtlBytes + 1024;  // + alignment slack
  static constexpr uint32_t kColS = 0;    // S_t at kColS + 128 t
  static constexpr uint32_t kColO = 256;  // O_t at kColO + 128 t
  static constexpr uint32_t kTmemCols = 512;
};

template <int NK, int NV>
struct PrefillCtl {
  uint64_t q_full;
  uint64_t k_full[NK], k_empty[NK];
  uint64_t v_full[NV], v_empty[NV];
  uint64_t s_full[2], p_full[2];
  uint64_t o_done;
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort_flag;
  int dec[2];
  float red[2][2][4];
};

template <int D, Mode MODE>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const PrefillParams p) {
  using C = PrefillCfg<D>;
  constexpr int NK = C::kKStages, NV = C::kVStages;
  constexpr bool kPV = (MODE != Mode::kCount);
  constexpr bool kVote = (MODE != Mode::kDense);
  using Ctl = PrefillCtl<NK, NV>;
  static_assert(sizeof(Ctl) <= C::kCtlBytes, "control block overflow");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem + C::kQOff;
  uint8_t* sK = smem + C::kKOff;
  uint8_t* sV = smem + C::kVOff;
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
    for (int t = 0; t < 2; ++t) {
      mbar_init(&ctl->s_full[t], 1);
      mbar_init(&ctl->p_full[t], 128);
    }
    mbar_init(&ctl->o_done, 1);
    mbar_init(&ctl->mma_done, 1);
    ctl->abort_flag = 0;
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
  setmaxnreg_dec<kRegsIssue>();
  int n_k_issued = 0, n_v_issued = 0;  // producer bookkeeping for teardown
  if (warp == kWarpK) {
    // ---------------------------------------------------------- Q + K producer
    if (lane == 0 && nmax > 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      const int nq = (rows[0] > 0 ? 1 : 0) + (rows[1] > 0 ? 1 : 0);
      mbar_arrive_expect_tx(&ctl->q_full, nq * C::kTileBytes);
#pragma unroll
      for (int t = 0; t < 2; ++t)
        if (rows[t] > 0)
#pragma unroll
          for (int c = 0; c < C::kChunks; ++c)
            tma_load_3d(sQ + t * C::kTileBytes + c * 16384, &tmQ, &ctl->q_full, c * 64, r0[t], bh);
      for (int i = 0; i < nmax; ++i) {
        const int st = i % NK;
        if (!mbar_wait(&ctl->k_empty[st], ((i / NK) & 1) ^ 1, abort_flag)) break;
        mbar_arrive_expect_tx(&ctl->k_full[st], C::kTileBytes);
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_3d(sK + st * C::kTileBytes + c * 16384, &tmK, &ctl->k_full[st], c * 64,
                      i * kTile, zk);
        n_k_issued = i + 1;
      }
    }
  } else if (warp == kWarpV) {
    // ---------------------------------------------------------- V producer
    if (kPV && lane == 0 && nmax > 0) {
      tma_prefetch_desc(&tmV);
      for (int i = 0; i < nmax; ++i) {
        const int st = i % NV;
        if (!mbar_wait(&ctl->v_empty[st], ((i / NV) & 1) ^ 1, abort_flag)) break;
        mbar_arrive_expect_tx(&ctl->v_full[st], C::kTileBytes);
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_3d(sV + st * C::kTileBytes + c * 16384, &tmV, &ctl->v_full[st], c * 64,
                      i * kTile, zk);
        n_v_issued = i + 1;
      }
    }
  } else if (warp == kWarpMma) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0 && nmax > 0) {
      constexpr uint32_t idS = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t idO = idesc_bf16_f32(128, D, false, true);
      const uint32_t sQa = smem_u32(sQ), sKa = smem_u32(sK), sVa = smem_u32(sV);
      // Descriptors are built once per operand tile and advanced by adding the
      // encoded (>>4) byte offset to the start-address field; shared-memory
      // offsets here stay far below the field's 2^18-byte range, so the add
      // never carries out of it.
      auto issue_s = [&](int t, int kst) {
        const uint64_t dq = smem_desc(sQa + t * C::kTileBytes, 16, 1024);
        const uint64_t dk = smem_desc(sKa + kst * C::kTileBytes, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = ((kk >> 2) * 16384 + (kk & 3) * 32) >> 4;
          mma_bf16_ss(tmem + C::kColS + 128 * t, dq + koff, dk + koff, idS, kk > 0 ? 1u : 0u);
        }
      };
      auto issue_pv = [&](int t, int vst, uint32_t acc) {
        const uint64_t dv = smem_desc(sVa + vst * C::kTileBytes, 16384, 1024);
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          mma_bf16_ts(tmem + C::kColO + 128 * t, tmem + C::kColS + 128 * t + kk * 8,
                      dv + ((kk * 2048) >> 4), idO, (acc | kk) ? 1u : 0u);
      };
      bool ok = mbar_wait(&ctl->q_full, 0, abort_flag) && mbar_wait(&ctl->k_full[0], 0, abort_flag);
      uint32_t o_acc[2] = {0u, 0u};
      if (ok) {
        tc_fence_after();
#pragma unroll
        for (int t = 0; t < 2; ++t)
          if (n_t[t] > 0) {
            issue_s(t, 0);
            mma_commit(&ctl->s_full[t]);
          }
        mma_commit(&ctl->k_empty[0]);
      }
      for (int i = 1; ok && i <= nmax; ++i) {
        const int kst = i % NK, vst = (i - 1) % NV;
        bool k_ready = false, v_ready = false, any_pv = false;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (i - 1 < n_t[t]) {
            // block t has read S_t(i-1) (and written P_t(i-1) if kept)
            if (!mbar_wait(&ctl->p_full[t], (i - 1) & 1, abort_flag)) {
              ok = false;
              break;
            }
            if (kPV && *reinterpret_cast<volatile int*>(&ctl->dec[t])) {
              if (!v_ready) {
                if (!mbar_wait(&ctl->v_full[vst], ((i - 1) / NV) & 1, abort_flag)) {
                  ok = false;
                  break;
                }
                v_ready = true;
              }
              tc_fence_after();
              issue_pv(t, vst, o_acc[t]);
              o_acc[t] = 1u;
              any_pv = true;
            }
          }
          if (i < n_t[t]) {
            if (!k_ready) {
              if (!mbar_wait(&ctl->k_full[kst], (i / NK) & 1, abort_flag)) {
                ok = false;
                break;
              }
              k_ready = true;
            }
            tc_fence_after();
            issue_s(t, kst);
            mma_commit(&ctl->s_full[t]);
          }
        }
        if (!ok) break;
        if (k_ready) mma_commit(&ctl->k_empty[kst]);
        if (kPV) {
          // V(i-1) is free once the MMAs reading it are done (or, if no block
          // kept the tile, once its copy has landed).
          if (any_pv) {
            mma_commit(&ctl->v_empty[vst]);
          } else {
            if (!v_ready && !mbar_wait(&ctl->v_full[vst], ((i - 1) / NV) & 1, abort_flag)) {
              ok = false;
              break;
            }
            mbar_arrive(&ctl->v_empty[vst]);
          }
        }
      }
      if (ok) mma_commit(&ctl->o_done);
    }
    __syncwarp();
  }
  // ------------------------------------------------------------ teardown (warps 8-11)
  if (warp == kWarpMma && lane == 0 && nmax > 0) {
    // Every MMA this thread issued must have finished before TMEM is freed.
    mma_commit(&ctl->mma_done);
    mbar_wait(&ctl->mma_done, 0, nullptr);
  }
  if ((warp == kWarpK || warp == kWarpV) && lane == 0 && *abort_flag) {
    // On an abort, let in-flight TMA writes land before shared memory is released.
    // The newest load issued into stage s is the largest i < n with i % stages == s.
    if (warp == kWarpK) {
      if (nmax > 0) mbar_wait(&ctl->q_full, 0, nullptr);
      for (int s = 0; s < NK; ++s)
        if (n_k_issued > s)
          mbar_wait(&ctl->k_full[s], ((s + ((n_k_issued - 1 - s) / NK) * NK) / NK) & 1, nullptr);
    } else {
      for (int s = 0; s < NV; ++s)
        if (n_v_issued > s)
          mbar_wait(&ctl->v_full[s], ((s + ((n_v_issued - 1 - s) / NV) * NV) / NV) & 1, nullptr);
    }
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
    setmaxnreg_inc<kRegsSoftmax>();
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
    // Warp-uniform waits: tcgen05.ld/st are warp-collective, so a failed wait
    // ends the loop for the whole warp; the other warps then time out too.
    auto wwait = [&](uint64_t* bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag));
    };

    // Vote path: the block's four warps meet at named barrier 2 + t once per
    // tile (bar.red), and no thread may skip it -- a failed wait is carried
    // to the barrier and the warps leave the loop together.  The dense path
    // has no barrier inside the loop and leaves on its own.
    const bool team = kVote || p.margin != nullptr;
    const uint32_t bar_id = 2 + t;
    for (int i = 0; i < n_mine; ++i) {
      const bool got = wwait(&ctl->s_full[t], i & 1);
      if (!got && !team) {
        ok = false;
        break;
      }
      tc_fence_after();
      const long k0 = static_cast<long>(i) * kTile;
      const bool full = (k0 + kTile - 1 <= lim);
      // last visible column of this tile for this row (-1: none), 32-bit
      const int vis = static_cast<int>(max(-1L, min(static_cast<long>(kTile - 1), lim - k0)));

      // All 128 scores of the row in registers (one TMEM round trip); masked
      // keys become -inf; four independent partial maxima.
      uint32_t sr[128];
      if (got) {
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32p(colS + 32 * c, sr + 32 * c);
        tmem_wait_ld();
      } else {
#pragma unroll
        for (int e = 0; e < 128; ++e) sr[e] = __float_as_uint(-INFINITY);
      }
      float mx[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) mx[e] = -INFINITY;
      if (full) {
#pragma unroll
        for (int e = 0; e < 128; ++e) mx[e & 3] = fmaxf(mx[e & 3], __uint_as_float(sr[e]));
      } else {
#pragma unroll
        for (int e = 0; e < 128; ++e) {
          if (e > vis) sr[e] = __float_as_uint(-INFINITY);
          mx[e & 3] = fmaxf(mx[e & 3], __uint_as_float(sr[e]));
        }
      }
      const float tmax = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));

      // Skip vote: every row of the block must pass exp(scale*(tmax - m)) < lambda.
      // (The dense path runs the same reduction only to report margins.)
      bool skip = false;
      if (team) {
        float c_r = -INFINITY;  // a row with no visible key does not veto
        if (tmax != -INFINITY) c_r = (m_true == -INFINITY) ? INFINITY : tmax - m_true;
        const bool all_pass = named_bar_and(bar_id, 128, got && c_r < p.thr_raw);
        if (!all_pass && named_bar_or(bar_id, 128, !got)) {
          ok = false;
          break;
        }
        skip = kVote && all_pass;
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
      }
      m_true = fmaxf(m_true, tmax);
      if (tid_t == 0) {
        skipped += skip ? 1u : 0u;
        if (p.mask != nullptr) p.mask[unit * p.nT + i] = skip ? 1 : 0;
      }

      if (kPV && !skip) {
        // O_t may be touched: the commit behind s_full covers P.V of tile i-1.
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
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t orr[32];
            tmem_ld32p(colO + c * 32, orr);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) orr[e] = __float_as_uint(__uint_as_float(orr[e]) * alpha);
            tmem_st32p(colO + c * 32, orr);
          }
        }
        // P = exp2(s*scale*log2e - m) packed in place as bf16 pairs, then
        // written over the first 64 columns of S (already read).
        const float mb = (m_used == -INFINITY) ? 0.f : m_used * sl2;
        float ls[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) ls[e] = 0.f;
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const float p0 = ex2_approx(fmaf(__uint_as_float(sr[2 * c]), sl2, -mb));
          const float p1 = ex2_approx(fmaf(__uint_as_float(sr[2 * c + 1]), sl2, -mb));
          ls[c & 3] += p0 + p1;
          sr[c] = pack_bf16x2(p0, p1);
        }
        tmem_st32p(colS, sr);
        tmem_st32p(colS + 32, sr + 32);
        tmem_wait_st();
        l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
      }
      tc_fence_before();
      if (tid_t == 0) *reinterpret_cast<volatile int*>(&ctl->dec[t]) = skip ? 0 : 1;
      mbar_arrive(&ctl->p_full[t]);
    }

    if (kPV && ok && n_mine > 0) {
      ok = wwait(&ctl->o_done, 0);
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
