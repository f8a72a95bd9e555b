// Skip-softmax (BLASST) prefill forward for sm_103a.
//
// Method ("Skip-Softmax" design doc, §The online-softmax pass and §The skip
// test; BLASST summary, §Methodologie and §Kernel-ontwerp): one streaming
// pass over 128-key tiles; the scores S_j = Q K_j^T * scale always run on the
// tensor cores; when every row of the 128-row query block has
// exp(scale*(tile_max - m)) < lambda the tile's exponentials and its P.V MMA
// are skipped and it adds nothing to l or O.
//
// One CTA = one (b, h_q, 128-row query block); 192 threads:
//   warps 0-3  softmax: thread t owns query row t (TMEM lane t): tile max,
//              vote (per-warp __all_sync, combined across the four warps
//              through shared memory and an mbarrier), exponentials,
//              P -> TMEM, lazy O rescale, epilogue O / l -> bf16.
//   warp 4     TMA producer: Q once, then K_j / V_j into a ring of stages.
//   warp 5     TMEM allocator + single-thread tcgen05 MMA issuer:
//              S_j = Q K_j^T (SS form, K-major operands) and, for kept tiles,
//              O += P_j V_j (TS form: P from TMEM, V MN-major from smem).
// TMEM (512 columns): S double buffer [0,256), P double buffer (packed bf16)
// [256,384), O [384, 384+d).
//
// Exactness of the decisions: the vote uses the true running maximum
// m_true (max over every earlier tile).  The exponentials use m_used, which
// only follows m_true when it has grown by more than 2^8 in the exp2 domain
// (then O and l are rescaled); O / l is the same either way.
#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx_sm103.cuh"

namespace ssattn {

namespace {

constexpr float kRescaleLog2 = 8.0f;  // lazy-rescale slack, exp2 domain

template <int D>
struct PrefillCfg {
  static constexpr int kChunks = D / 64;            // 128-byte swizzle chunks per row
  static constexpr int kTileBytes = kTile * D * 2;  // one 128 x D bf16 tile
  static constexpr int kStages = (D == 128) ? 3 : 4;
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + kTileBytes;
  static constexpr int kVOff = kKOff + kStages * kTileBytes;
  static constexpr int kCtlOff = kVOff + kStages * kTileBytes;
  static constexpr int kCtlBytes = 512;
  static constexpr int kSmemBytes = kCtlOff + kCtlBytes + 1024;  // + alignment slack
  static constexpr uint32_t kColS = 0;
  static constexpr uint32_t kColP = 256;
  static constexpr uint32_t kColO = 384;
  static constexpr uint32_t kTmemCols = 512;
};

template <int NS>
struct PrefillCtl {
  uint64_t q_full;
  uint64_t k_full[NS], k_empty[NS], v_full[NS], v_empty[NS];
  uint64_t s_full[2], s_empty[2], p_full[2], pv_done[2];
  uint64_t vote_bar[2];  // one arrival per softmax warp per tile
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort_flag;
  int dec[2];
  int verdict[2][4];
  float red[2][4];
};

template <int D, Mode MODE>
__global__ void __launch_bounds__(192, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const PrefillParams p) {
  using C = PrefillCfg<D>;
  constexpr int NS = C::kStages;
  constexpr bool kPV = (MODE != Mode::kCount);
  constexpr bool kVote = (MODE != Mode::kDense);
  static_assert(sizeof(PrefillCtl<NS>) <= C::kCtlBytes, "control block overflow");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem + C::kQOff;
  uint8_t* sK = smem + C::kKOff;
  uint8_t* sV = smem + C::kVOff;
  auto* ctl = reinterpret_cast<PrefillCtl<NS>*>(smem + C::kCtlOff);
  volatile int* abort_flag = &ctl->abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // Unit: (b, h_q, query block).  Causal: heaviest blocks of a head first.
  const int x = blockIdx.x;
  const int bh = x / p.nQB;
  const int i_qb = x - bh * p.nQB;
  const int qb = p.causal ? (p.nQB - 1 - i_qb) : i_qb;
  const int b = bh / p.Hq, h = bh - (bh / p.Hq) * p.Hq;
  const int kvh = h / p.G;
  const int r0 = qb * kTile;
  const int rows = min(kTile, p.Lq - r0);
  const long off = static_cast<long>(p.Lk) - p.Lq;
  int n_tiles = p.nT;
  if (p.causal) {
    const long last = static_cast<long>(r0) + rows - 1 + off;  // last key seen by the last row
    n_tiles = last < 0 ? 0 : min(p.nT, static_cast<int>(last / kTile) + 1);
  }
  const long unit = static_cast<long>(bh) * p.nQB + qb;

  if (tid == 0) {
    mbar_init(&ctl->q_full, 1);
    for (int s = 0; s < NS; ++s) {
      mbar_init(&ctl->k_full[s], 1);
      mbar_init(&ctl->k_empty[s], 1);
      mbar_init(&ctl->v_full[s], 1);
      mbar_init(&ctl->v_empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&ctl->s_full[s], 1);
      mbar_init(&ctl->s_empty[s], 128);
      mbar_init(&ctl->p_full[s], 128);
      mbar_init(&ctl->pv_done[s], 1);
      mbar_init(&ctl->vote_bar[s], 4);
    }
    mbar_init(&ctl->mma_done, 1);
    ctl->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(&ctl->tmem_base, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;

  int n_k_issued = 0, n_v_issued = 0;  // producer bookkeeping for teardown

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && n_tiles > 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      if (kPV) tma_prefetch_desc(&tmV);
      const int zk = b * p.Hkv + kvh;
      mbar_arrive_expect_tx(&ctl->q_full, C::kTileBytes);
#pragma unroll
      for (int c = 0; c < C::kChunks; ++c)
        tma_load_3d(sQ + c * 16384, &tmQ, &ctl->q_full, c * 64, r0, bh);
      for (int i = 0; i < n_tiles; ++i) {
        const int st = i % NS;
        const uint32_t ph = (i / NS) & 1;
        if (!mbar_wait(&ctl->k_empty[st], ph ^ 1, abort_flag)) break;
        mbar_arrive_expect_tx(&ctl->k_full[st], C::kTileBytes);
#pragma unroll
        for (int c = 0; c < C::kChunks; ++c)
          tma_load_3d(sK + st * C::kTileBytes + c * 16384, &tmK, &ctl->k_full[st], c * 64,
                      i * kTile, zk);
        n_k_issued = i + 1;
        if (kPV) {
          if (!mbar_wait(&ctl->v_empty[st], ph ^ 1, abort_flag)) break;
          mbar_arrive_expect_tx(&ctl->v_full[st], C::kTileBytes);
#pragma unroll
          for (int c = 0; c < C::kChunks; ++c)
            tma_load_3d(sV + st * C::kTileBytes + c * 16384, &tmV, &ctl->v_full[st], c * 64,
                        i * kTile, zk);
          n_v_issued = i + 1;
        }
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n_tiles > 0) {
      constexpr uint32_t idS = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t idO = idesc_bf16_f32(128, D, false, true);
      const uint32_t sQa = smem_u32(sQ), sKa = smem_u32(sK), sVa = smem_u32(sV);
      bool ok = mbar_wait(&ctl->q_full, 0, abort_flag);
      uint32_t o_acc = 0;
      for (int i = 0; ok && i <= n_tiles; ++i) {
        if (i < n_tiles) {
          const int st = i % NS;
          const uint32_t ph = (i / NS) & 1;
          const int sb = i & 1;
          const uint32_t sph = (i >> 1) & 1;
          if (!mbar_wait(&ctl->k_full[st], ph, abort_flag) ||
              !mbar_wait(&ctl->s_empty[sb], sph ^ 1, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t kbase = sKa + st * C::kTileBytes;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t koff = (kk >> 2) * 16384 + (kk & 3) * 32;
            mma_bf16_ss(tmem + C::kColS + sb * 128, smem_desc(sQa + koff, 16, 1024),
                        smem_desc(kbase + koff, 16, 1024), idS, kk > 0 ? 1u : 0u);
          }
          mma_commit(&ctl->s_full[sb]);
          mma_commit(&ctl->k_empty[st]);
        }
        if (kPV && i >= 1) {
          const int t = i - 1;
          const int pb = t & 1;
          const int vst = t % NS;
          if (!mbar_wait(&ctl->p_full[pb], (t >> 1) & 1, abort_flag) ||
              !mbar_wait(&ctl->v_full[vst], (t / NS) & 1, abort_flag)) {
            ok = false;
            break;
          }
          const int keep = *reinterpret_cast<volatile int*>(&ctl->dec[pb]);
          if (keep) {
            tc_fence_after();
            const uint32_t vbase = sVa + vst * C::kTileBytes;
#pragma unroll
            for (int kk = 0; kk < kTile / 16; ++kk)
              mma_bf16_ts(tmem + C::kColO, tmem + C::kColP + pb * 64 + kk * 8,
                          smem_desc(vbase + kk * 2048, 16384, 1024), idO, (o_acc | kk) ? 1u : 0u);
            o_acc = 1;
            mma_commit(&ctl->pv_done[pb]);
            mma_commit(&ctl->v_empty[vst]);
          } else {
            mbar_arrive(&ctl->pv_done[pb]);
            mbar_arrive(&ctl->v_empty[vst]);
          }
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int row = tid;
    const long grow = static_cast<long>(r0) + row;
    const bool row_valid = row < rows;
    long lim = static_cast<long>(p.Lk) - 1;  // last key index this row may see
    if (p.causal && grow + off < lim) lim = grow + off;
    if (!row_valid) lim = -1;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const float sl2 = p.scale_log2;
    float m_true = -INFINITY, m_used = -INFINITY, l = 0.f;
    uint32_t skipped = 0;
    bool ok = true;

    // Waits are made warp-uniform so that the warp-collective tcgen05.ld/st
    // below never run with part of a warp gone; a failed wait ends the loop
    // for the whole warp, and the other warps time out on their own waits.
    auto wwait = [&](uint64_t* bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag));
    };

    for (int i = 0; i < n_tiles; ++i) {
      const int sb = i & 1;
      if (!wwait(&ctl->s_full[sb], (i >> 1) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32p(lane_base + C::kColS + sb * 128 + c * 32, sr + c * 32);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&ctl->s_empty[sb]);

      // Mask (causal / tails / padding rows) and the row's tile maximum.
      const long k0 = static_cast<long>(i) * kTile;
      float tmax = -INFINITY;
      if (k0 + kTile - 1 <= lim) {
#pragma unroll
        for (int c = 0; c < 128; ++c) tmax = fmaxf(tmax, __uint_as_float(sr[c]));
      } else {
#pragma unroll
        for (int c = 0; c < 128; ++c) {
          const float sv = (k0 + c <= lim) ? __uint_as_float(sr[c]) : -INFINITY;
          sr[c] = __float_as_uint(sv);
          tmax = fmaxf(tmax, sv);
        }
      }

      // Skip vote: every row must pass exp(scale*(tile_max - m)) < lambda.
      // (The dense path runs the same reduction only to report margins.)
      bool skip = false;
      if (kVote || p.margin != nullptr) {
        float c_r = -INFINITY;  // a row with no visible key does not veto
        if (tmax != -INFINITY) c_r = (m_true == -INFINITY) ? INFINITY : tmax - m_true;
        const bool warp_pass = __all_sync(0xffffffffu, c_r < p.thr_raw);
        float cm = c_r;
        if (p.margin != nullptr) {
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, o));
        }
        // Combine the four warps' verdicts through shared memory and an
        // mbarrier (double-buffered by tile parity; a warp cannot reach tile
        // i+2 before every warp has read tile i's verdicts).
        const int vb = i & 1;
        if (lane == 0) {
          *reinterpret_cast<volatile int*>(&ctl->verdict[vb][warp]) = warp_pass ? 1 : 0;
          *reinterpret_cast<volatile float*>(&ctl->red[vb][warp]) = cm;
          mbar_arrive(&ctl->vote_bar[vb]);
        }
        if (!wwait(&ctl->vote_bar[vb], (i >> 1) & 1)) {
          ok = false;
          break;
        }
        const volatile int* vv = ctl->verdict[vb];
        skip = kVote && vv[0] && vv[1] && vv[2] && vv[3];
        if (tid == 0 && p.margin != nullptr) {
          const volatile float* rr = ctl->red[vb];
          const float cmax = fmaxf(fmaxf(rr[0], rr[1]), fmaxf(rr[2], rr[3]));
          p.margin[unit * p.nT + i] = (cmax == INFINITY) ? INFINITY : cmax * p.scale;
        }
      }
      m_true = fmaxf(m_true, tmax);
      if (tid == 0) {
        skipped += skip ? 1u : 0u;
        if (p.mask != nullptr) p.mask[unit * p.nT + i] = skip ? 1 : 0;
      }
      if constexpr (!kPV) continue;

      const int pb = i & 1;
      // P buffer pb (and its decision slot) is free once P.V of tile i-2 is done.
      if (i >= 2 && !wwait(&ctl->pv_done[pb], ((i - 2) >> 1) & 1)) {
        ok = false;
        break;
      }
      if (!skip) {
        float alpha = 1.f;
        bool need_rescale = false;
        if (m_used == -INFINITY) {
          m_used = m_true;  // first visible key of this row: O row is still zero
        } else if ((m_true - m_used) * sl2 > kRescaleLog2) {
          alpha = ex2_approx((m_used - m_true) * sl2);
          need_rescale = true;
          m_used = m_true;
          l *= alpha;
        }
        if (__any_sync(0xffffffffu, need_rescale)) {
          // O may only be touched once every earlier P.V has landed.
          if (i >= 1 && !wwait(&ctl->pv_done[(i - 1) & 1], ((i - 1) >> 1) & 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t orr[32];
            tmem_ld32p(lane_base + C::kColO + c * 32, orr);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) orr[e] = __float_as_uint(__uint_as_float(orr[e]) * alpha);
            tmem_st32p(lane_base + C::kColO + c * 32, orr);
          }
        }
        const float mb = (m_used == -INFINITY) ? 0.f : m_used * sl2;
        float lsum = 0.f;
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const float p0 = ex2_approx(fmaf(__uint_as_float(sr[2 * c]), sl2, -mb));
          const float p1 = ex2_approx(fmaf(__uint_as_float(sr[2 * c + 1]), sl2, -mb));
          lsum += p0 + p1;
          sr[c] = pack_bf16x2(p0, p1);
        }
        l += lsum;
        tmem_st32p(lane_base + C::kColP + pb * 64, sr);
        tmem_st32p(lane_base + C::kColP + pb * 64 + 32, sr + 32);
        tmem_wait_st();
      }
      tc_fence_before();
      if (tid == 0) *reinterpret_cast<volatile int*>(&ctl->dec[pb]) = skip ? 0 : 1;
      mbar_arrive(&ctl->p_full[pb]);
    }

    if (kPV && ok && n_tiles > 0) {
      const int t = n_tiles - 1;
      ok = wwait(&ctl->pv_done[t & 1], (t >> 1) & 1);
      tc_fence_after();
    }
    if (kPV && ok) {
      // Epilogue: O / l -> bf16 (a row that saw no key writes zeros).
      const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
      __nv_bfloat16* orow = p.o + (static_cast<size_t>(bh) * p.Lq + grow) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t orr[32];
        if (n_tiles > 0) {
          tmem_ld32p(lane_base + C::kColO + c * 32, orr);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) orr[e] = 0u;
        }
        uint32_t w[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          w[e] = pack_bf16x2(__uint_as_float(orr[2 * e]) * inv_l, __uint_as_float(orr[2 * e + 1]) * inv_l);
        if (row_valid) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int e = 0; e < 4; ++e) dst[e] = make_uint4(w[4 * e], w[4 * e + 1], w[4 * e + 2], w[4 * e + 3]);
        }
      }
    }
    if (tid == 0) {
      if (p.counts != nullptr) p.counts[unit] = skipped;
      for (int j = n_tiles; j < p.nT; ++j) {
        if (p.mask != nullptr) p.mask[unit * p.nT + j] = 2;
        if (p.margin != nullptr) p.margin[unit * p.nT + j] = NAN;
      }
    }
  }

  // ---------------------------------------------------------------- teardown
  if (warp == 5 && lane == 0 && n_tiles > 0) {
    // Every MMA this thread issued must have finished before TMEM is freed.
    mma_commit(&ctl->mma_done);
    mbar_wait(&ctl->mma_done, 0, nullptr);
  }
  if (warp == 4 && lane == 0 && *abort_flag) {
    // On an abort, let in-flight TMA writes land before shared memory is released.
    if (n_tiles > 0) mbar_wait(&ctl->q_full, 0, nullptr);
    // The newest load issued into stage s is the largest i < n with i % NS == s.
    for (int s = 0; s < NS; ++s) {
      if (n_k_issued > s) {
        const int ik = s + ((n_k_issued - 1 - s) / NS) * NS;
        mbar_wait(&ctl->k_full[s], (ik / NS) & 1, nullptr);
      }
      if (n_v_issued > s) {
        const int iv = s + ((n_v_issued - 1 - s) / NS) * NS;
        mbar_wait(&ctl->v_full[s], (iv / NS) & 1, nullptr);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  if (tid == 0 && *abort_flag) report_timeout(p.status);
}

template <int D, Mode MODE>
cudaError_t launch_one(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const PrefillParams& p, cudaStream_t st) {
  using C = PrefillCfg<D>;
  auto* fn = prefill_kernel<D, MODE>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  const long units = static_cast<long>(p.B) * p.Hq * p.nQB;
  fn<<<dim3(static_cast<unsigned>(units)), dim3(192), C::kSmemBytes, st>>>(tq, tk, tv, p);
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
