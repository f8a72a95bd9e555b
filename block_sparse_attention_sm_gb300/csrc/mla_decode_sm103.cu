// Skip-softmax (BLASST) split-KV decode for multi-head latent attention
// (MLA) on sm_103a, plus the log-sum-exp merge of the splits.
//
// The BLASST summary lists MLA among the attention kinds its prefill and
// decode kernels support (§Belangrijkste Bijdragen, item 4: MHA, GQA, MQA and
// MLA), without shapes.  Read here in the absorbed decode form:
// every sequence keeps one latent cache row per token, 512 latent entries
// followed by 64 rotary entries; the keys are the whole 576-entry rows, the
// values their 512 latent entries, and all Hq query heads share that one
// latent head.  The heads are therefore the voting group of a tile (BLASST
// summary, §Methodologie: skip when the local maximum stays ln(lambda) below
// the running maximum; "Skip-Softmax" §What this bounds: one decision per
// tile), and the tile test, the split of the tiles and the merge are those of
// the GQA decode kernel.
//
// Every key tile is streamed (576 entries per key, as nine 64-entry chunks
// of 16 KB; a chunk's copy slot is free once the score MMAs have read it).
// The values are the latent part of the same rows: for a kept tile they are
// fetched again as soon as the vote has decided -- the rows were read a few
// microseconds earlier, so the second read is normally served by L2 -- and a
// skipped tile's values are never fetched.  A skip therefore saves the
// exponentials, the P.V MMAs and the value copy; the cache crosses HBM once.
// (Holding a whole 144 KB tile in shared memory until its vote left too
// little room to keep the stream in flight.)
//
// One CTA = one (sequence b, split); WG softmax warpgroups (one for up to 16
// heads, two for 17..32) and four role warps, 128 WG + 128 threads:
//   warps 0 .. 4WG-1  vote / softmax: warpgroup w keeps heads 16w .. 16w + 15;
//              thread i of a warpgroup = TMEM lane i, which is key i of the
//              tile for the scores and latent entry i of a 128-entry chunk
//              for the P.V results.  With two warpgroups each tile's vote
//              takes two exchanges: the warp maxima of every head, then each
//              warpgroup's vote statistic over its heads.
//   warp 4WG   TMA producer of the key stream (ring of 64-entry chunks).
//   +1         TMA producer of the values of kept tiles (ring of 128-entry
//              latent pairs, in kept order).
//   +2         TMEM allocator + issuer of the score MMAs
//              S^T = K_tile . Q^T (M = 128 keys, N = 16 WG heads padded with
//              zero rows, K = 576), fp32 in TMEM.
//   +3         issuer of the value MMAs O_i,c^T = V_c^T . P_i^T for the four
//              latent pairs c (M = 128 entries, N = 16 WG, K = 128 keys), one
//              fresh TMEM accumulator per kept tile, folded into registers
//              by the softmax warps in kept order.
// Each thread keeps the state of its warpgroup's 16 heads (one warpgroup for
// 32 heads would need ~290 registers).  With two warpgroups the kernel is
// launched at 168 registers per thread (384 x 168 = 64512) and setmaxnreg
// moves the role warpgroup to 40 and the softmax warpgroups to 232
// (128 x 40 + 256 x 232 = 64512, the launch pool).
#include <cuda_bf16.h>

#include "mla.cuh"
#include "ptx_sm103.cuh"

namespace ssattn {

namespace {

template <int WG>
constexpr int kMThreads = 128 * WG + 128;
// Two warpgroups: registers re-split from the launch pool.
constexpr int kMLaunchRegs = 168, kMRegsRole = 40, kMRegsSoftmax = 232;
static_assert(128 * kMRegsRole + 256 * kMRegsSoftmax == kMThreads<2> * kMLaunchRegs,
              "register split must equal the launch pool");

// Ring depths.  One warpgroup: the same for every mode (at 16 heads the
// voting kernel with two value slots and seven or eight key slots measured
// 3-4% slower).  Two warpgroups: the dense kernel fetches every tile's values
// and keeps three value slots; the voting kernels fetch fewer and give that
// room to the key stream (measured on 128 x 32K, 32 heads: dense 5.0 vs 3.7
// TB/s with two value slots; 70% skipped 5.3 vs 5.6 TB/s with six key slots).
template <Mode MODE, int WG>
struct MCfg {
  static constexpr int NQ = 16 * WG;     // MMA N (heads padded with zero rows)
  static constexpr int HG = 16;          // heads per softmax warpgroup
  static constexpr int NKB = (WG == 2 && MODE == Mode::kDense) ? 4 : 6;  // key-chunk slots
  static constexpr int NVP = (WG == 2 && MODE != Mode::kDense) ? 2 : 3;  // value slots (latent pairs)
  static constexpr int NS = 4;           // score buffers in TMEM
  static constexpr int NV = 2;           // P slots, P.V result slots, kept-tile queue
  static constexpr int kChunks = kMlaDk / 64;
  static constexpr int kPairs = kMlaLatent / 128;
  static constexpr int kChunkBytes = kTile * 64 * 2;
  static constexpr int kPairBytes = kTile * 128 * 2;
  static constexpr int kPBytes = NQ * kTile * 2;
  static constexpr int kVOff = 0;
  static constexpr int kKOff = kVOff + NVP * kPairBytes;
  static constexpr int kQOff = kKOff + NKB * kChunkBytes;
  static constexpr int kPOff = kQOff + kChunks * NQ * 128;
  static constexpr int kRedOff = kPOff + NV * kPBytes;         // float [2][NQ][4]
  static constexpr int kPartOff = kRedOff + 2 * NQ * 4 * 4;    // float [2][2]
  static constexpr int kLRedOff = kPartOff + 16;               // float [NQ][4]
  static constexpr int kMsOff = kLRedOff + NQ * 4 * 4;         // float [2 NV][NQ]
  static constexpr int kCtlOff = kMsOff + 2 * NV * NQ * 4;
  static constexpr int kCtlBytes = 512;
  static constexpr int kSmemBytes = kCtlOff + kCtlBytes + 1024;  // + alignment slack
  static constexpr uint32_t kColS = 0;        // score buffer b at kColS + NQ b
  static constexpr uint32_t kColO = NS * NQ;  // result slot s, pair c at kColO + (4 s + c) NQ
  static constexpr uint32_t kTmemCols = (WG == 1) ? 256 : 512;
  static_assert(kColO + NV * kPairs * NQ <= kTmemCols, "TMEM columns");
  static_assert(kSmemBytes <= 227 * 1024, "shared memory");
};

template <Mode MODE, int WG>
struct MCtl {
  using C = MCfg<MODE, WG>;
  uint64_t kb_full[C::NKB], kb_empty[C::NKB];
  uint64_t vp_full[C::NVP], vp_empty[C::NVP];
  uint64_t s_full[C::NS], s_empty[C::NS];
  uint64_t vq_full[C::NV], p_full[C::NV], slot_free[C::NV];
  uint64_t s_done, pv_done;
  int kq[C::NV];    // kept tile for the value producer (-1: no more)
  int prec[C::NV];  // 1: P written, 0: no more (value-MMA issuer)
  uint32_t tmem_base;
  int abort_flag;
};

template <Mode MODE, int WG>
__global__ void __launch_bounds__(kMThreads<WG>, 1)
    mla_decode_kernel(const __grid_constant__ CUtensorMap tmKV, const MlaParams p) {
  using C = MCfg<MODE, WG>;
  constexpr int kWarpK = 4 * WG, kWarpV = kWarpK + 1, kWarpS = kWarpK + 2;  // +3: value MMAs
  constexpr int kSoftThreads = 128 * WG;
  constexpr int NQ = C::NQ, HG = C::HG, NKB = C::NKB, NVP = C::NVP, NS = C::NS, NV = C::NV;
  constexpr int kChunks = C::kChunks, kPairs = C::kPairs;
  constexpr bool kPV = (MODE != Mode::kCount);
  constexpr bool kVote = (MODE != Mode::kDense);
  static_assert(sizeof(MCtl<MODE, WG>) <= C::kCtlBytes, "control block overflow");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sV = smem + C::kVOff;
  uint8_t* sK = smem + C::kKOff;
  uint8_t* sQ = smem + C::kQOff;
  uint8_t* sP = smem + C::kPOff;
  float* sRed = reinterpret_cast<float*>(smem + C::kRedOff);
  float* sPart = reinterpret_cast<float*>(smem + C::kPartOff);
  float* sLRed = reinterpret_cast<float*>(smem + C::kLRedOff);
  float* sMs = reinterpret_cast<float*>(smem + C::kMsOff);
  auto* ctl = reinterpret_cast<MCtl<MODE, WG>*>(smem + C::kCtlOff);
  volatile int* abort_flag = &ctl->abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = p.Hq;
  const int split = blockIdx.x % p.S;
  const int b = blockIdx.x / p.S;
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
  if (warp == kWarpK && lane == 0) {
    for (int s = 0; s < NKB; ++s) {
      mbar_init(&ctl->kb_full[s], 1);
      mbar_init(&ctl->kb_empty[s], 1);
    }
    for (int s = 0; s < NVP; ++s) {
      mbar_init(&ctl->vp_full[s], 1);
      mbar_init(&ctl->vp_empty[s], 1);
    }
    for (int s = 0; s < NS; ++s) {
      mbar_init(&ctl->s_full[s], 1);
      mbar_init(&ctl->s_empty[s], 4 * WG);
    }
    for (int s = 0; s < NV; ++s) {
      mbar_init(&ctl->vq_full[s], 1);
      mbar_init(&ctl->p_full[s], 4 * WG);
      mbar_init(&ctl->slot_free[s], 1);
    }
    mbar_init(&ctl->s_done, 1);
    mbar_init(&ctl->pv_done, 1);
    ctl->abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tmKV);
    for (int e = 0; e < min(nt * kChunks, NKB); ++e) issue_chunk(e);
  }
  if (warp == kWarpS) {
    tmem_alloc(&ctl->tmem_base, C::kTmemCols);
    tmem_relinquish();
  }
  if (warp < 4 * WG) {
    // Queries as the score MMA's B operand: NQ rows x 576, K-major, one
    // 64-entry box after another, 128-byte swizzle; rows >= G are zero.  P
    // slots: zero, so that their rows >= G stay zero for good.
    constexpr int kGran = kMlaDk / 8;
    for (int idx = tid; idx < NQ * kGran; idx += kSoftThreads) {
      const int g = idx / kGran, e8 = idx - (idx / kGran) * kGran;
      uint4 val = make_uint4(0u, 0u, 0u, 0u);
      if (g < G)
        val = *reinterpret_cast<const uint4*>(p.q + (static_cast<size_t>(b) * p.Hq + g) * kMlaDk +
                                              e8 * 8);
      *reinterpret_cast<uint4*>(sQ + (e8 >> 3) * NQ * 128 + g * 128 + (((e8 & 7) ^ (g & 7)) << 4)) =
          val;
    }
    if (kPV)
      for (int idx = tid; idx < NV * C::kPBytes / 16; idx += kSoftThreads)
        reinterpret_cast<uint4*>(sP)[idx] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;

  // Each warpgroup's code below runs to the end of the kernel under its own
  // register budget; the paths meet only at the final barrier.
  if (warp >= 4 * WG) {
    if constexpr (WG == 2) setmaxnreg_dec<kMRegsRole>();
    int n_v = 0;  // value copies issued
    if (warp == kWarpK) {
      // ------------------------------------------------------ key producer
      if (lane == 0)
        for (int e = NKB; e < nt * kChunks; ++e) {
          if (!mbar_wait(&ctl->kb_empty[e % NKB], ((e / NKB) & 1) ^ 1, abort_flag)) break;
          issue_chunk(e);
        }
    } else if (warp == kWarpV) {
      // ---------------------------------------------------- value producer
      if (kPV && lane == 0 && nt > 0) {
        bool fine = true;
        for (int i = 0; fine; ++i) {
          const int s = i % NV;
          if (!mbar_wait(&ctl->vq_full[s], (i / NV) & 1, abort_flag)) break;
          const int t = *reinterpret_cast<volatile int*>(&ctl->kq[s]);
          if (t < 0) break;
          for (int c = 0; c < kPairs; ++c) {
            const int f = kPairs * i + c, vs = f % NVP;
            if (!mbar_wait(&ctl->vp_empty[vs], ((f / NVP) & 1) ^ 1, abort_flag)) {
              fine = false;
              break;
            }
            mbar_arrive_expect_tx(&ctl->vp_full[vs], C::kPairBytes);
            uint8_t* dst = sV + vs * C::kPairBytes;
            tma_load_3d(dst, &tmKV, &ctl->vp_full[vs], 128 * c, tile_y(t), tile_z(t));
            tma_load_3d(dst + 16384, &tmKV, &ctl->vp_full[vs], 128 * c + 64, tile_y(t), tile_z(t));
            n_v = f + 1;
          }
        }
      }
    } else if (warp == kWarpS) {
      // ---------------------------------------------------------- score MMAs
      if (lane == 0 && nt > 0) {
        constexpr uint32_t idS = idesc_bf16_f32(128, NQ, false, false);
        const uint64_t dq = smem_desc(smem_u32(sQ), 16, 1024);
        const uint32_t sKa = smem_u32(sK);
        bool fine = true;
        for (int t = 0; t < nt && fine; ++t) {
          const int sb = t % NS;
          const uint32_t dcol = tmem + C::kColS + NQ * sb;
          if (!mbar_wait(&ctl->s_empty[sb], ((t / NS) & 1) ^ 1, abort_flag)) break;
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
              const uint32_t qa = (c * NQ * 128 + kk * 32) >> 4;
              mma_bf16_ss(dcol, dk + ((kk * 32) >> 4), dq + qa, idS, (c | kk) ? 1u : 0u);
            }
            mma_commit(&ctl->kb_empty[st]);
          }
          if (fine) mma_commit(&ctl->s_full[sb]);
        }
        mma_commit(&ctl->s_done);
        mbar_wait(&ctl->s_done, 0, nullptr);  // all score MMAs done before TMEM is freed
      }
    } else {
      // ---------------------------------------------------------- value MMAs
      // The whole warp runs the loop (it zeroes the rows of a partial page);
      // lane 0 issues the MMAs and commits.
      if (kPV && nt > 0) {
        constexpr uint32_t idO = idesc_bf16_f32(128, NQ, true, false);
        const uint32_t sVa = smem_u32(sV), sPa = smem_u32(sP);
        bool fine = true;
        for (int i = 0; fine; ++i) {
          const int s = i % NV;
          if (!__all_sync(0xffffffffu, mbar_wait(&ctl->p_full[s], (i / NV) & 1, abort_flag))) break;
          if (*reinterpret_cast<volatile int*>(&ctl->prec[s]) == 0) break;
          // Rows of a page past the sequence end hold whatever the cache
          // holds: zero them so that P = 0 there cannot meet a non-finite value.
          const int rows = paged ? tile_rows(*reinterpret_cast<volatile int*>(&ctl->kq[s])) : kTile;
          const uint64_t dp = smem_desc(sPa + s * C::kPBytes, 16, 1024);
          for (int c = 0; c < kPairs; ++c) {
            const int f = kPairs * i + c, vs = f % NVP;
            if (!__all_sync(0xffffffffu, mbar_wait(&ctl->vp_full[vs], (f / NVP) & 1, abort_flag))) {
              fine = false;
              break;
            }
            if (rows < kTile) {
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
              for (int kk = 0; kk < kTile / 16; ++kk) {
                const uint32_t va = (kk * 2048) >> 4;
                const uint32_t pa = ((kk >> 2) * NQ * 128 + (kk & 3) * 32) >> 4;
                mma_bf16_ss(tmem + C::kColO + (kPairs * s + c) * NQ, dv + va, dp + pa, idO,
                            kk > 0 ? 1u : 0u);
              }
              mma_commit(&ctl->vp_empty[vs]);
            }
            __syncwarp();
          }
          if (fine && lane == 0) mma_commit(&ctl->slot_free[s]);
        }
        if (lane == 0) {
          mma_commit(&ctl->pv_done);
          mbar_wait(&ctl->pv_done, 0, nullptr);
        }
      }
    }
    if (lane == 0 && *abort_flag) {
      // Let in-flight copies land before shared memory is released.
      if (warp == kWarpK) mla_drain_ring<NKB>(ctl->kb_full, n_k);
      if (warp == kWarpV) mla_drain_ring<NVP>(ctl->vp_full, n_v);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ vote / softmax
    if constexpr (WG == 2) setmaxnreg_inc<kMRegsSoftmax>();
    const int wg = warp >> 2;          // softmax warpgroup: heads hg .. hg + 15
    const int hg = HG * wg;
    const int wq = warp & 3;           // warp within the warpgroup
    const int key = tid & 127;         // TMEM lane: key of the tile (scores), latent entry (P.V)
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(wq * 32) << 16) + hg;
    const float sl2 = p.scale_log2;
    auto wwait = [&](uint64_t* bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag));
    };
    float m[HG], l[HG], macc[HG];
    float acc[kPairs][HG];
#pragma unroll
    for (int g = 0; g < HG; ++g) {
      m[g] = -INFINITY;
      l[g] = 0.f;
      macc[g] = -INFINITY;
#pragma unroll
      for (int c = 0; c < kPairs; ++c) acc[c][g] = 0.f;
    }
    uint32_t skipped = 0;
    int kept = 0;
    bool ok = true;

    // Fold the P.V results of kept tile j (slot j % NV) into acc (own heads).
    auto accumulate = [&](int j) {
      const float* ms = sMs + (j % (2 * NV)) * NQ + hg;
      float f[HG];
#pragma unroll
      for (int g = 0; g < HG; ++g) {
        const float mj = ms[g];
        f[g] = (macc[g] == -INFINITY) ? 0.f : ex2_approx((macc[g] - mj) * sl2);
        macc[g] = mj;
      }
#pragma unroll
      for (int c = 0; c < kPairs; ++c) {
        float o[HG];
        mla_tmem_ld16(lane_base + C::kColO + (kPairs * (j % NV) + c) * NQ, o);
        tmem_wait_ld();
#pragma unroll
        for (int g = 0; g < HG; ++g) acc[c][g] = fmaf(acc[c][g], f[g], o[g]);
      }
    };

    for (int t = 0; t < nt; ++t) {
      const int sb = t % NS;
      const bool got = wwait(&ctl->s_full[sb], (t / NS) & 1);
      ok = ok && got;
      tc_fence_after();
      float s[HG];
      if (got) {
        mla_tmem_ld16(lane_base + C::kColS + NQ * sb, s);
        tmem_wait_ld();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->s_empty[sb]);
      const bool valid_key = got && key < tile_rows(t);
#pragma unroll
      for (int g = 0; g < HG; ++g)
        if (!valid_key || hg + g >= G) s[g] = -INFINITY;

      // Tile maximum of each own head: warp maxima exchanged within the
      // warpgroup through shared memory (first 256-thread barrier).
      float mine = -INFINITY;
#pragma unroll
      for (int g = 0; g < HG; ++g) {
        const float wmx = mla_warp_max(s[g]);
        if (lane == g) mine = wmx;
      }
      if (lane < HG) sRed[((t & 1) * NQ + hg + lane) * 4 + wq] = mine;
      named_bar_sync(1, kSoftThreads);
      float tm[HG];
#pragma unroll
      for (int g = 0; g < HG; ++g) {
        const float4 r = *reinterpret_cast<const float4*>(sRed + ((t & 1) * NQ + hg + g) * 4);
        tm[g] = fmaxf(fmaxf(r.x, r.y), fmaxf(r.z, r.w));
      }

      // Vote: skip iff every head g has tile_max_g - m_g < ln(lambda)/scale;
      // each warpgroup's statistic over its heads (with two warpgroups, then
      // the maximum of both at a second barrier).
      float cpart = -INFINITY;
#pragma unroll
      for (int g = 0; g < HG; ++g)
        if (hg + g < G && tm[g] != -INFINITY)
          cpart = fmaxf(cpart, (m[g] == -INFINITY) ? INFINITY : tm[g] - m[g]);
      float cval = cpart;
      if constexpr (WG == 2) {
        if (key == 0) sPart[(t & 1) * 2 + wg] = cpart;
        named_bar_sync(1, kSoftThreads);
        cval = fmaxf(sPart[(t & 1) * 2], sPart[(t & 1) * 2 + 1]);
      }
      const bool skip = kVote && cval < thr_raw;
      if (tid == 0) {
        const long gi = static_cast<long>(b) * row_stride + j0 + t;
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
        // The slot's previous tile (kept - NV) must be through its P.V MMAs
        // before its queue entry, P and result space are reused.
        if (kept >= NV) ok = wwait(&ctl->slot_free[sl], ((kept / NV) - 1) & 1) && ok;
        if (tid == 0) {  // the values of this tile may be fetched now
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
          if (hg + g >= G) break;
          const float alpha = (m[g] == -INFINITY) ? 0.f : ex2_approx((m[g] - mn[g]) * sl2);
          const float mb = (mn[g] == -INFINITY) ? 0.f : mn[g] * sl2;
          const float pv = ex2_approx(fmaf(s[g], sl2, -mb));
          l[g] = fmaf(l[g], alpha, pv);
          const int row = hg + g;
          *reinterpret_cast<__nv_bfloat16*>(ps + row * 128 + ((j8 ^ (row & 7)) << 4)) =
              __float2bfloat16_rn(pv);
        }
        float mine_m = 0.f;
#pragma unroll
        for (int g = 0; g < HG; ++g)
          if (key == g) mine_m = mn[g];
        if (key < HG) sMs[(kept % (2 * NV)) * NQ + hg + key] = mine_m;
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
      // End of the kept stream for the value producer and the value-MMA issuer.
      const int sl = kept % NV;
      if (kept >= NV) ok = wwait(&ctl->slot_free[sl], ((kept / NV) - 1) & 1) && ok;
      if (tid == 0) {
        ctl->kq[sl] = -1;
        mbar_arrive(&ctl->vq_full[sl]);
        ctl->prec[sl] = 0;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->p_full[sl]);
      named_bar_sync(1, kSoftThreads);  // the last tile's maxima (sMs) are visible
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
      named_bar_sync(1, kSoftThreads);
      if (ok && !*abort_flag) {
#pragma unroll
        for (int g = 0; g < HG; ++g) {
          if (hg + g >= G) break;
          const float4 r = *reinterpret_cast<const float4*>(sLRed + (hg + g) * 4);
          const float lt = (r.x + r.y) + (r.z + r.w);
          const size_t row = static_cast<size_t>(b) * p.Hq + hg + g;
          if (p.S == 1) {
            const float inv = lt > 0.f ? 1.f / lt : 0.f;
#pragma unroll
            for (int c = 0; c < kPairs; ++c)
              p.o[row * kMlaLatent + 128 * c + key] = __float2bfloat16_rn(acc[c][g] * inv);
          } else {
            float* pr = p.part + (row * p.S + split) * (kMlaLatent + 2);
#pragma unroll
            for (int c = 0; c < kPairs; ++c) pr[128 * c + key] = acc[c][g];
            if (key == 0) {
              pr[kMlaLatent] = (m[g] == -INFINITY) ? -INFINITY : m[g] * sl2;
              pr[kMlaLatent + 1] = lt;
            }
          }
        }
      }
    }
    if (tid == 0 && p.counts != nullptr) p.counts[static_cast<long>(b) * p.S + split] = skipped;
    if (paged && split == 0 && tid < 32)
      for (int j = nT_b + tid; j < p.max_pages; j += 32) {
        const long gi = static_cast<long>(b) * row_stride + j;
        if (p.mask != nullptr) p.mask[gi] = 2;
        if (p.margin != nullptr) p.margin[gi] = NAN;
      }
    tc_fence_before();
    __syncwarp();
  }

  // ------------------------------------------------------------------ teardown
  barrier_sync(2, kMThreads<WG>);
  if (warp == kWarpS) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
  if (tid == 0 && *abort_flag) report_timeout(p.status);
}

// Log-sum-exp merge of the per-split partial states: one warp per (b, head),
// 16 latent entries per lane.
__global__ void __launch_bounds__(256) mla_merge_kernel(const float* __restrict__ part,
                                                        __nv_bfloat16* __restrict__ o, int rows,
                                                        int S) {
  constexpr int D = kMlaLatent, E = D / 32;
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const float* pr = part + static_cast<size_t>(row) * S * (D + 2);
  float mstar = -INFINITY;
  for (int s = 0; s < S; ++s)
    if (pr[s * (D + 2) + D + 1] > 0.f) mstar = fmaxf(mstar, pr[s * (D + 2) + D]);
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  float L = 0.f;
  for (int s = 0; s < S; ++s) {
    const float ls = pr[s * (D + 2) + D + 1];
    if (!(ls > 0.f)) continue;
    const float w = ex2_approx(pr[s * (D + 2) + D] - mstar);
    L = fmaf(ls, w, L);
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = fmaf(pr[s * (D + 2) + lane + 32 * e], w, acc[e]);
  }
  const float inv = (L > 0.f) ? 1.f / L : 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e)
    o[static_cast<size_t>(row) * D + lane + 32 * e] = __float2bfloat16_rn(acc[e] * inv);
}

template <Mode MODE, int WG>
cudaError_t launch_mla(const CUtensorMap& tkv, const MlaParams& p, cudaStream_t st) {
  using C = MCfg<MODE, WG>;
  auto* fn = mla_decode_kernel<MODE, WG>;
  if constexpr (WG == 2) {
    // The setmaxnreg split assumes exactly kMLaunchRegs registers per thread
    // at launch; with fewer, the softmax warpgroups' increase could never be met.
    static const int launch_regs = [fn] {
      cudaFuncAttributes attr{};
      return cudaFuncGetAttributes(&attr, fn) == cudaSuccess ? attr.numRegs : -1;
    }();
    if (launch_regs != kMLaunchRegs) return cudaErrorInvalidKernelImage;
  }
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  const long ctas = static_cast<long>(p.B) * p.S;
  fn<<<dim3(static_cast<unsigned>(ctas)), dim3(kMThreads<WG>), C::kSmemBytes, st>>>(tkv, p);
  e = cudaGetLastError();
  if (e != cudaSuccess || MODE == Mode::kCount || p.S == 1) return e;
  return launch_mla_merge(p, st);
}

template <int WG>
cudaError_t launch_mla_mode(const CUtensorMap& tkv, const MlaParams& p, Mode mode,
                            cudaStream_t st) {
  switch (mode) {
    case Mode::kDense: return launch_mla<Mode::kDense, WG>(tkv, p, st);
    case Mode::kSparse: return launch_mla<Mode::kSparse, WG>(tkv, p, st);
    default: return launch_mla<Mode::kCount, WG>(tkv, p, st);
  }
}

}  // namespace

cudaError_t launch_mla_merge(const MlaParams& p, cudaStream_t st) {
  const int rows = p.B * p.Hq;
  mla_merge_kernel<<<dim3((rows + 7) / 8), dim3(256), 0, st>>>(p.part, p.o, rows, p.S);
  return cudaGetLastError();
}

cudaError_t launch_mla_decode(const CUtensorMap& tkv, const MlaParams& p, Mode mode,
                              cudaStream_t st) {
  return (p.Hq > kMlaNarrowHeads) ? launch_mla_mode<2>(tkv, p, mode, st)
                                  : launch_mla_mode<1>(tkv, p, mode, st);
}

}  // namespace ssattn
