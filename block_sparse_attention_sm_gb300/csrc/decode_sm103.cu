// Skip-softmax (BLASST) split-KV decode forward for sm_103a, plus the
// log-sum-exp merge of the splits.
//
// Method (BLASST summary, §Methodologie and §Kernel-ontwerp; "Skip-Softmax"
// design doc, §The skip test): decode is bound by HBM traffic.  Every K tile
// of a split is streamed (the scores decide the skip), but a skipped tile's
// V block is never loaded.  To keep the pipeline free of bubbles the
// decisions are taken a chunk of tiles at a time and the surviving V tiles of
// that chunk are fetched as one batch, while the next chunk's scores run.
//
// One CTA = one (sequence b, KV head, split); 512 threads (256 for 8-row groups).  The G
// query heads sharing the KV head (one token each) form the voting group:
// a tile is skipped only if every one of them passes the test.
//
// Pipeline per chunk c of 2 tiles (iteration c), two block barriers:
//   A(c)    scores of tiles 2c, 2c+1 (each by half of the warps) from the K
//           ring (4 stages, 1-D bulk copies of contiguous 128-key tiles),
//           plus per-warp partial row maxima;
//   -- barrier; the two freed K stages are refilled 2 chunks ahead;
//   vote(c) one warp (lane = row): tile maxima, the vote with the exact
//           running maximum, counters / mask / margin, survivor list;
//   C(c-1)  meanwhile, online softmax + P.V over chunk c-1's survivors;
//   -- barrier; the batch of V loads for chunk c's survivors is issued.
// Scores use fp32 FMAs on bf16 K read from shared memory (the contraction
// has only G <= 8 rows; the kernel is bound by the K stream, not by math).
#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx_sm103.cuh"

namespace ssattn {

namespace {

constexpr int kKStages = 4;

struct DecodeCtl {
  uint64_t k_full[kKStages];
  uint64_t v_full[2];
  int abort_flag;
  int n_surv[2];           // [chunk parity]
  int surv_tile[2][2];     // [chunk parity][slot]
  uint32_t surv_par[2][2];
};

template <int D, int GP>
struct DecodeCfg {
  // 16 warps (8 per tile of a chunk) hide shared-memory latency; the
  // 8-row vote group keeps 8 warps to stay within the register budget.
  static constexpr int kThreads = (GP >= 8) ? 256 : 512;
  static constexpr int kWarpsPerTile = kThreads / 64;
  static constexpr int kKeysPerWarp = kTile / kWarpsPerTile;
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kLPR = D / 16;          // lanes per key row (two 16-byte chunks each)
  static constexpr int kKPI = 32 / kLPR;       // keys per warp iteration
  static constexpr int kIters = kKeysPerWarp / kKPI;  // iterations for the warp's keys
  static constexpr int kNDP = D / 2;           // threads per key group in P.V (bf16 pairs)
  static constexpr int kNKG = kThreads / kNDP;  // key groups
  static constexpr int kKPG = kTile / kNKG;    // keys per group
  // shared memory layout (bytes, 16-byte aligned pieces)
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kKOff + kKStages * kTileBytes;
  static constexpr int kQOff = kVOff + 2 * kTileBytes;                 // float [GP][D]
  static constexpr int kScOff = kQOff + GP * D * 4;                    // float [2][2][GP][128]
  static constexpr int kPOff = kScOff + 2 * 2 * GP * kTile * 4;        // float [2][128][GP]
  static constexpr int kTmOff = kPOff + 2 * kTile * GP * 4;            // float [2][2][GP]
  static constexpr int kAlOff = kTmOff + 2 * 2 * GP * 4;               // float [2][GP]
  static constexpr int kMlOff = kAlOff + 2 * GP * 4;                   // float [GP][2]
  static constexpr int kPmOff = kMlOff + GP * 2 * 4;                   // float [2][2][WPT][GP]
  static constexpr int kCtlOff = (kPmOff + 2 * 2 * kWarpsPerTile * GP * 4 + 15) / 16 * 16;
  static constexpr int kVoteWarp = kThreads / 32 - 1;
  static constexpr int kSmemBytes = kCtlOff + 128;
  static_assert(sizeof(DecodeCtl) <= 128, "control block overflow");
  static_assert(kNKG * GP * D * 4 <= kKStages * kTileBytes, "reduction buffer must fit the K ring");
};


// Packed fp32 pair arithmetic (two IEEE fp32 FMAs per instruction).
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
  return static_cast<uint64_t>(__float_as_uint(lo)) | (static_cast<uint64_t>(__float_as_uint(hi)) << 32);
}
// bf16 pair (one 32-bit word) -> fp32 pair (exact: bf16 is the upper half).
__device__ __forceinline__ uint64_t bf16x2_to_f32x2(uint32_t w) {
  return static_cast<uint64_t>(w << 16) | (static_cast<uint64_t>(w & 0xffff0000u) << 32);
}
__device__ __forceinline__ float f32x2_sum(uint64_t v) {
  return __uint_as_float(static_cast<uint32_t>(v)) + __uint_as_float(static_cast<uint32_t>(v >> 32));
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4& raw, float (&f)[8]) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

template <int D, int GP, Mode MODE>
__global__ void __launch_bounds__(DecodeCfg<D, GP>::kThreads, 1) decode_kernel(const DecodeParams p) {
  using C = DecodeCfg<D, GP>;
  constexpr int kDecThreads = C::kThreads;
  constexpr bool kPV = (MODE != Mode::kCount);
  constexpr bool kVote = (MODE != Mode::kDense);
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* sK = smem + C::kKOff;
  uint8_t* sV = smem + C::kVOff;
  float* sQ = reinterpret_cast<float*>(smem + C::kQOff);
  float* sSc = reinterpret_cast<float*>(smem + C::kScOff);
  float* sP = reinterpret_cast<float*>(smem + C::kPOff);
  float* sTm = reinterpret_cast<float*>(smem + C::kTmOff);
  float* sAl = reinterpret_cast<float*>(smem + C::kAlOff);
  float* sMl = reinterpret_cast<float*>(smem + C::kMlOff);
  float* sPm = reinterpret_cast<float*>(smem + C::kPmOff);
  auto* ctl = reinterpret_cast<DecodeCtl*>(smem + C::kCtlOff);
  volatile int* abort_flag = &ctl->abort_flag;
  auto SC = [&](int buf, int tl, int g) { return sSc + ((buf * 2 + tl) * GP + g) * kTile; };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = p.G;
  const int split = blockIdx.x % p.S;
  const int bk = blockIdx.x / p.S;  // b * Hkv + kvh
  const int b = bk / p.Hkv, kvh = bk - (bk / p.Hkv) * p.Hkv;
  const int j0 = split * p.T;
  const int nt = max(0, min(p.nT, j0 + p.T) - j0);
  const int nchunks = (nt + 1) / 2;
  const __nv_bfloat16* kbase = p.k + (static_cast<size_t>(bk) * p.Lk) * D;
  const __nv_bfloat16* vbase = p.v + (static_cast<size_t>(bk) * p.Lk) * D;
  auto tile_rows = [&](int t) { return min(kTile, p.Lk - (j0 + t) * kTile); };

  if (tid == 0) {
    for (int s = 0; s < kKStages; ++s) mbar_init(&ctl->k_full[s], 1);
    for (int s = 0; s < 2; ++s) mbar_init(&ctl->v_full[s], 1);
    ctl->abort_flag = 0;
    ctl->n_surv[0] = ctl->n_surv[1] = 0;
    fence_mbar_init();
  }
  // Query rows of the group (fp32 copy; padding rows are zero).
  for (int idx = tid; idx < GP * D; idx += kDecThreads) {
    const int g = idx / D, e = idx - (idx / D) * D;
    sQ[idx] = (g < G) ? __bfloat162float(p.q[(static_cast<size_t>(b) * p.Hq + kvh * G + g) * D + e]) : 0.f;
  }
  __syncthreads();

  // Thread 0 owns every bulk copy; it records the newest tile issued into
  // each K stage so that an aborted kernel waits for exactly those copies.
  int k_last[kKStages];
#pragma unroll
  for (int s2 = 0; s2 < kKStages; ++s2) k_last[s2] = -1;
  uint32_t nv_issued[2] = {0u, 0u};
  auto issue_k = [&](int t) {
    if (p.fault_inject == 1 && t == 1) return;  // test only: this copy never comes
    const int st = t % kKStages;
    const uint32_t bytes = static_cast<uint32_t>(tile_rows(t)) * D * 2;
    mbar_arrive_expect_tx(&ctl->k_full[st], bytes);
    bulk_load(sK + st * C::kTileBytes, kbase + static_cast<size_t>(j0 + t) * kTile * D, bytes,
              &ctl->k_full[st]);
    k_last[st] = t;
  };
  if (tid == 0)
    for (int t = 0; t < min(nt, kKStages); ++t) issue_k(t);

  // Per-lane query slice for the score phase: the lane owns 16 dimensions,
  // chunks c and c + kLPR of eight (c = lane % kLPR), as fp32 pairs.
  uint64_t qp[GP][8];
  {
    const int e0 = (lane % C::kLPR) * 8, e1 = e0 + C::kLPR * 8;
#pragma unroll
    for (int g = 0; g < GP; ++g)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        qp[g][j] = pack_f32x2(sQ[g * D + e0 + 2 * j], sQ[g * D + e0 + 2 * j + 1]);
        qp[g][4 + j] = pack_f32x2(sQ[g * D + e1 + 2 * j], sQ[g * D + e1 + 2 * j + 1]);
      }
  }

  // Running state.  Vote warp, lane g: exact running max of row g.
  // Warp g (< GP): softmax state of row g (all lanes hold the same values).
  float mt = -INFINITY;
  float m_run = -INFINITY, l_run = 0.f;
  float acc[GP][2];
#pragma unroll
  for (int g = 0; g < GP; ++g) acc[g][0] = acc[g][1] = 0.f;
  uint32_t skipped = 0;
  const float sl2 = p.scale_log2;

  for (int c = 0; c <= nchunks; ++c) {
    const int cb = c & 1;
    // ---------------------------------------------------------------- A(c)
    // Scores of tiles 2c, 2c+1 (half of the warps each), plus each warp's
    // partial row maxima for the vote.
    if (c < nchunks) {
      const int tl = warp / C::kWarpsPerTile;
      const int t = 2 * c + tl;
      if (t < nt) {
        const int st = t % kKStages;
        // warp-uniform: the loop below shuffles across the whole warp
        if (__all_sync(0xffffffffu, mbar_wait(&ctl->k_full[st], (t / kKStages) & 1, abort_flag))) {
          const uint8_t* kt = sK + st * C::kTileBytes;
          const int valid = tile_rows(t);
          float* sc = SC(cb, tl, 0);
          float rmax[GP];
#pragma unroll
          for (int j = 0; j < GP; ++j) rmax[j] = -INFINITY;
          int gsel = 0, n = GP;
          bool writer = true;
#pragma unroll 2
          for (int it = 0; it < C::kIters; ++it) {
            const int key = (warp % C::kWarpsPerTile) * C::kKeysPerWarp + it * C::kKPI + lane / C::kLPR;
            // Two 16-byte chunks of the key row.  For d = 128 the first load
            // of the warp covers bytes [0,128) of its four rows (all eight
            // bank groups); for d = 64 the chunk order alternates with the
            // key's parity for the same reason.
            const int cc = lane % C::kLPR;
            const bool swap = (D == 64) && (key & 1);
            const uint8_t* row = kt + key * D * 2;
            const uint4 r0 = *reinterpret_cast<const uint4*>(row + (swap ? cc + C::kLPR : cc) * 16);
            const uint4 r1 = *reinterpret_cast<const uint4*>(row + (swap ? cc : cc + C::kLPR) * 16);
            const uint4 ra = swap ? r1 : r0, rb = swap ? r0 : r1;
            const uint32_t w[8] = {ra.x, ra.y, ra.z, ra.w, rb.x, rb.y, rb.z, rb.w};
            uint64_t kp[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) kp[j] = bf16x2_to_f32x2(w[j]);
            float part[GP];
#pragma unroll
            for (int g = 0; g < GP; ++g) {
              uint64_t a = 0;
#pragma unroll
              for (int j = 0; j < 8; ++j) a = ffma2(qp[g][j], kp[j], a);
              part[g] = f32x2_sum(a);
            }
            // Transpose-reduce over the kLPR lanes of this key: each halving
            // step hands half of the rows to the partner lane, so the lane
            // ends up holding the full dot products of rows gsel .. gsel+n-1
            // (n > 1 only when a key has fewer lanes than the group rows).
            gsel = 0;
            n = GP;
            writer = true;
#pragma unroll
            for (int o = C::kLPR / 2; o >= 1; o >>= 1) {
              const bool upper = (lane & o) != 0;
              if (n > 1) {
                const int hn = n / 2;
#pragma unroll
                for (int j = 0; j < GP / 2; ++j) {
                  if (j < hn) {
                    const float send = upper ? part[j] : part[j + hn];
                    const float keep = upper ? part[j + hn] : part[j];
                    part[j] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                  }
                }
                gsel += upper ? hn : 0;
                n = hn;
              } else {
                part[0] += __shfl_xor_sync(0xffffffffu, part[0], o);
                writer = writer && !upper;
              }
            }
#pragma unroll
            for (int j = 0; j < GP; ++j) {
              if (j < n) {
                const float sv = (key < valid) ? part[j] : -INFINITY;
                rmax[j] = fmaxf(rmax[j], sv);
                if (writer && gsel + j < G) sc[(gsel + j) * kTile + key] = sv;
              }
            }
          }
          // Partial maxima of this warp's keys: combine over the lanes that
          // hold the same rows for different keys.
#pragma unroll
          for (int j = 0; j < GP; ++j) {
            if (j < n) {
#pragma unroll
              for (int o = C::kLPR; o < 32; o <<= 1) rmax[j] = fmaxf(rmax[j], __shfl_xor_sync(0xffffffffu, rmax[j], o));
              if (lane < C::kLPR && writer && gsel + j < G)
                sPm[((cb * 2 + tl) * C::kWarpsPerTile + warp % C::kWarpsPerTile) * GP + gsel + j] = rmax[j];
            }
          }
        }
      }
    }
    __syncthreads();
    if (tid == 0 && !*abort_flag) {
      // Refill the stages the two tiles of this chunk just released.
      for (int t = 2 * c + kKStages; t < min(nt, 2 * c + kKStages + 2); ++t) issue_k(t);
    }

    // ---------------------------------------------------------------- vote(c)
    // One warp, lane g = row g: tile maxima from the partials, the vote with
    // the exact running maximum, counters and the survivor list of chunk c.
    if (c < nchunks && warp == C::kVoteWarp) {
      int ns = 0;
      for (int tl = 0; tl < 2; ++tl) {
        const int t = 2 * c + tl;
        if (t >= nt) break;
        float tm = -INFINITY;
        if (lane < G)
#pragma unroll
          for (int w2 = 0; w2 < C::kWarpsPerTile; ++w2)
            tm = fmaxf(tm, sPm[((cb * 2 + tl) * C::kWarpsPerTile + w2) * GP + lane]);
        float cval = -INFINITY;
        if (lane < G && tm != -INFINITY) cval = (mt == -INFINITY) ? INFINITY : tm - mt;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) cval = fmaxf(cval, __shfl_xor_sync(0xffffffffu, cval, o));
        const bool skip = kVote && (cval < p.thr_raw);
        if (lane < G) {
          mt = fmaxf(mt, tm);
          sTm[(cb * 2 + tl) * GP + lane] = tm;
        }
        if (lane == 0) {
          const long gi = static_cast<long>(bk) * p.nT + j0 + t;
          if (p.mask != nullptr) p.mask[gi] = skip ? 1 : 0;
          if (p.margin != nullptr) p.margin[gi] = (cval == INFINITY) ? INFINITY : cval * p.scale;
          if (skip) ++skipped;
          else if (kPV) ctl->surv_tile[cb][ns] = t;
        }
        if (!skip && kPV) ++ns;
      }
      if (lane == 0) ctl->n_surv[cb] = ns;
    }

    // ---------------------------------------------------------------- C(c-1)
    // Online softmax + P.V over the survivors of chunk c-1 (their V tiles
    // were fetched after the previous iteration's barrier).
    if (kPV && c >= 1) {
      const int pc = c - 1, pcb = pc & 1;
      const int ns = ctl->n_surv[pcb];
      if (ns > 0) {
        bool ok = true;
        for (int s2 = 0; s2 < ns; ++s2)
          ok = ok && mbar_wait(&ctl->v_full[s2], ctl->surv_par[pcb][s2], abort_flag);
        if (warp < GP) {
          const int g = warp;
          for (int s2 = 0; s2 < ns; ++s2) {
            const int tl = ctl->surv_tile[pcb][s2] - 2 * pc;
            float* prow = sP + s2 * kTile * GP;
            if (g < G) {
              const float tm = sTm[(pcb * 2 + tl) * GP + g];
              const float m_new = fmaxf(m_run, tm);
              const float alpha = (m_run == -INFINITY) ? 0.f : ex2_approx((m_run - m_new) * sl2);
              const float mb = (m_new == -INFINITY) ? 0.f : m_new * sl2;
              const float* sc = SC(pcb, tl, g);
              float sum = 0.f;
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                const int k = lane + 32 * kk;
                const float pv = ex2_approx(fmaf(sc[k], sl2, -mb));
                prow[k * GP + g] = pv;
                sum += pv;
              }
#pragma unroll
              for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
              l_run = alpha * l_run + sum;
              m_run = m_new;
              if (lane == 0) sAl[s2 * GP + g] = alpha;
            } else {
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) prow[(lane + 32 * kk) * GP + g] = 0.f;
              if (lane == 0) sAl[s2 * GP + g] = 1.f;
            }
          }
        }
        __syncthreads();
        if (ok) {
          const int dp = tid % C::kNDP, kg = tid / C::kNDP;
          for (int s2 = 0; s2 < ns; ++s2) {
#pragma unroll
            for (int g = 0; g < GP; ++g) {
              const float a = sAl[s2 * GP + g];
              acc[g][0] *= a;
              acc[g][1] *= a;
            }
            const int valid = tile_rows(ctl->surv_tile[pcb][s2]);
            const uint8_t* vt = sV + s2 * C::kTileBytes;
            const float* prow = sP + s2 * kTile * GP;
            const int k0 = kg * C::kKPG;
            const int kend = min(C::kKPG, valid - k0);
#pragma unroll 4
            for (int kk = 0; kk < kend; ++kk) {
              const int k = k0 + kk;
              const uint32_t wv = *reinterpret_cast<const uint32_t*>(vt + k * D * 2 + dp * 4);
              const float v0 = __uint_as_float(wv << 16), v1 = __uint_as_float(wv & 0xffff0000u);
              float pk[GP];
              if constexpr (GP >= 4) {
#pragma unroll
                for (int g4 = 0; g4 < GP; g4 += 4) {
                  const float4 q4 = *reinterpret_cast<const float4*>(prow + k * GP + g4);
                  pk[g4] = q4.x; pk[g4 + 1] = q4.y; pk[g4 + 2] = q4.z; pk[g4 + 3] = q4.w;
                }
              } else {
#pragma unroll
                for (int g = 0; g < GP; ++g) pk[g] = prow[k * GP + g];
              }
#pragma unroll
              for (int g = 0; g < GP; ++g) {
                acc[g][0] = fmaf(pk[g], v0, acc[g][0]);
                acc[g][1] = fmaf(pk[g], v1, acc[g][1]);
              }
            }
          }
        }
      }
    }
    __syncthreads();
    // ---------------------------------------------------------------- V(c)
    // Batched fetch of chunk c's surviving V tiles (BLASST §Kernel-ontwerp):
    // the slots are free now that C(c-1) is done.
    if (kPV && tid == 0 && c < nchunks && !*abort_flag) {
      const int ns = ctl->n_surv[cb];
      for (int s2 = 0; s2 < ns; ++s2) {
        const int t = ctl->surv_tile[cb][s2];
        const uint32_t bytes = static_cast<uint32_t>(tile_rows(t)) * D * 2;
        ctl->surv_par[cb][s2] = nv_issued[s2] & 1u;
        mbar_arrive_expect_tx(&ctl->v_full[s2], bytes);
        bulk_load(sV + s2 * C::kTileBytes, vbase + static_cast<size_t>(j0 + t) * kTile * D, bytes,
                  &ctl->v_full[s2]);
        ++nv_issued[s2];
      }
    }
  }

  // ------------------------------------------------------------------ output
  if (kPV && !*abort_flag) {
    if (warp < GP && lane == 0) {
      sMl[warp * 2] = m_run;
      sMl[warp * 2 + 1] = l_run;
    }
    float* red = reinterpret_cast<float*>(sK);  // every K load has been consumed
    const int dp = tid % C::kNDP, kg = tid / C::kNDP;
#pragma unroll
    for (int g = 0; g < GP; ++g) {
      red[(kg * GP + g) * D + 2 * dp] = acc[g][0];
      red[(kg * GP + g) * D + 2 * dp + 1] = acc[g][1];
    }
    __syncthreads();
    for (int idx = tid; idx < G * D; idx += kDecThreads) {
      const int g = idx / D, e = idx - (idx / D) * D;
      float sum = 0.f;
#pragma unroll
      for (int kg2 = 0; kg2 < C::kNKG; ++kg2) sum += red[(kg2 * GP + g) * D + e];
      const size_t row = static_cast<size_t>(b) * p.Hq + kvh * G + g;
      if (p.S == 1) {
        const float l = sMl[g * 2 + 1];
        p.o[row * D + e] = __float2bfloat16_rn(l > 0.f ? sum / l : 0.f);
      } else {
        float* pr = p.part + (row * p.S + split) * (D + 2);
        pr[e] = sum;
        if (e == 0) {
          const float m = sMl[g * 2];
          pr[D] = (m == -INFINITY) ? -INFINITY : m * sl2;
          pr[D + 1] = sMl[g * 2 + 1];
        }
      }
    }
  }
  if (warp == C::kVoteWarp && lane == 0 && p.counts != nullptr)
    p.counts[static_cast<long>(bk) * p.S + split] = skipped;
  if (tid == 0) {
    if (*abort_flag) {
      // Let in-flight copies land before shared memory is released.
#pragma unroll
      for (int s2 = 0; s2 < kKStages; ++s2)
        if (k_last[s2] >= 0) mbar_wait(&ctl->k_full[s2], (k_last[s2] / kKStages) & 1, nullptr);
      for (int s = 0; s < 2; ++s)
        if (nv_issued[s] > 0) mbar_wait(&ctl->v_full[s], (nv_issued[s] - 1) & 1, nullptr);
      report_timeout(p.status);
    }
  }
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
cudaError_t launch_dec(const DecodeParams& p, cudaStream_t st) {
  using C = DecodeCfg<D, GP>;
  auto* fn = decode_kernel<D, GP, MODE>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  const long ctas = static_cast<long>(p.B) * p.Hkv * p.S;
  fn<<<dim3(static_cast<unsigned>(ctas)), dim3(C::kThreads), C::kSmemBytes, st>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess || MODE == Mode::kCount || p.S == 1) return e;
  const int rows = p.B * p.Hq;
  decode_merge_kernel<D><<<dim3((rows + 7) / 8), dim3(256), 0, st>>>(p.part, p.o, rows, p.S);
  return cudaGetLastError();
}

template <int D, int GP>
cudaError_t launch_dec_mode(const DecodeParams& p, Mode mode, cudaStream_t st) {
  switch (mode) {
    case Mode::kDense: return launch_dec<D, GP, Mode::kDense>(p, st);
    case Mode::kSparse: return launch_dec<D, GP, Mode::kSparse>(p, st);
    default: return launch_dec<D, GP, Mode::kCount>(p, st);
  }
}

template <int D>
cudaError_t launch_dec_g(const DecodeParams& p, Mode mode, cudaStream_t st) {
  if (p.G <= 1) return launch_dec_mode<D, 1>(p, mode, st);
  if (p.G <= 2) return launch_dec_mode<D, 2>(p, mode, st);
  if (p.G <= 4) return launch_dec_mode<D, 4>(p, mode, st);
  return launch_dec_mode<D, 8>(p, mode, st);
}

}  // namespace

cudaError_t launch_decode(const DecodeParams& p, Mode mode, cudaStream_t st) {
  return (p.d == 128) ? launch_dec_g<128>(p, mode, st) : launch_dec_g<64>(p, mode, st);
}

}  // namespace ssattn
