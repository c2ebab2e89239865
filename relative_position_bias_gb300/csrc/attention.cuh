// Global self-attention with decomposed relative-position bias on tcgen05.
//
// Computes, for every (batch*head) b and token n = qh*W + qw,
//   out[b, n] = sum_m softmax_m(scale * q_n.k_m + rel_h[n, kh(m)] + rel_w[n, kw(m)]) v_m
// without materialising the HW x HW bias (vLLM PR #55629 page, sections
// 实现拆解 item 1 and 关键源码片段).  The softmax is online, in base 2, with
// fp32 statistics (section 风险与影响).
//
// One CTA owns a pair of 128-row query tiles of one head and streams the
// head's keys/values once for both.  Warp roles:
//   warp 0      TMA producer: Q pair, [tables,] K/V ring (3 stages)
//   warp 1      tcgen05.mma issuer (one thread)
//   warp 2      TMEM allocator; with warp 3, converts bf16 V tiles to fp16
//   warps 4-7   softmax / epilogue of query tile 0 (one thread per row)
//   warps 8-11  softmax / epilogue of query tile 1
// TMEM (512 columns): S0 [0,128) S1 [128,256) P0 [256,320) P1 [320,384)
//                     O0 [384,448) O1 [448,512); the fused prologue uses all
//                     512 columns for G_i = Q_i [T_h ; T_w]^T before the loop.
#pragma once
#include "common.cuh"

namespace dera {

constexpr int kStages = 3;
constexpr int kAttnThreads = 384;
constexpr float kRescaleTau = 8.0f;   // lazy rescale threshold (log2 units)
constexpr int kBiasStride = 66;       // floats per row of a bias staging area

struct AttnSmem {
  static constexpr int kQ = 0;                                   // 2 x 16 KB
  static constexpr int kRing = 2 * kTileBytes;                   // stages: [K 16 KB][V 16 KB]
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kBias = kRing + kStages * kStageBytes;    // 2 x 128 x 66 floats
  static constexpr int kBiasBytes = 2 * kBlockM * kBiasStride * 4;
  static constexpr int kBars = kBias + kBiasBytes;
  static constexpr int kNumBars = 24;
  static constexpr int kMisc = kBars + kNumBars * 8;             // tmem slot, abort flag
  static constexpr int kTotal = kMisc + 16;
  static constexpr int kAlloc = kTotal + 1024;                   // slack for 1 KB alignment
};
static_assert(AttnSmem::kAlloc <= 232448, "shared memory budget");

// barrier indices
enum : int {
  kBarQFull = 0,
  kBarKVFull = 1,                 // + stage
  kBarKVEmpty = kBarKVFull + kStages,
  kBarVReady = kBarKVEmpty + kStages,
  kBarSFull = kBarVReady + kStages,   // + tile
  kBarPFull = kBarSFull + 2,
  kBarODone = kBarPFull + 2,
  kBarGFull = kBarODone + 2,
  kBarGFree = kBarGFull + 1,
  kBarMmaDone = kBarGFree + 1,
  kBarCount = kBarMmaDone + 1
};
static_assert(kBarCount <= AttnSmem::kNumBars, "barrier slots");

// Warp-uniform wait result: tcgen05.ld/st are warp-collective, so a warp
// either proceeds as a whole or stops as a whole.
__device__ __forceinline__ bool warp_all(bool ok) { return __all_sync(0xffffffffu, ok); }

__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
  const float lo = __uint_as_float(w << 16);
  const float hi = __uint_as_float(w & 0xFFFF0000u);
  return pack_f16x2(lo, hi);
}

template <int WP, bool FUSED>
__global__ void __launch_bounds__(kAttnThreads, 1)
    relpos_attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_th,
                       const __grid_constant__ CUtensorMap tm_tw, const AttnArgs args) {
  using KT = KeyTile<WP>;
  constexpr int KHT = KT::KHT;
  constexpr int BN = KT::BN;
  constexpr int kChunks = BN / 16;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_u + 1023u) & ~1023u) - raw_u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + AttnSmem::kBars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + AttnSmem::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + AttnSmem::kMisc + 4);
  int* status = args.status;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int bh = blockIdx.x / args.n_pairs;         // consecutive CTAs share one head's K/V
  const int qt0 = 2 * (blockIdx.x % args.n_pairs);
  const int n_kv = args.n_kv;
  const int ring0 = FUSED ? 1 : 0;  // ring slot 0 carries the tables in the fused kernel
  const bool convert_v = args.in_fmt == kBF16;

  auto sQ = [&](int i) { return smem + AttnSmem::kQ + i * kTileBytes; };
  auto sK = [&](int s) { return smem + AttnSmem::kRing + s * AttnSmem::kStageBytes; };
  auto sV = [&](int s) { return smem + AttnSmem::kRing + s * AttnSmem::kStageBytes + kTileBytes; };

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    mbar_init(&bars[kBarQFull], 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars[kBarKVFull + s], 1);
      mbar_init(&bars[kBarKVEmpty + s], 1);
      mbar_init(&bars[kBarVReady + s], 64);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[kBarSFull + i], 1);
      mbar_init(&bars[kBarPFull + i], kBlockM);
      mbar_init(&bars[kBarODone + i], 1);
    }
    mbar_init(&bars[kBarGFull], 1);
    mbar_init(&bars[kBarGFree], 2 * kBlockM);
    mbar_init(&bars[kBarMmaDone], 1);
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      mbar_arrive_expect_tx(&bars[kBarQFull], 2 * kTileBytes);
      tma_load_3d(sQ(0), &tm_q, &bars[kBarQFull], 0, qt0 * kBlockM, bh);
      tma_load_3d(sQ(1), &tm_q, &bars[kBarQFull], 0, (qt0 + 1) * kBlockM, bh);
      int issued = 0;
      bool ok = true;
      if (FUSED) {
        mbar_arrive_expect_tx(&bars[kBarKVFull + 0], 2 * kTileBytes);
        tma_load_2d(sK(0), &tm_th, &bars[kBarKVFull + 0], 0, 0);
        tma_load_2d(sV(0), &tm_tw, &bars[kBarKVFull + 0], 0, 0);
        issued = 1;
      }
      for (int j = 0; j < n_kv && ok; ++j) {
        const int r = ring0 + j, s = r % kStages;
        ok = mbar_wait(&bars[kBarKVEmpty + s], ((r / kStages) & 1) ^ 1, abort_flag, status);
        if (!ok) break;
        mbar_arrive_expect_tx(&bars[kBarKVFull + s], 2 * BN * kRowBytes);
        tma_load_4d(sK(s), &tm_k, &bars[kBarKVFull + s], 0, 0, j * KHT, bh);
        tma_load_4d(sV(s), &tm_v, &bars[kBarKVFull + s], 0, 0, j * KHT, bh);
        issued = r + 1;
      }
      if (!ok) {
        // Let the copies already in flight land before the CTA exits.
        mbar_wait_budget(&bars[kBarQFull], 0, kWaitBudgetCycles);
        for (int r = max(0, issued - kStages); r < issued; ++r)
          mbar_wait_budget(&bars[kBarKVFull + r % kStages], (r / kStages) & 1, kWaitBudgetCycles);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t fmt = static_cast<uint32_t>(args.in_fmt);
      const uint32_t id_qk = idesc_f16(kBlockM, BN, fmt, fmt, 0, 0);
      const uint32_t id_pv = idesc_f16(kBlockM, kHeadDim, kF16, kF16, 0, 1);
      const uint32_t id_g = idesc_f16(kBlockM, 256, fmt, fmt, 0, 0);
      auto issue_qk = [&](int i, int s) {
        #pragma unroll
        for (int k = 0; k < 4; ++k)
          umma_ss(tbase + 128 * i, sdesc_sw128(smem_u32(sQ(i)) + 32 * k, 16, 1024),
                  sdesc_sw128(smem_u32(sK(s)) + 32 * k, 16, 1024), id_qk, k > 0);
      };
      auto issue_pv = [&](int i, int s, bool acc) {
        #pragma unroll
        for (int k = 0; k < BN / 16; ++k)
          umma_ts(tbase + 384 + 64 * i, tbase + 256 + 64 * i + 8 * k,
                  sdesc_sw128(smem_u32(sV(s)) + 2048 * k, 16, 1024), id_pv, (acc || k > 0) ? 1u : 0u);
      };
      bool ok = mbar_wait(&bars[kBarQFull], 0, abort_flag, status);
      if (FUSED && ok) {
        ok = mbar_wait(&bars[kBarKVFull + 0], 0, abort_flag, status);
        if (ok) {
          tc_fence_after();
          for (int i = 0; i < 2; ++i) {
            #pragma unroll
            for (int k = 0; k < 4; ++k)
              umma_ss(tbase + 256 * i, sdesc_sw128(smem_u32(sQ(i)) + 32 * k, 16, 1024),
                      sdesc_sw128(smem_u32(sK(0)) + 32 * k, 16, 1024), id_g, k > 0);
          }
          umma_commit(&bars[kBarGFull]);
          umma_commit(&bars[kBarKVEmpty + 0]);
          ok = mbar_wait(&bars[kBarGFree], 0, abort_flag, status);
          tc_fence_after();
        }
      }
      if (ok) {
        const int s0 = ring0 % kStages;
        ok = mbar_wait(&bars[kBarKVFull + s0], (ring0 / kStages) & 1, abort_flag, status);
        if (ok) {
          tc_fence_after();
          issue_qk(0, s0);
          umma_commit(&bars[kBarSFull + 0]);
          issue_qk(1, s0);
          umma_commit(&bars[kBarSFull + 1]);
        }
      }
      for (int j = 0; j < n_kv && ok; ++j) {
        const int r = ring0 + j, s = r % kStages, ph = (r / kStages) & 1;
        const int rn = r + 1, sn = rn % kStages, phn = (rn / kStages) & 1;
        const bool more = j + 1 < n_kv;
        if (convert_v) {
          ok = mbar_wait(&bars[kBarVReady + s], ph, abort_flag, status);
          if (!ok) break;
        }
        ok = mbar_wait(&bars[kBarPFull + 0], j & 1, abort_flag, status);
        if (!ok) break;
        tc_fence_after();
        issue_pv(0, s, j > 0);
        umma_commit(&bars[kBarODone + 0]);
        if (more) {
          ok = mbar_wait(&bars[kBarKVFull + sn], phn, abort_flag, status);
          if (!ok) break;
          tc_fence_after();
          issue_qk(0, sn);
          umma_commit(&bars[kBarSFull + 0]);
        }
        ok = mbar_wait(&bars[kBarPFull + 1], j & 1, abort_flag, status);
        if (!ok) break;
        tc_fence_after();
        issue_pv(1, s, j > 0);
        umma_commit(&bars[kBarODone + 1]);
        if (more) {
          issue_qk(1, sn);
          umma_commit(&bars[kBarSFull + 1]);
        }
        umma_commit(&bars[kBarKVEmpty + s]);
      }
      // Drain: every MMA issued above completes before TMEM is released.
      umma_commit(&bars[kBarMmaDone]);
      mbar_wait_budget(&bars[kBarMmaDone], 0, kWaitBudgetCycles);
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------ bf16 -> fp16 V conversion
    // The fused kernel's table slot (ring index 0) is passed through
    // unconverted so that v_ready completes once per ring index.
    if (convert_v) {
      const int ct = threadIdx.x - 64;
      for (int r = 0; r < ring0 + n_kv; ++r) {
        const int s = r % kStages;
        if (!mbar_wait(&bars[kBarKVFull + s], (r / kStages) & 1, abort_flag, status)) break;
        if (r >= ring0) {
          uint4* vp = reinterpret_cast<uint4*>(sV(s));
          for (int idx = ct; idx < BN * kRowBytes / 16; idx += 64) {
            uint4 w = vp[idx];
            w.x = bf16x2_to_f16x2(w.x);
            w.y = bf16x2_to_f16x2(w.y);
            w.z = bf16x2_to_f16x2(w.z);
            w.w = bf16x2_to_f16x2(w.w);
            vp[idx] = w;
          }
          fence_proxy_async_smem();
        }
        mbar_arrive(&bars[kBarVReady + s]);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax / epilogue
    const int wg = (warp - 4) >> 2;          // query tile of this warpgroup
    const int wq = warp & 3;                 // TMEM lane quarter
    const int r = wq * 32 + lane;            // row inside the tile
    const int H = args.H, W = args.W, N = args.N;
    const int n = (qt0 + wg) * kBlockM + r;
    const bool row_valid = n < N;
    const int qh = row_valid ? n / W : 0;
    const int qw = row_valid ? n - qh * W : 0;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tbase + lane_off + 128 * wg;
    const uint32_t tP = tbase + lane_off + 256 + 64 * wg;
    const uint32_t tO = tbase + lane_off + 384 + 64 * wg;
    float* area = reinterpret_cast<float*>(smem + AttnSmem::kBias) + wg * kBlockM * kBiasStride;
    const int Hpad = n_kv * KHT;
    const int HS = Hpad + 1;
    float* bh_row = area + r * HS;
    const float NEG_INF = -__int_as_float(0x7f800000);

    float bw[WP];
    bool ok = true;
    if (FUSED) {
      ok = warp_all(mbar_wait(&bars[kBarGFull], 0, abort_flag, status));
      tc_fence_after();
      float* stg = area + r * kBiasStride;
      if (ok) skew_row_to_smem(tbase + lane_off + 256 * wg + 128, qw, W, stg, kLog2e);
      #pragma unroll
      for (int kw = 0; kw < WP; ++kw) bw[kw] = (ok && kw < W) ? stg[kw] : NEG_INF;
      // the staging rows (stride kBiasStride) overlap the bias rows (stride HS)
      named_bar_sync(1 + wg, kBlockM);
      if (ok) {
        skew_row_to_smem(tbase + lane_off + 256 * wg, qh, H, bh_row, kLog2e);
        for (int kh = H; kh < Hpad; ++kh) bh_row[kh] = NEG_INF;
      }
      tc_fence_before();
      mbar_arrive(&bars[kBarGFree]);
    } else {
      const size_t row = static_cast<size_t>(bh) * N + n;
      #pragma unroll
      for (int kw = 0; kw < WP; ++kw)
        bw[kw] = kw < W ? (row_valid ? kLog2e * load_elem(args.rel_w, row * W + kw, args.bias_fmt) : 0.f)
                        : NEG_INF;
      for (int kh = 0; kh < Hpad; ++kh)
        bh_row[kh] = kh < H ? (row_valid ? kLog2e * load_elem(args.rel_h, row * H + kh, args.bias_fmt) : 0.f)
                            : NEG_INF;
    }

    const float sl2 = args.scale_log2;
    const float2 sl2v = make_float2(sl2, sl2);
    float m_used = 0.f;
    float2 lsum = make_float2(0.f, 0.f);
    for (int j = 0; j < n_kv && ok; ++j) {
      ok = warp_all(mbar_wait(&bars[kBarSFull + wg], j & 1, abort_flag, status));
      if (!ok) break;
      tc_fence_after();
      float bhv[KHT];
      #pragma unroll
      for (int g = 0; g < KHT; ++g) bhv[g] = bh_row[j * KHT + g];

      // pass 1: per-grid-row maxima of scale*s*log2e + rel_w*log2e
      float gm[KHT];
      #pragma unroll
      for (int g = 0; g < KHT; ++g) gm[g] = NEG_INF;
      #pragma unroll
      for (int c = 0; c < kChunks; ++c) {
        uint32_t u[16];
        tmem_ld16(tS + 16 * c, u);
        tmem_wait_ld();
        #pragma unroll
        for (int k = 0; k < 16; k += 2) {
          const int col = 16 * c + k;
          const int g = col / WP, kw = col % WP;
          const float2 t = ffma2(make_float2(__uint_as_float(u[k]), __uint_as_float(u[k + 1])), sl2v,
                                 make_float2(bw[kw], bw[kw + 1]));
          gm[g] = fmax3(gm[g], t.x, t.y);
        }
      }
      float mt = NEG_INF;
      #pragma unroll
      for (int g = 0; g < KHT; ++g) mt = fmaxf(mt, gm[g] + bhv[g]);

      if (j > 0) {
        ok = warp_all(mbar_wait(&bars[kBarODone + wg], (j - 1) & 1, abort_flag, status));
        if (!ok) break;
        tc_fence_after();
      }
      if (j == 0) {
        m_used = mt;
      } else if (__any_sync(0xffffffffu, mt > m_used + kRescaleTau)) {
        // Lazy rescale: only when some row of the warp outgrew its stale max.
        const float m_new = fmaxf(m_used, mt);
        const float alpha = ex2_approx(m_used - m_new);
        m_used = m_new;
        lsum.x *= alpha;
        lsum.y *= alpha;
        #pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t o[16];
          tmem_ld16(tO + 16 * c, o);
          tmem_wait_ld();
          #pragma unroll
          for (int k = 0; k < 16; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
          tmem_st16(tO + 16 * c, o);
        }
      }
      float2 off[KHT];
      #pragma unroll
      for (int g = 0; g < KHT; ++g) off[g] = make_float2(bhv[g] - m_used, bhv[g] - m_used);

      // pass 2: p = 2^(x - m), row sums, P (fp16) into TMEM
      #pragma unroll
      for (int c = 0; c < kChunks; ++c) {
        uint32_t u[16];
        tmem_ld16(tS + 16 * c, u);
        tmem_wait_ld();
        uint32_t pk[8];
        #pragma unroll
        for (int k = 0; k < 16; k += 2) {
          const int col = 16 * c + k;
          const int g = col / WP, kw = col % WP;
          float2 t = ffma2(make_float2(__uint_as_float(u[k]), __uint_as_float(u[k + 1])), sl2v,
                           make_float2(bw[kw], bw[kw + 1]));
          t = fadd2(t, off[g]);
          const float2 p = make_float2(ex2_approx(t.x), ex2_approx(t.y));
          lsum = fadd2(lsum, p);
          pk[k / 2] = pack_f16x2(p.x, p.y);
        }
        tmem_st8(tP + 8 * c, pk);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars[kBarPFull + wg]);
    }

    // epilogue: out = O / l
    if (ok) ok = warp_all(mbar_wait(&bars[kBarODone + wg], (n_kv - 1) & 1, abort_flag, status));
    if (ok) {
      tc_fence_after();
      const float inv_l = 1.0f / (lsum.x + lsum.y);
      uint8_t* orow = reinterpret_cast<uint8_t*>(args.out) +
                      (static_cast<size_t>(bh) * N + (row_valid ? n : 0)) * kHeadDim * (args.out_fmt == kF32 ? 4 : 2);
      #pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t o[16];
        tmem_ld16(tO + 16 * c, o);
        tmem_wait_ld();
        if (row_valid) {
          if (args.out_fmt == kF32) {
            float4* dst = reinterpret_cast<float4*>(orow) + 4 * c;
            #pragma unroll
            for (int q4 = 0; q4 < 4; ++q4)
              dst[q4] = make_float4(__uint_as_float(o[4 * q4]) * inv_l, __uint_as_float(o[4 * q4 + 1]) * inv_l,
                                    __uint_as_float(o[4 * q4 + 2]) * inv_l, __uint_as_float(o[4 * q4 + 3]) * inv_l);
          } else {
            uint32_t w[8];
            #pragma unroll
            for (int k = 0; k < 8; ++k) {
              const float a = __uint_as_float(o[2 * k]) * inv_l, b = __uint_as_float(o[2 * k + 1]) * inv_l;
              w[k] = args.out_fmt == kBF16 ? pack_bf16x2(a, b) : pack_f16x2(a, b);
            }
            uint4* dst = reinterpret_cast<uint4*>(orow) + 2 * c;
            dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
            dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

}  // namespace dera
