// Decomposed rel-pos projection (vLLM PR #55629 page, section 关键源码片段:
// add_decomposed_rel_pos, squeezed to the compact [.., HW, H] / [.., HW, W]
// form of section 实现拆解 item 2):
//   rel_h[b, n, kh] = q[b, n] . rel_pos_h[qh - kh + H - 1]
//   rel_w[b, n, kw] = q[b, n] . rel_pos_w[qw - kw + W - 1]
//
// Persistent, one CTA per SM: CTA c handles the 128-token tiles c, c + G,
// c + 2G, ...  A tile's products with every table row, G = Q [T_h ; T_w]^T
// (128 x 256, fp32), come from one tcgen05.mma of N = 256 into one half of
// TMEM.  The roles run decoupled, through mbarriers:
//   - warp 8 (one lane) keeps kProjQStages Q tiles in flight through TMA and
//     issues each tile's MMA as soon as its Q has landed and its TMEM half is
//     free, so the loads and MMAs of later tiles overlap this tile's copy-out;
//   - warps 0-3 skew the rel_h half of each row through shared memory (a
//     per-row shift, see skew_row_to_smem) and store the tile's rel_h rows,
//     which are contiguous in global memory, with coalesced stores; warps 4-7
//     do the same for rel_w.  Each group syncs on its own named barrier.
#pragma once
#include "common.cuh"

namespace dera {

constexpr int kProjCopyWarps = 8;
constexpr int kProjThreads = 32 * (kProjCopyWarps + 1);
constexpr int kProjQStages = 4;

struct ProjSmem {
  static constexpr int kQ = 0;                                  // kProjQStages x 16 KB
  static constexpr int kTables = kProjQStages * kTileBytes;     // T_h rows 0..127, T_w rows 128..255 (32 KB)
  static constexpr int kStage = kTables + 2 * kTileBytes;
  static constexpr int kStride = 65;                            // floats per staged row (>= 64 + 1)
  static constexpr int kStageBytes = kBlockM * kStride * 4;     // one per part (rel_h, rel_w)
  static constexpr int kBars = kStage + 2 * kStageBytes;
  // Q full [S], Q free [S], tables full, G full [2], G free [2]
  static constexpr int kNumBars = 2 * kProjQStages + 5;
  static constexpr int kMisc = kBars + ((kNumBars * 8 + 15) & ~15);
  static constexpr int kTotal = kMisc + 16;
  static constexpr int kAlloc = kTotal + 1024;
};
static_assert(ProjSmem::kAlloc <= 232448, "shared memory budget");

__device__ __forceinline__ void store_elem(void* p, size_t i, float x, int fmt) {
  if (fmt == kF32) {
    reinterpret_cast<float*>(p)[i] = x;
  } else if (fmt == kBF16) {
    reinterpret_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(x);
  } else {
    reinterpret_cast<__half*>(p)[i] = __float2half_rn(x);
  }
}

__global__ void __launch_bounds__(kProjThreads, 1)
    relpos_project_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_th,
                          const __grid_constant__ CUtensorMap tm_tw, const ProjArgs args, int in_fmt,
                          int n_qtiles) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_u + 1023u) & ~1023u) - raw_u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + ProjSmem::kBars);
  uint64_t* q_full = bars;
  uint64_t* q_free = bars + kProjQStages;
  uint64_t* t_full = bars + 2 * kProjQStages;
  uint64_t* g_full = t_full + 1;
  uint64_t* g_free = t_full + 3;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + ProjSmem::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + ProjSmem::kMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = args.H, W = args.W, N = args.N;
  const int n_tiles = n_qtiles * args.BH;
  // this CTA's tiles: blockIdx.x + i * gridDim.x for i < T (the grid is at most n_tiles)
  const int T = (n_tiles - 1 - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x) + 1;
  auto tile_of = [&](int i) { return static_cast<int>(blockIdx.x) + i * static_cast<int>(gridDim.x); };
  auto sQ = [&](int i) { return smem + ProjSmem::kQ + (i % kProjQStages) * kTileBytes; };

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int k = 0; k < kProjQStages; ++k) {
      mbar_init(&q_full[k], 1);
      mbar_init(&q_free[k], 1);
    }
    mbar_init(t_full, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&g_full[b], 1);
      mbar_init(&g_free[b], kProjCopyWarps);
    }
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  if (warp == kProjCopyWarps) {
    // ------------------------------------------------------- loads and MMAs
    if (lane == 0) {
      auto load_q = [&](int i) {
        const int t = tile_of(i);
        mbar_arrive_expect_tx(&q_full[i % kProjQStages], kTileBytes);
        tma_load_3d(sQ(i), &tm_q, &q_full[i % kProjQStages], 0, (t % n_qtiles) * kBlockM, t / n_qtiles);
      };
      mbar_arrive_expect_tx(t_full, 2 * kTileBytes);
      tma_load_2d(smem + ProjSmem::kTables, &tm_th, t_full, 0, 0);
      tma_load_2d(smem + ProjSmem::kTables + kTileBytes, &tm_tw, t_full, 0, 0);
      int loaded = 0, mmas = 0;
      for (; loaded < min(kProjQStages, T); ++loaded) load_q(loaded);
      bool ok = mbar_wait(t_full, 0, abort_flag, args.status);
      const uint32_t fmt = static_cast<uint32_t>(in_fmt);
      const uint32_t id = idesc_f16(kBlockM, 256, fmt, fmt, 0, 0);
      for (int i = 0; i < T && ok; ++i) {
        // the buffer that MMA(i - 1) read takes tile i - 1 + kProjQStages
        if (i >= 1 && loaded < T) {
          ok = mbar_wait(&q_free[(i - 1) % kProjQStages], ((i - 1) / kProjQStages) & 1, abort_flag, args.status);
          if (!ok) break;
          load_q(loaded++);
        }
        ok = mbar_wait(&q_full[i % kProjQStages], (i / kProjQStages) & 1, abort_flag, args.status);
        // TMEM half i & 1 was last read by the copy-out of tile i - 2
        if (ok && i >= 2) ok = mbar_wait(&g_free[i & 1], ((i >> 1) & 1) ^ 1, abort_flag, args.status);
        if (!ok) break;
        tc_fence_after();
        #pragma unroll
        for (int k = 0; k < 4; ++k)
          umma_ss(tbase + 256 * (i & 1), sdesc_sw128(smem_u32(sQ(i)) + 32 * k, 16, 1024),
                  sdesc_sw128(smem_u32(smem + ProjSmem::kTables) + 32 * k, 16, 1024), id, k > 0);
        umma_commit(&g_full[i & 1]);
        umma_commit(&q_free[i % kProjQStages]);
        ++mmas;
      }
      if (!ok) {
        // let the copies already issued and the MMAs already committed finish
        // before the CTA frees its TMEM and exits
        mbar_wait_budget(t_full, 0, kWaitBudgetCycles);
        for (int k = max(0, loaded - kProjQStages); k < loaded; ++k)
          mbar_wait_budget(&q_full[k % kProjQStages], (k / kProjQStages) & 1, kWaitBudgetCycles);
        for (int k = max(0, mmas - 2); k < mmas; ++k)
          mbar_wait_budget(&g_full[k & 1], (k >> 1) & 1, kWaitBudgetCycles);
      }
    }
  } else {
    // ------------------------------------------------------- copy-out
    const int part = warp >> 2;    // 0: rel_h, 1: rel_w
    const int wq = warp & 3;       // TMEM lane quarter
    const int bar_id = 1 + part;   // this part's named barrier
    const int r = wq * 32 + lane;  // tile row = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    float* stage = reinterpret_cast<float*>(smem + ProjSmem::kStage + part * ProjSmem::kStageBytes);
    const int len = part == 0 ? H : W;
    void* dst = part == 0 ? args.rel_h : args.rel_w;
    const int pt = threadIdx.x & 127;
    // fp32 rows with len % 4 == 0 leave as 16-byte chunks: chunk e of the tile
    // is row e / cpr, column 4 (e % cpr); thread pt takes e = pt, pt + 128, ...
    const int cpr = len / 4;
    const bool vec = args.bias_fmt == kF32 && len % 4 == 0;
    const int e_row0 = vec ? pt / cpr : 0, e_col0 = vec ? pt - e_row0 * cpr : 0;
    const int e_drow = vec ? 128 / cpr : 0, e_dcol = vec ? 128 - e_drow * cpr : 0;
    bool ok = true;
    for (int i = 0; i < T; ++i) {
      const int t = tile_of(i);
      const int qt = t % n_qtiles, bh = t / n_qtiles;
      ok = bar_and(bar_id, 128, mbar_wait(&g_full[i & 1], (i >> 1) & 1, abort_flag, args.status) && ok);
      if (!ok) break;
      tc_fence_after();
      const int n0 = qt * kBlockM;
      const int n = n0 + r;
      const int qh = n < N ? n / W : 0;
      const int qw = n < N ? n - qh * W : 0;
      const int rows = min(kBlockM, N - n0);
      skew_row_to_smem(tbase + 256 * (i & 1) + lane_off + 128 * part, part == 0 ? qh : qw, len,
                       stage + r * ProjSmem::kStride, 1.0f);
      tc_fence_before();  // this warp's TMEM reads of the half are done
      __syncwarp();
      if (lane == 0) mbar_arrive(&g_free[i & 1]);
      bar_sync(bar_id, 128);  // the part's stage is complete
      const size_t base = (static_cast<size_t>(bh) * N + n0) * len;
      if (vec) {
        float4* out4 = reinterpret_cast<float4*>(static_cast<float*>(dst) + base);
        int rr = e_row0, c = e_col0;
        for (int e = pt; e < rows * cpr; e += 128) {
          const float* src = stage + rr * ProjSmem::kStride + 4 * c;
          out4[e] = make_float4(src[0], src[1], src[2], src[3]);
          rr += e_drow;
          c += e_dcol;
          if (c >= cpr) {
            c -= cpr;
            ++rr;
          }
        }
      } else {
        // a row per warp pass, lanes along it (len <= 64)
        for (int rr = wq; rr < rows; rr += 4)
          for (int cc = lane; cc < len; cc += 32)
            store_elem(dst, base + static_cast<size_t>(rr) * len + cc, stage[rr * ProjSmem::kStride + cc],
                       args.bias_fmt);
      }
      bar_sync(bar_id, 128);  // every thread of the part has read the stage
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

}  // namespace dera
