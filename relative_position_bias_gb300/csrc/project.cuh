// Decomposed rel-pos projection (vLLM PR #55629 page, section 关键源码片段:
// add_decomposed_rel_pos, squeezed to the compact [.., HW, H] / [.., HW, W]
// form of section 实现拆解 item 2):
//   rel_h[b, n, kh] = q[b, n] . rel_pos_h[qh - kh + H - 1]
//   rel_w[b, n, kw] = q[b, n] . rel_pos_w[qw - kw + W - 1]
//
// Persistent, one CTA per SM: CTA c handles the 128-token tiles c, c + G,
// c + 2G, ...  A tile's products with every table row, G = Q [T_h ; T_w]^T
// (128 x 256, fp32), come from one tcgen05.mma of N = 256 into one half of
// TMEM.  Three kinds of warps run decoupled, through mbarriers:
//   - warp 16 (one lane) keeps a ring of Q tiles in flight through TMA and
//     issues each tile's MMA as soon as its Q has landed and its TMEM half is
//     free;
//   - skew warps 0-7 read G out of TMEM and write each row, shifted (see
//     skew_row_to_smem), into one of two staging buffers: warps 0-3 the
//     rel_h half, warps 4-7 the rel_w half, each warp its TMEM lane quarter;
//   - store warps 8-15 copy a staged tile to global memory, where its rel_h
//     rows (warps 8-11) and rel_w rows (warps 12-15) are contiguous, with
//     coalesced stores.
// So the MMA of tile i + 1, the skew of tile i and the stores of tile i - 1
// run at the same time.  With head_dim 128 (Q tiles and tables twice as wide)
// the Q ring is two deep and one staging buffer per half has to do, so there
// the skew of a tile waits for the stores of the previous one.
//
// Staged row strides: rel_h rows use 65 floats, so that the skew's stores
// (one column for the whole warp when its rows share qh) fall in 32 different
// banks; rel_w rows use 68 floats, where the skew's columns already differ
// per lane (qw follows the lane) and rows stay 16-byte aligned, so the stores
// read whole 16-byte chunks.
#pragma once
#include "common.cuh"

namespace dera {

constexpr int kProjSkewWarps = 8;
constexpr int kProjStoreWarps = 8;
constexpr int kProjThreads = 32 * (kProjSkewWarps + kProjStoreWarps + 1);

template <int D>
struct ProjSmem {
  static constexpr int kQStages = D == 64 ? 3 : 2;    // Q ring depth
  static constexpr int kBufs = D == 64 ? 2 : 1;       // staging buffers per half
  static constexpr int kQTile = kBlockM * 2 * D;
  static constexpr int kStrideH = 65;  // floats per staged rel_h row
  static constexpr int kStrideW = 68;  // floats per staged rel_w row
  static constexpr int kStageH = kBlockM * kStrideH * 4;
  static constexpr int kStageW = kBlockM * kStrideW * 4;
  static constexpr int kQ = 0;                                  // kQStages query tiles
  // tables, per atom (64 elements of a row): T_h rows 0..127 then T_w rows 128..255
  static constexpr int kTables = kQStages * kQTile;
  static constexpr int kTableAtom = 2 * kTileBytes;
  static constexpr int kStagesH = kTables + atoms_of<D>() * kTableAtom;  // rel_h staging
  static constexpr int kStagesW = kStagesH + kBufs * kStageH;           // rel_w staging
  static constexpr int kBars = kStagesW + kBufs * kStageW;
  // Q full [S], Q free [S], tables full, G full [2], G free [2],
  // stage full [part][buffer], stage free [part][buffer]
  static constexpr int kNumBars = 2 * kQStages + 5 + 8;
  static constexpr int kMisc = kBars + ((kNumBars * 8 + 15) & ~15);
  static constexpr int kTotal = kMisc + 16;
  static constexpr int kAlloc = kTotal + 1024;
  static_assert(kAlloc <= 232448, "shared memory budget");
  static_assert(kStagesW % 16 == 0 && kStageW % 16 == 0, "16-byte aligned rel_w stage rows");
};

__device__ __forceinline__ void store_elem(void* p, size_t i, float x, int fmt) {
  if (fmt == kF32) {
    reinterpret_cast<float*>(p)[i] = x;
  } else if (fmt == kBF16) {
    reinterpret_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(x);
  } else {
    reinterpret_cast<__half*>(p)[i] = __float2half_rn(x);
  }
}

template <int D>
__global__ void __launch_bounds__(kProjThreads, 1)
    relpos_project_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_th,
                          const __grid_constant__ CUtensorMap tm_tw, const ProjArgs args, int in_fmt,
                          int n_qtiles) {
  using PS = ProjSmem<D>;
  constexpr int kQS = PS::kQStages, NB = PS::kBufs;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_u + 1023u) & ~1023u) - raw_u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + PS::kBars);
  uint64_t* q_full = bars;
  uint64_t* q_free = bars + kQS;
  uint64_t* t_full = bars + 2 * kQS;
  uint64_t* g_full = t_full + 1;
  uint64_t* g_free = t_full + 3;
  uint64_t* s_full = t_full + 5;  // [part * 2 + buffer]
  uint64_t* s_free = t_full + 9;  // [part * 2 + buffer]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + PS::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + PS::kMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = args.H, W = args.W, N = args.N;
  const int n_tiles = n_qtiles * args.BH;
  // this CTA's tiles: blockIdx.x + i * gridDim.x for i < T (the grid is at most n_tiles)
  const int T = (n_tiles - 1 - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x) + 1;
  auto tile_of = [&](int i) { return static_cast<int>(blockIdx.x) + i * static_cast<int>(gridDim.x); };
  auto sQ = [&](int i) { return smem + PS::kQ + (i % kQS) * PS::kQTile; };
  // staging buffer of tile i: buffer i % NB, used for the (i / NB)-th time
  auto stage_of = [&](int part, int i) {
    return reinterpret_cast<float*>(smem + (part == 0 ? PS::kStagesH + (i % NB) * PS::kStageH
                                                      : PS::kStagesW + (i % NB) * PS::kStageW));
  };

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int k = 0; k < kQS; ++k) {
      mbar_init(&q_full[k], 1);
      mbar_init(&q_free[k], 1);
    }
    mbar_init(t_full, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&g_full[b], 1);
      mbar_init(&g_free[b], kProjSkewWarps);
    }
    for (int k = 0; k < 4; ++k) {
      mbar_init(&s_full[k], 128);  // the part's 4 skew warps, every thread
      mbar_init(&s_free[k], 128);  // the part's 4 store warps, every thread
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

  if (warp == kProjSkewWarps + kProjStoreWarps) {
    // ------------------------------------------------------- loads and MMAs
    if (lane == 0) {
      auto load_q = [&](int i) {
        const int t = tile_of(i);
        mbar_arrive_expect_tx(&q_full[i % kQS], PS::kQTile);
        #pragma unroll
        for (int a = 0; a < atoms_of<D>(); ++a)
          tma_load_3d(sQ(i) + a * kTileBytes, &tm_q, &q_full[i % kQS], 64 * a, (t % n_qtiles) * kBlockM,
                      t / n_qtiles);
      };
      mbar_arrive_expect_tx(t_full, atoms_of<D>() * PS::kTableAtom);
      #pragma unroll
      for (int a = 0; a < atoms_of<D>(); ++a) {
        tma_load_2d(smem + PS::kTables + a * PS::kTableAtom, &tm_th, t_full, 64 * a, 0);
        tma_load_2d(smem + PS::kTables + a * PS::kTableAtom + kTileBytes, &tm_tw, t_full, 64 * a, 0);
      }
      int loaded = 0, mmas = 0;
      for (; loaded < min(kQS, T); ++loaded) load_q(loaded);
      bool ok = mbar_wait(t_full, 0, abort_flag, args.status);
      const uint32_t fmt = static_cast<uint32_t>(in_fmt);
      const uint32_t id = idesc_f16(kBlockM, 256, fmt, fmt, 0, 0);
      for (int i = 0; i < T && ok; ++i) {
        // the buffer that MMA(i - 1) read takes tile i - 1 + kQS
        if (i >= 1 && loaded < T) {
          ok = mbar_wait(&q_free[(i - 1) % kQS], ((i - 1) / kQS) & 1, abort_flag, args.status);
          if (!ok) break;
          load_q(loaded++);
        }
        ok = mbar_wait(&q_full[i % kQS], (i / kQS) & 1, abort_flag, args.status);
        // TMEM half i & 1 was last read by the skew of tile i - 2
        if (ok && i >= 2) ok = mbar_wait(&g_free[i & 1], ((i >> 1) & 1) ^ 1, abort_flag, args.status);
        if (!ok) break;
        tc_fence_after();
        // K-step k (16 elements): atom k / 4, 32 bytes per step inside it
        #pragma unroll
        for (int k = 0; k < D / 16; ++k)
          umma_ss(tbase + 256 * (i & 1), sdesc_sw128(smem_u32(sQ(i)) + (k / 4) * kTileBytes + 32 * (k % 4), 16, 1024),
                  sdesc_sw128(smem_u32(smem + PS::kTables) + (k / 4) * PS::kTableAtom + 32 * (k % 4), 16, 1024), id,
                  k > 0);
        umma_commit(&g_full[i & 1]);
        umma_commit(&q_free[i % kQS]);
        ++mmas;
      }
      if (!ok) {
        // let the copies already issued and the MMAs already committed finish
        // before the CTA frees its TMEM and exits
        mbar_wait_budget(t_full, 0, kWaitBudgetCycles);
        for (int k = max(0, loaded - kQS); k < loaded; ++k)
          mbar_wait_budget(&q_full[k % kQS], (k / kQS) & 1, kWaitBudgetCycles);
        for (int k = max(0, mmas - 2); k < mmas; ++k)
          mbar_wait_budget(&g_full[k & 1], (k >> 1) & 1, kWaitBudgetCycles);
      }
    }
  } else if (warp < kProjSkewWarps) {
    // ------------------------------------------------------- skew
    const int part = warp >> 2;    // 0: rel_h, 1: rel_w
    const int wq = warp & 3;       // TMEM lane quarter
    const int r = wq * 32 + lane;  // tile row = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const int stride = part == 0 ? PS::kStrideH : PS::kStrideW;
    const int len = part == 0 ? H : W;
    for (int i = 0; i < T; ++i) {
      const int n = (tile_of(i) % n_qtiles) * kBlockM + r;
      // tcgen05.ld is warp-collective: the warp goes on or stops as a whole
      bool ok = __all_sync(0xffffffffu, mbar_wait(&g_full[i & 1], (i >> 1) & 1, abort_flag, args.status));
      // staging buffer i % NB was last read by the stores of tile i - NB
      if (ok && i >= NB)
        ok = __all_sync(0xffffffffu, mbar_wait(&s_free[part * 2 + i % NB], ((i / NB) & 1) ^ 1, abort_flag,
                                               args.status));
      if (!ok) break;
      tc_fence_after();
      const int qh = n < N ? n / W : 0;
      const int qw = n < N ? n - qh * W : 0;
      skew_row_to_smem(tbase + 256 * (i & 1) + lane_off + 128 * part, part == 0 ? qh : qw, len,
                       stage_of(part, i) + r * stride, 1.0f);
      tc_fence_before();  // this warp's TMEM reads of the half are done
      __syncwarp();
      if (lane == 0) mbar_arrive(&g_free[i & 1]);
      mbar_arrive(&s_full[part * 2 + i % NB]);  // releases this thread's staged row
    }
  } else {
    // ------------------------------------------------------- stores
    const int part = (warp - kProjSkewWarps) >> 2;  // 0: rel_h, 1: rel_w
    const int pt = threadIdx.x & 127;               // thread within the part
    const int len = part == 0 ? H : W;
    const int stride = part == 0 ? PS::kStrideH : PS::kStrideW;
    void* dst = part == 0 ? args.rel_h : args.rel_w;
    // fp32 rows with len % 4 == 0 leave as 16-byte chunks: chunk e is row
    // e / cpr, column 4 (e % cpr).  Otherwise element e is row e / len,
    // column e % len.  Thread pt takes e = pt, pt + 128, ..., stepping
    // (row, column) without a division.
    const bool vec = args.bias_fmt == kF32 && len % 4 == 0;
    const int per_row = vec ? len / 4 : len;
    const int e_row0 = pt / per_row, e_col0 = pt - e_row0 * per_row;
    const int e_drow = 128 / per_row, e_dcol = 128 - e_drow * per_row;
    for (int i = 0; i < T; ++i) {
      if (!mbar_wait(&s_full[part * 2 + i % NB], (i / NB) & 1, abort_flag, args.status)) break;
      const int t = tile_of(i);
      const int n0 = (t % n_qtiles) * kBlockM, bh = t / n_qtiles;
      const int rows = min(kBlockM, N - n0);
      const float* stage = stage_of(part, i);
      const size_t base = (static_cast<size_t>(bh) * N + n0) * len;
      int rr = e_row0, c = e_col0;
      if (vec) {
        float4* out4 = reinterpret_cast<float4*>(static_cast<float*>(dst) + base);
        for (int e = pt; e < rows * per_row; e += 128) {
          const float* src = stage + rr * stride + 4 * c;
          out4[e] = part == 1 ? *reinterpret_cast<const float4*>(src) : make_float4(src[0], src[1], src[2], src[3]);
          rr += e_drow;
          c += e_dcol;
          if (c >= per_row) {
            c -= per_row;
            ++rr;
          }
        }
      } else {
        for (int e = pt; e < rows * per_row; e += 128) {
          store_elem(dst, base + static_cast<size_t>(e), stage[rr * stride + c], args.bias_fmt);
          rr += e_drow;
          c += e_dcol;
          if (c >= per_row) {
            c -= per_row;
            ++rr;
          }
        }
      }
      mbar_arrive(&s_free[part * 2 + i % NB]);  // this thread has read the stage
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
