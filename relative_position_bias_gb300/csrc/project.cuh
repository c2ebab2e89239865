// Decomposed rel-pos projection (vLLM PR #55629 page, section 关键源码片段:
// add_decomposed_rel_pos, squeezed to the compact [.., HW, H] / [.., HW, W]
// form of section 实现拆解 item 2):
//   rel_h[b, n, kh] = q[b, n] . rel_pos_h[qh - kh + H - 1]
//   rel_w[b, n, kw] = q[b, n] . rel_pos_w[qw - kw + W - 1]
//
// Persistent: CTA c handles the 128-token tiles c, c + G, c + 2G, ... (G CTAs,
// two per SM).  The tables are loaded once per CTA and the next tile's Q is
// loaded while the current tile is processed.  A tile's products with every
// table row, G = Q [T_h ; T_w]^T (128 x 256, fp32), come from one tcgen05.mma
// of N = 256 into TMEM; each thread then skews its row through shared memory
// (a per-row shift, see skew_row_to_smem), and the CTA writes the tile's
// rel_h rows and rel_w rows, which are contiguous in global memory, with
// coalesced stores.
#pragma once
#include "common.cuh"

namespace dera {

constexpr int kProjThreads = 128;

struct ProjSmem {
  static constexpr int kQ = 0;                       // 2 x 16 KB (double-buffered)
  static constexpr int kTables = 2 * kTileBytes;     // T_h rows 0..127, T_w rows 128..255 (32 KB)
  static constexpr int kStage = kTables + 2 * kTileBytes;
  static constexpr int kStride = 65;                 // floats per staged row (>= 64 + 1)
  static constexpr int kStageBytes = kBlockM * kStride * 4;
  static constexpr int kBars = kStage + kStageBytes;  // Q full [2], tables full, MMA done
  static constexpr int kMisc = kBars + 32;
  static constexpr int kTotal = kMisc + 16;
  static constexpr int kAlloc = kTotal + 1024;
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

__global__ void __launch_bounds__(kProjThreads, 1)
    relpos_project_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_th,
                          const __grid_constant__ CUtensorMap tm_tw, const ProjArgs args, int in_fmt,
                          int n_qtiles) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_u + 1023u) & ~1023u) - raw_u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + ProjSmem::kBars);  // [0,1] Q, [2] tables, [3] MMA
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + ProjSmem::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + ProjSmem::kMisc + 4);
  float* stage = reinterpret_cast<float*>(smem + ProjSmem::kStage);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = args.H, W = args.W, N = args.N;
  const int n_tiles = n_qtiles * args.BH;
  auto sQ = [&](int b) { return smem + ProjSmem::kQ + b * kTileBytes; };
  // Q tile of this CTA's i-th tile into buffer i & 1
  auto load_q = [&](int i) {
    const int t = blockIdx.x + i * gridDim.x;
    mbar_arrive_expect_tx(&bars[i & 1], kTileBytes);
    tma_load_3d(sQ(i & 1), &tm_q, &bars[i & 1], 0, (t % n_qtiles) * kBlockM, t / n_qtiles);
  };

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int k = 0; k < 4; ++k) mbar_init(&bars[k], 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(&bars[2], 2 * kTileBytes);
    tma_load_2d(smem + ProjSmem::kTables, &tm_th, &bars[2], 0, 0);
    tma_load_2d(smem + ProjSmem::kTables + kTileBytes, &tm_tw, &bars[2], 0, 0);
    if (static_cast<int>(blockIdx.x) < n_tiles) load_q(0);
  }
  const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
  const int r = warp * 32 + lane;
  bool ok = true;
  int i = 0;
  for (int t = blockIdx.x; t < n_tiles && ok; t += gridDim.x, ++i) {
    const int qt = t % n_qtiles, bh = t / n_qtiles;
    if (threadIdx.x == 0) {
      // buffer (i + 1) & 1 was last read by tile i - 1's MMA, which has completed
      if (t + static_cast<int>(gridDim.x) < n_tiles) load_q(i + 1);
      ok = mbar_wait(&bars[i & 1], (i >> 1) & 1, abort_flag, args.status);
      if (ok && i == 0) ok = mbar_wait(&bars[2], 0, abort_flag, args.status);
      if (ok) {
        tc_fence_after();
        const uint32_t fmt = static_cast<uint32_t>(in_fmt);
        const uint32_t id = idesc_f16(kBlockM, 256, fmt, fmt, 0, 0);
        #pragma unroll
        for (int k = 0; k < 4; ++k)
          umma_ss(tbase, sdesc_sw128(smem_u32(sQ(i & 1)) + 32 * k, 16, 1024),
                  sdesc_sw128(smem_u32(smem + ProjSmem::kTables) + 32 * k, 16, 1024), id, k > 0);
      }
      umma_commit(&bars[3]);
    }
    ok = mbar_wait(&bars[3], i & 1, abort_flag, args.status) && ok;
    ok = __syncthreads_and(ok);
    tc_fence_after();
    if (!ok) break;

    const int n0 = qt * kBlockM;
    const int n = n0 + r;
    const bool row_valid = n < N;
    const int qh = row_valid ? n / W : 0;
    const int qw = row_valid ? n - qh * W : 0;
    const int rows = min(kBlockM, N - n0);
    // rel_h rows of the tile, then rel_w rows (both contiguous in global memory)
    for (int part = 0; part < 2; ++part) {
      const int len = part == 0 ? H : W;
      skew_row_to_smem(tbase + lane_off + 128 * part, part == 0 ? qh : qw, len,
                       stage + r * ProjSmem::kStride, 1.0f);
      if (part == 1) tc_fence_before();  // TMEM reads of this tile done before the next MMA
      __syncthreads();
      void* dst = part == 0 ? args.rel_h : args.rel_w;
      const size_t base = (static_cast<size_t>(bh) * N + n0) * len;
      if (args.bias_fmt == kF32 && len % 4 == 0) {
        // 16-byte stores: a row of len floats is len / 4 chunks; the warp's
        // lanes cover consecutive chunks of consecutive rows
        const int cpr = len / 4;  // chunks per row
        const int total = rows * cpr;
        float4* out4 = reinterpret_cast<float4*>(static_cast<float*>(dst) + base);
        for (int e = threadIdx.x; e < total; e += kProjThreads) {
          const int rr = e / cpr, c4 = 4 * (e - rr * cpr);
          const float* src = stage + rr * ProjSmem::kStride + c4;
          out4[e] = make_float4(src[0], src[1], src[2], src[3]);
        }
      } else {
        // a row per warp pass, lanes along it (len <= 64)
        for (int rr = warp; rr < rows; rr += kProjThreads / 32)
          for (int cc = lane; cc < len; cc += 32)
            store_elem(dst, base + static_cast<size_t>(rr) * len + cc, stage[rr * ProjSmem::kStride + cc],
                       args.bias_fmt);
      }
      __syncthreads();
    }
  }
  if (!ok && threadIdx.x == 0) {
    // let the copies already issued (tables, Q of tiles i and i + 1) land before the CTA exits
    mbar_wait_budget(&bars[2], 0, kWaitBudgetCycles);
    for (int k = i; k <= i + 1; ++k)
      if (blockIdx.x + k * gridDim.x < static_cast<unsigned>(n_tiles))
        mbar_wait_budget(&bars[k & 1], (k >> 1) & 1, kWaitBudgetCycles);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tbase, 256);
  }
}

}  // namespace dera
