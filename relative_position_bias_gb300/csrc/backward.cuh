// Backward pass of global attention with decomposed relative-position bias
// (head_dim 64), on tcgen05.
//
// The forward (vLLM PR #55629 page, sections 实现拆解 item 1 and 关键源码片段)
// is out = softmax(Z) v with Z = scale q k^T + rel_h[n, kh(m)] + rel_w[n, kw(m)]
// and rel_h, rel_w the projections of q on the tables.  The pages print no
// backward; this is its chain-rule gradient.  With P = softmax(Z), an upstream
// gradient dO, D[n] = dO[n] . out[n] and dZ = P * (dO v^T - D):
//   dv = P^T dO,  dk = scale dZ^T q,  dq = scale dZ k + (bias part),
//   drel_h[n, kh] = sum_kw dZ[n, (kh, kw)],  drel_w[n, kw] = sum_kh dZ[n, (kh, kw)],
// and through the projection
//   dq[n] += sum_kh drel_h[n, kh] T_h[qh - kh + H - 1] + sum_kw drel_w[n, kw] T_w[qw - kw + W - 1],
//   dT_h[i] = sum over (b, n, kh) with qh - kh + H - 1 = i of drel_h[b, n, kh] q[b, n]  (same for T_w).
// P is recomputed from the forward's base-2 log-sum-exp of each row:
//   P[n, m] = 2^(Z[n, m] log2(e) - lse2[n]).
//
// Three kernels, in stream order (the projection kernel of the forward first
// writes the compact rel_h, rel_w in fp32):
//   relpos_bwd_rows   one CTA per (head, 128-row query tile), key tiles streamed:
//                     S = q k^T and dP = dO v^T on the tensor core, P and dZ on
//                     the softmax threads (one per query row), dZ k accumulated
//                     on the tensor core; then, also on the tensor core, dq's
//                     part through the projection and the tile's partial table
//                     gradients from the on-chip bias gradients; writes dq, the
//                     partials, and for the cols kernel -D and the exponent's
//                     rel_h term log2(e) rel_h - lse by key grid row.
//   relpos_bwd_cols   one CTA per (head, key tile), query tiles streamed:
//                     S^T = k q^T and dP^T = v dO^T, P^T and dZ^T per key row,
//                     dv += P^T dO and dk += dZ^T q accumulated in TMEM; runs
//                     after the rows kernel, whose -D and rel_h term it reads.
//   relpos_bwd_tables sums the per-tile partials in a fixed order.
// Nothing is accumulated with atomics, so the result does not depend on the
// order in which CTAs run.
#pragma once
#include <cfloat>

#include "common.cuh"

namespace dera {

// cols kernel: warp 0 TMA, warp 1 MMA, then kColsParts softmax warps per TMEM
// lane quarter, which split each query tile's 128 columns into 16-column
// blocks, 3 + 3 + 2
constexpr int kColsParts = 3;
constexpr int kBwdColsThreads = 64 + 128 * kColsParts;
constexpr int kBwdStages = 3;      // K/V (rows kernel) or Q/dO (cols kernel) ring depth


// Shared-memory layout shared by the two attention kernels (1024-byte aligned
// operand tiles first).
template <int KS, int kStagingBytes_>
struct BwdSmem {
  static constexpr int kTile = kTileBytes;                  // 128 rows x 128 B
  static constexpr int kA = 0;                              // rows: Q tile; cols: K tile
  static constexpr int kB = kA + kTile;                     // rows: dO tile; cols: V tile
  static constexpr int kRing = kB + kTile;                  // KS stages of two 16 KB tiles
  static constexpr int kStage = 2 * kTile;
  static constexpr int kStaging = kRing + KS * kStage;
  static constexpr int kStagingBytes = kStagingBytes_;
  static constexpr int kBars = kStaging + kStagingBytes;
  static constexpr int kNumBars = 24;
  static constexpr int kMisc = kBars + kNumBars * 8;
  static constexpr int kBytes = kMisc + 64;
  static constexpr int kAlloc = kBytes + 1024;
  static_assert(kAlloc <= 232448, "shared memory");
};

// The two 16-bit values of a packed pair, low half first.
__device__ __forceinline__ float2 unpack_in(uint32_t u, int fmt) {
  if (fmt == kBF16) return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xFFFF0000u));
  return make_float2(__half2float(__ushort_as_half(static_cast<unsigned short>(u & 0xFFFFu))),
                     __half2float(__ushort_as_half(static_cast<unsigned short>(u >> 16))));
}

__device__ __forceinline__ uint32_t pack_in(float lo, float hi, int fmt) {
  return fmt == kBF16 ? pack_bf16x2(lo, hi) : pack_f16x2(lo, hi);
}

// Stores 4 consecutive gradient values of a row in the gradient dtype.
__device__ __forceinline__ void st_grad4(void* base, size_t i, float a, float b, float c, float d, int fmt) {
  if (fmt == kF32) {
    *reinterpret_cast<float4*>(reinterpret_cast<float*>(base) + i) = make_float4(a, b, c, d);
  } else {
    const uint2 w = make_uint2(pack_in(a, b, fmt), pack_in(c, d, fmt));
    *reinterpret_cast<uint2*>(reinterpret_cast<unsigned short*>(base) + i) = w;
  }
}

// Barrier slots of the two attention kernels.
enum : int {
  kBwQFull = 0,                            // rows: Q and dO tiles; cols: K and V tiles
  kBwRingFull = 1,                         // [kBwdStages]
  kBwRingEmpty = kBwRingFull + kBwdStages,
  kBwSFull = kBwRingEmpty + kBwdStages,    // S and dP (or S^T and dP^T) of the current tile in TMEM
  kBwPFull = kBwSFull + 1,                 // softmax threads wrote dZ (and P^T), read S and dP (count 128)
  kBwMmaDone = kBwPFull + 1,               // the products that read dZ (and P^T) of a tile are complete
  kBwStg = kBwMmaDone + 1,                 // staging barrier of the softmax threads (count 128)
  kBwAllDone = kBwStg + 1,                 // rows kernel: every product of the key-tile loop is complete
  kBwTFull = kBwAllDone + 1,               // rows kernel: both tables landed
  kBwGFull = kBwTFull + 1,                 // rows kernel: the softmax threads wrote dG and dG^T (count 128)
  kBwBDone = kBwGFull + 1,                 // rows kernel: the bias products of one table are complete
  kBwSFree = kBwBDone + 1,                 // softmax threads hold this tile's S and dP in registers
  kBwCount = kBwSFree + 1
};
// rows kernel: a three-stage K/V ring; staging holds each thread's rel_h row
// (later its drel_h row) and its drel_w row, 2 x 128 rows of 65 floats
using BwdRowsSmem = BwdSmem<3, 2 * 128 * 65 * 4>;
// cols kernel: a three-stage Q/dO ring; staging holds two buffers of one query
// tile's rel_w (query rows of WP floats, at most 128 x 64 floats) and, in rows
// of 132 floats, its log2(e) rel_h - lse for the key tile's grid rows and -D
// (73 such rows in all)
constexpr int kColsStageRow = 132;
constexpr int kColsStageFloats = 73 * kColsStageRow;
using BwdColsSmem = BwdSmem<3, 2 * kColsStageFloats * 4>;
static_assert(kBwCount <= BwdRowsSmem::kNumBars, "barrier slots");

// Common set-up of the two attention kernels: barriers, TMEM (all 512
// columns), and the aligned shared-memory base.
struct BwdCta {
  uint8_t* smem;
  uint64_t* bars;
  volatile int* abort_flag;
  uint32_t tbase;
};

template <class SM>
__device__ __forceinline__ BwdCta bwd_setup(uint8_t* smem_raw, int warp, int n_compute) {
  BwdCta c;
  const uint32_t raw_u = smem_u32(smem_raw);
  c.smem = smem_raw + (((raw_u + 1023u) & ~1023u) - raw_u);
  c.bars = reinterpret_cast<uint64_t*>(c.smem + SM::kBars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(c.smem + SM::kMisc);
  c.abort_flag = reinterpret_cast<volatile int*>(c.smem + SM::kMisc + 4);
  if (threadIdx.x == 0) {
    *c.abort_flag = 0;
    mbar_init(&c.bars[kBwQFull], 1);
    for (int s = 0; s < kBwdStages; ++s) {   // the rows kernel uses the first two
      mbar_init(&c.bars[kBwRingFull + s], 1);
      mbar_init(&c.bars[kBwRingEmpty + s], 1);
    }
    mbar_init(&c.bars[kBwSFull], 1);
    mbar_init(&c.bars[kBwPFull], n_compute);
    mbar_init(&c.bars[kBwMmaDone], 1);
    mbar_init(&c.bars[kBwStg], n_compute);
    mbar_init(&c.bars[kBwAllDone], 1);
    mbar_init(&c.bars[kBwTFull], 1);
    mbar_init(&c.bars[kBwGFull], n_compute);
    mbar_init(&c.bars[kBwBDone], 1);
    mbar_init(&c.bars[kBwSFree], n_compute);
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  c.tbase = *tmem_slot;
  return c;
}

__device__ __forceinline__ void bwd_teardown(uint32_t tbase, int warp) {
  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

// ---------------------------------------------------------------------------
// Rows kernel: one CTA per (head, query tile), 192 threads: warp 0 TMA, warp 1
// MMA, warps 2-5 the softmax threads, one per query row (TMEM lane).
//  - Key-tile loop: S = q k^T and dP = dO v^T (SS) into TMEM; P and dZ on the
//    softmax threads; dZ k (TS) accumulated in TMEM.  The sums of dZ over each
//    key grid row's columns (drel_h) and over the grid rows (drel_w) stay on
//    chip.
//  - Epilogue, on the tensor core, one table at a time: the bias gradient,
//    unskewed into dG[r][i] = drel[r][coord(r) - i + L - 1] (input dtype),
//    gives dq's part through the projection, dG T, and the tile's table-gradient
//    partial, dG^T q.  dG and its transpose sit in two ring stages so that both
//    products read a K-major A; the tables arrive in the third.
// TMEM columns: S [0, 128), dP [128, 256), dZ [256, 320), dZ k [320, 384); in
// the epilogue dG T [0, 64), dG_h^T q [128, 192), dG_w^T q [192, 256).
constexpr int kBwdRowsThreads = 192;

// Byte offset of 16-bit element (row, k) of a K-major, 128-byte-swizzled
// operand of 128 rows whose K extent is 128 (two 64-element atoms of 16 KB).
__device__ __forceinline__ uint32_t sw128_off(int row, int k) {
  const int a = k >> 6, kk = k & 63;
  return static_cast<uint32_t>(a * kTileBytes + row * 128 + ((((kk >> 3) ^ (row & 7))) << 4) + ((kk & 7) << 1));
}

template <int WP, bool BF16>
__global__ void __launch_bounds__(kBwdRowsThreads, 1)
relpos_bwd_rows_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_th, const __grid_constant__ CUtensorMap tm_tw,
                       const BwdArgs args) {
  using KT = KeyTile<WP, 64>;
  constexpr int KHT = KT::KHT, BN = KT::BN, KS = 3;
  using SM = BwdRowsSmem;
  constexpr int fmt = BF16 ? kBF16 : kF16;
  extern __shared__ uint8_t smem_raw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const BwdCta cta = bwd_setup<SM>(smem_raw, warp, kBlockM);
  uint8_t* smem = cta.smem;
  uint64_t* bars = cta.bars;
  volatile int* abort_flag = cta.abort_flag;
  const uint32_t tbase = cta.tbase;
  int* status = args.status;
  const int bh = blockIdx.x / args.n_qtiles, qt = blockIdx.x - bh * args.n_qtiles;
  const int n_kv = args.n_kv;
  auto sK = [&](int s) { return smem + SM::kRing + s * SM::kStage; };

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_do);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      mbar_arrive_expect_tx(&bars[kBwQFull], 2 * kTileBytes);
      tma_load_3d(smem + SM::kA, &tm_q, &bars[kBwQFull], 0, qt * kBlockM, bh);
      tma_load_3d(smem + SM::kB, &tm_do, &bars[kBwQFull], 0, qt * kBlockM, bh);
      for (int j = 0; j < n_kv; ++j) {
        const int s = j % KS;
        if (!mbar_wait(&bars[kBwRingEmpty + s], ((j / KS) & 1) ^ 1, abort_flag, status)) break;
        mbar_arrive_expect_tx(&bars[kBwRingFull + s], 2 * BN * 128);
        tma_load_4d(sK(s), &tm_k, &bars[kBwRingFull + s], 0, 0, j * KHT, bh);
        tma_load_4d(sK(s) + kTileBytes, &tm_v, &bars[kBwRingFull + s], 0, 0, j * KHT, bh);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    constexpr uint32_t id_s = idesc_f16(kBlockM, BN, fmt, fmt, 0, 0);   // S, dP: both K-major
    constexpr uint32_t id_n = idesc_f16(kBlockM, 64, fmt, fmt, 0, 1);   // A K-major, B N-major (64 columns)
    const uint64_t d_q = sdesc_sw128(smem_u32(smem + SM::kA), 16, 1024);
    const uint64_t d_do = sdesc_sw128(smem_u32(smem + SM::kB), 16, 1024);
    const uint64_t d_ring = sdesc_sw128(smem_u32(smem + SM::kRing), 16, 1024);
    constexpr uint32_t kStageStep = SM::kStage >> 4, kVOfs = kTileBytes >> 4, kAtom = kTileBytes >> 4;
    auto issue_dq = [&](int jj) {
      const int sp = jj % KS;
      #pragma unroll
      for (int k = 0; k < BN / 16; ++k)
        umma_ts_w(tbase + 320, tbase + 256 + 8 * k, d_ring + sp * kStageStep + 128 * k, id_n,
                  (jj > 0 || k > 0) ? 1u : 0u);
      umma_commit_w(&bars[kBwMmaDone]);
      umma_commit_w(&bars[kBwRingEmpty + sp]);
    };
    bool ok = warp_all(mbar_wait(&bars[kBwQFull], 0, abort_flag, status));
    for (int j = 0; ok && j < n_kv; ++j) {
      const int s = j % KS;
      ok = warp_all(mbar_wait(&bars[kBwRingFull + s], (j / KS) & 1, abort_flag, status));
      if (!ok) break;
      if (j > 0) {
        // the softmax threads hold S(j-1) and dP(j-1) in registers
        ok = warp_all(mbar_wait(&bars[kBwSFree], (j - 1) & 1, abort_flag, status));
        if (!ok) break;
      }
      tc_fence_after();
      // S(j) and dP(j) first, so that they run while the softmax threads finish
      // tile j - 1 and start on tile j while dZ(j-1) k runs; they store dZ(j)
      // only once that product has read dZ(j-1)
      #pragma unroll
      for (int k = 0; k < 4; ++k)
        umma_ss_w(tbase + 0, d_q + 2 * k, d_ring + s * kStageStep + 2 * k, id_s, k > 0);
      #pragma unroll
      for (int k = 0; k < 4; ++k)
        umma_ss_w(tbase + 128, d_do + 2 * k, d_ring + s * kStageStep + kVOfs + 2 * k, id_s, k > 0);
      umma_commit_w(&bars[kBwSFull]);
      if (j > 0) {
        // dZ(j-1) is written
        ok = warp_all(mbar_wait(&bars[kBwPFull], (j - 1) & 1, abort_flag, status));
        if (!ok) break;
        tc_fence_after();
        issue_dq(j - 1);
      }
    }
    if (ok) ok = warp_all(mbar_wait(&bars[kBwPFull], (n_kv - 1) & 1, abort_flag, status));
    if (ok) {
      tc_fence_after();
      issue_dq(n_kv - 1);
      // the ring is idle once every product above is complete: the tables go to stage 0
      umma_commit_w(&bars[kBwAllDone]);
      ok = warp_all(mbar_wait(&bars[kBwAllDone], 0, abort_flag, status));
    }
    if (ok) {
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars[kBwTFull], 2 * kTileBytes);
        tma_load_2d(sK(0), &tm_th, &bars[kBwTFull], 0, 0);
        tma_load_2d(sK(0) + kTileBytes, &tm_tw, &bars[kBwTFull], 0, 0);
      }
      __syncwarp();
      ok = warp_all(mbar_wait(&bars[kBwTFull], 0, abort_flag, status));
    }
    const uint64_t d_g = sdesc_sw128(smem_u32(sK(1)), 16, 1024);    // dG: rows r, K = table rows i
    const uint64_t d_gt = sdesc_sw128(smem_u32(sK(2)), 16, 1024);   // dG^T: rows i, K = query rows r
    for (int tb = 0; ok && tb < 2; ++tb) {
      ok = warp_all(mbar_wait(&bars[kBwGFull], tb, abort_flag, status));
      if (!ok) break;
      tc_fence_after();
      const uint64_t d_t = sdesc_sw128(smem_u32(sK(0) + tb * kTileBytes), 16, 1024);
      #pragma unroll
      for (int k = 0; k < 8; ++k)   // dq's bias part, both tables into one accumulator
        umma_ss_w(tbase + 0, d_g + (k / 4) * kAtom + 2 * (k % 4), d_t + 128 * k, id_n, (tb > 0 || k > 0) ? 1u : 0u);
      #pragma unroll
      for (int k = 0; k < 8; ++k)   // this tile's partial table gradient
        umma_ss_w(tbase + 128 + 64 * tb, d_gt + (k / 4) * kAtom + 2 * (k % 4), d_q + 128 * k, id_n, k > 0);
      umma_commit_w(&bars[kBwBDone]);
    }
    // every product issued above completes before TMEM is released
    umma_commit_w(&bars[kBwQFull]);
    mbar_wait_budget(&bars[kBwQFull], 1, kWaitBudgetCycles);
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- softmax threads
    const int H = args.H, W = args.W, N = args.N;
    const int wq = warp & 3;
    const int r = wq * 32 + lane;
    const int n = qt * kBlockM + r;
    const bool row_valid = n < N;
    const int qh = row_valid ? n / W : 0, qw = row_valid ? n - (n / W) * W : 0;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tbase + lane_off, tdP = tS + 128, tdZ = tS + 256, tdQ = tS + 320;
    const size_t row = static_cast<size_t>(bh) * N + (row_valid ? n : 0);
    const float NEG_INF = -__int_as_float(0x7f800000);
    const float sl2 = args.scale_log2;
    float* stg = reinterpret_cast<float*>(smem + SM::kStaging);
    float* bh_row = stg + r * 65;             // rel_h (base 2); each entry becomes drel_h once read
    float* dw_row = stg + 128 * 65 + r * 65;  // drel_w
    const int Hpad = n_kv * KHT;
    // a row past N takes lse = +inf, so that its P is exactly 0 (its S and dP
    // are 0: the TMA fills its q and dO rows with zeros)
    const float lse2 = row_valid ? args.lse[row] : __int_as_float(0x7f800000);
    // The row loads below are independent 16-byte loads where the row allows
    // (rows of the 16-byte aligned workspace whose length is a multiple of 4;
    // dO and out rows of 64 elements), so that they are all in flight at once.
    if (row_valid && (H & 3) == 0) {
      const float4* src = reinterpret_cast<const float4*>(args.rel_h + row * H);
      #pragma unroll
      for (int c = 0; c < 16; ++c) {
        if (4 * c < H) {
          const float4 v = src[c];
          bh_row[4 * c] = kLog2e * v.x;
          bh_row[4 * c + 1] = kLog2e * v.y;
          bh_row[4 * c + 2] = kLog2e * v.z;
          bh_row[4 * c + 3] = kLog2e * v.w;
        }
      }
      for (int kh = H; kh < Hpad; ++kh) bh_row[kh] = NEG_INF;
    } else {
      for (int kh = 0; kh < Hpad; ++kh)
        bh_row[kh] = (kh < H) ? (row_valid ? kLog2e * args.rel_h[row * H + kh] : 0.f) : NEG_INF;
    }
    float bw[WP];
    if (row_valid && (W & 3) == 0) {
      const float4* src = reinterpret_cast<const float4*>(args.rel_w + row * W);
      #pragma unroll
      for (int c = 0; c < WP / 4; ++c) {
        const float4 v = 4 * c < W ? src[c] : make_float4(NEG_INF, NEG_INF, NEG_INF, NEG_INF);
        bw[4 * c] = 4 * c < W ? kLog2e * v.x : NEG_INF;
        bw[4 * c + 1] = 4 * c < W ? kLog2e * v.y : NEG_INF;
        bw[4 * c + 2] = 4 * c < W ? kLog2e * v.z : NEG_INF;
        bw[4 * c + 3] = 4 * c < W ? kLog2e * v.w : NEG_INF;
      }
    } else {
      #pragma unroll
      for (int kw = 0; kw < WP; ++kw)
        bw[kw] = (kw < W) ? (row_valid ? kLog2e * args.rel_w[row * W + kw] : 0.f) : NEG_INF;
    }
    if (row_valid) {
      // the exponent's rel_h term, log2(e) rel_h - lse, by key grid row for
      // the cols kernel (coalesced over the warp's rows)
      const size_t np = static_cast<size_t>(args.n_qtiles) * kBlockM;
      float* hl = args.hl + static_cast<size_t>(bh) * H * np + n;
      for (int kh = 0; kh < H; ++kh) hl[kh * np] = bh_row[kh] - lse2;
    }
    // D = dO . out for this row (out in fp32 or in the input dtype), summed in
    // column order
    float Dn = 0.f;
    if (row_valid) {
      const uint4* dsrc = reinterpret_cast<const uint4*>(args.dout) + row * 8;
      uint4 dv[8];
      #pragma unroll
      for (int c = 0; c < 8; ++c) dv[c] = dsrc[c];
      if (args.out_fmt == kF32) {
        const float4* osrc = reinterpret_cast<const float4*>(args.out) + row * 16;
        float4 ov[16];
        #pragma unroll
        for (int c = 0; c < 16; ++c) ov[c] = osrc[c];
        #pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint32_t dw[4] = {dv[c].x, dv[c].y, dv[c].z, dv[c].w};
          const float o[8] = {ov[2 * c].x, ov[2 * c].y, ov[2 * c].z, ov[2 * c].w,
                              ov[2 * c + 1].x, ov[2 * c + 1].y, ov[2 * c + 1].z, ov[2 * c + 1].w};
          #pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 d2 = unpack_in(dw[e], fmt);
            Dn = fmaf(d2.x, o[2 * e], Dn);
            Dn = fmaf(d2.y, o[2 * e + 1], Dn);
          }
        }
      } else {
        const uint4* osrc = reinterpret_cast<const uint4*>(args.out) + row * 8;
        uint4 ov[8];
        #pragma unroll
        for (int c = 0; c < 8; ++c) ov[c] = osrc[c];
        #pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint32_t dw[4] = {dv[c].x, dv[c].y, dv[c].z, dv[c].w};
          const uint32_t ow[4] = {ov[c].x, ov[c].y, ov[c].z, ov[c].w};
          #pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 d2 = unpack_in(dw[e], fmt), o2 = unpack_in(ow[e], fmt);
            Dn = fmaf(d2.x, o2.x, Dn);
            Dn = fmaf(d2.y, o2.y, Dn);
          }
        }
      }
      args.D[row] = -Dn;   // negated, as the cols kernel adds it
    }
    float dRW[WP];
    #pragma unroll
    for (int kw = 0; kw < WP; ++kw) dRW[kw] = 0.f;
    const float2 sl2v = make_float2(sl2, sl2), nD2 = make_float2(-Dn, -Dn);
    bool ok = true;
    for (int j = 0; ok && j < n_kv; ++j) {
      float bhv[KHT];
      #pragma unroll
      for (int g = 0; g < KHT; ++g) bhv[g] = bh_row[j * KHT + g] - lse2;   // the exponent's rel_h and lse terms
      ok = warp_all(mbar_wait(&bars[kBwSFull], j & 1, abort_flag, status));
      if (!ok) break;
      tc_fence_after();
      float2 dRH[KHT];   // even and odd columns apart
      #pragma unroll
      for (int g = 0; g < KHT; ++g) dRH[g] = make_float2(0.f, 0.f);
      // 16-column blocks, the next block's S and dP loads in flight while the
      // current one is computed
      uint32_t us[2][16], up[2][16];
      tmem_ld16(tS, us[0]);
      tmem_ld16(tdP, up[0]);
      #pragma unroll
      for (int bb = 0; bb < BN / 16; ++bb) {
        const int cb = 16 * bb, cur = bb & 1;
        tmem_wait_ld();
        if (bb + 1 < BN / 16) {
          tmem_ld16(tS + cb + 16, us[cur ^ 1]);
          tmem_ld16(tdP + cb + 16, up[cur ^ 1]);
        } else {
          // all of S(j) and dP(j) is in registers: S(j+1) and dP(j+1) may go ahead
          tc_fence_before();
          mbar_arrive(&bars[kBwSFree]);
        }
        uint32_t pk[8];
        #pragma unroll
        for (int k = 0; k < 16; k += 2) {
          // a pair of columns of one grid row, through the packed fp32x2 units
          const int col = cb + k;
          const int g = col / WP, kw = col % WP;
          const float2 s2 = make_float2(__uint_as_float(us[cur][k]), __uint_as_float(us[cur][k + 1]));
          const float2 dp2 = make_float2(__uint_as_float(up[cur][k]), __uint_as_float(up[cur][k + 1]));
          const float2 b2 = fadd2(make_float2(bw[kw], bw[kw + 1]), make_float2(bhv[g], bhv[g]));
          const float2 x = ffma2(s2, sl2v, b2);
          const float2 d = __fmul2_rn(make_float2(ex2_approx(x.x), ex2_approx(x.y)), fadd2(dp2, nD2));
          const float2 acc = fadd2(make_float2(dRW[kw], dRW[kw + 1]), d);
          dRW[kw] = acc.x;
          dRW[kw + 1] = acc.y;
          dRH[g] = fadd2(dRH[g], d);
          pk[k / 2] = pack_in(d.x, d.y, fmt);
        }
        if (bb == 0 && j > 0) {
          // dZ(j-1) has been read by its product before dZ(j) is written
          ok = warp_all(mbar_wait(&bars[kBwMmaDone], (j - 1) & 1, abort_flag, status));
          if (!ok) {
            tmem_wait_ld();   // the next block's loads are in flight
            break;
          }
          tc_fence_after();
        }
        tmem_st8(tdZ + cb / 2, pk);
      }
      if (!ok) break;
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars[kBwPFull]);
      #pragma unroll
      for (int g = 0; g < KHT; ++g)
        if (j * KHT + g < H) bh_row[j * KHT + g] = dRH[g].x + dRH[g].y;
    }
    #pragma unroll
    for (int kw = 0; kw < WP; ++kw)
      if (kw < W) dw_row[kw] = dRW[kw];
    if (ok) ok = warp_all(mbar_wait(&bars[kBwMmaDone], (n_kv - 1) & 1, abort_flag, status));
    // Epilogue: every product of the loop is complete, so ring stages 1 and 2
    // are free.  Per table: dG row r (stage 1) and column r of dG^T (stage 2),
    // then the two products.
    uint8_t* g_st = sK(1);
    uint8_t* gt_st = sK(2);
    for (int tb = 0; ok && tb < 2; ++tb) {
      const int L = tb == 0 ? H : W, coord = tb == 0 ? qh : qw;
      const float* drow = tb == 0 ? bh_row : dw_row;
      if (tb == 1) {
        // the first table's products have read both stages
        ok = warp_all(mbar_wait(&bars[kBwBDone], 0, abort_flag, status));
        if (!ok) break;
      }
      #pragma unroll 8
      for (int i = 0; i < 128; i += 2) {
        const int k0 = coord - i + L - 1, k1 = k0 - 1;
        const float v0 = (row_valid && k0 >= 0 && k0 < L) ? drow[k0] : 0.f;
        const float v1 = (row_valid && k1 >= 0 && k1 < L) ? drow[k1] : 0.f;
        const uint32_t pk = pack_in(v0, v1, fmt);
        *reinterpret_cast<uint32_t*>(g_st + sw128_off(r, i)) = pk;
        *reinterpret_cast<unsigned short*>(gt_st + sw128_off(i, r)) = static_cast<unsigned short>(pk & 0xFFFFu);
        *reinterpret_cast<unsigned short*>(gt_st + sw128_off(i + 1, r)) = static_cast<unsigned short>(pk >> 16);
      }
      fence_proxy_async_smem();
      mbar_arrive(&bars[kBwGFull]);
    }
    if (ok) ok = warp_all(mbar_wait(&bars[kBwBDone], 1, abort_flag, status));
    if (ok) {
      tc_fence_after();
      uint32_t a[32], b[32];
      const float sc = args.scale;
      #pragma unroll
      for (int h = 0; h < 2; ++h) {
        tmem_ld32(tdQ + 32 * h, a);
        tmem_ld32(tS + 32 * h, b);
        tmem_wait_ld();
        if (row_valid) {
          #pragma unroll
          for (int c = 0; c < 8; ++c)
            st_grad4(args.dq, row * 64 + 32 * h + 4 * c,
                     fmaf(sc, __uint_as_float(a[4 * c]), __uint_as_float(b[4 * c])),
                     fmaf(sc, __uint_as_float(a[4 * c + 1]), __uint_as_float(b[4 * c + 1])),
                     fmaf(sc, __uint_as_float(a[4 * c + 2]), __uint_as_float(b[4 * c + 2])),
                     fmaf(sc, __uint_as_float(a[4 * c + 3]), __uint_as_float(b[4 * c + 3])), args.grad_fmt);
        }
      }
      // table-gradient partials: TMEM lane r holds table row i = r
      const int LH = 2 * H - 1, LW = 2 * W - 1;
      float* part = args.parts + static_cast<size_t>(blockIdx.x) * (LH + LW) * 64;
      #pragma unroll
      for (int tb = 0; tb < 2; ++tb) {
        const int Lrows = tb == 0 ? LH : LW;
        float* dst = part + (tb == 0 ? 0 : LH * 64) + r * 64;
        #pragma unroll
        for (int h = 0; h < 2; ++h) {
          tmem_ld32(tS + 128 + 64 * tb + 32 * h, a);
          tmem_wait_ld();
          if (r < Lrows) {
            #pragma unroll
            for (int c = 0; c < 8; ++c)
              *reinterpret_cast<float4*>(dst + 32 * h + 4 * c) =
                  make_float4(__uint_as_float(a[4 * c]), __uint_as_float(a[4 * c + 1]), __uint_as_float(a[4 * c + 2]),
                              __uint_as_float(a[4 * c + 3]));
          }
        }
      }
    }
  }
  bwd_teardown(tbase, warp);
}

// 16-byte global -> shared copy that does not pass through registers (both
// addresses 16-byte aligned).
__device__ __forceinline__ void cp_async16(void* dst_smem, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst_smem)), "l"(src) : "memory");
}

// ---------------------------------------------------------------------------
// Cols kernel: one CTA per (head, key tile of KHT grid rows); key slot m of the
// tile is TMEM lane m, which the kColsParts softmax warps of lane quarter m / 32
// share, each taking some of every query tile's 16-column blocks (slots past
// the tile's BN keys, padded columns and padded grid rows compute nothing that
// is stored).  The next query tile's S^T and dP^T go ahead once every softmax
// thread holds the current ones in registers.  TMEM
// columns: S^T [0, 128), dP^T [128, 256), P^T and dZ^T in the input dtype as
// packed pairs [256, 320) and [320, 384), dv [384, 448), dk [448, 512).
// Per query tile the softmax threads stage (cp.async, one tile ahead) the
// tile's rel_w rows [128][WP], log2(e) rel_h - lse for this key tile's grid
// rows [KHT][128] (which the rows kernel wrote in that layout) and -D.
template <int WP, bool BF16>
__global__ void __launch_bounds__(kBwdColsThreads, 1)
relpos_bwd_cols_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                       const BwdArgs args) {
  using KT = KeyTile<WP, 64>;
  constexpr int KHT = KT::KHT, BN = KT::BN, KS = kBwdStages;
  using SM = BwdColsSmem;
  constexpr int fmt = BF16 ? kBF16 : kF16;
  extern __shared__ uint8_t smem_raw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const BwdCta cta = bwd_setup<SM>(smem_raw, warp, kColsParts * kBlockM);
  uint8_t* smem = cta.smem;
  uint64_t* bars = cta.bars;
  volatile int* abort_flag = cta.abort_flag;
  const uint32_t tbase = cta.tbase;
  int* status = args.status;
  const int n_kv = args.n_kv, n_qt = args.n_qtiles, H = args.H, W = args.W, N = args.N;
  const int bh = blockIdx.x / n_kv, j = blockIdx.x - bh * n_kv;
  auto sQ = [&](int s) { return smem + SM::kRing + s * SM::kStage; };

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_do);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      mbar_arrive_expect_tx(&bars[kBwQFull], 2 * BN * 128);
      tma_load_4d(smem + SM::kA, &tm_k, &bars[kBwQFull], 0, 0, j * KHT, bh);
      tma_load_4d(smem + SM::kB, &tm_v, &bars[kBwQFull], 0, 0, j * KHT, bh);
      for (int i = 0; i < n_qt; ++i) {
        const int s = i % KS;
        if (!mbar_wait(&bars[kBwRingEmpty + s], ((i / KS) & 1) ^ 1, abort_flag, status)) break;
        mbar_arrive_expect_tx(&bars[kBwRingFull + s], 2 * kTileBytes);
        tma_load_3d(sQ(s), &tm_q, &bars[kBwRingFull + s], 0, i * kBlockM, bh);
        tma_load_3d(sQ(s) + kTileBytes, &tm_do, &bars[kBwRingFull + s], 0, i * kBlockM, bh);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    constexpr uint32_t id_s = idesc_f16(kBlockM, kBlockM, fmt, fmt, 0, 0);  // S^T, dP^T: both K-major
    constexpr uint32_t id_acc = idesc_f16(kBlockM, 64, fmt, fmt, 0, 1);     // P^T dO, dZ^T q: N-major tiles
    const uint64_t d_k = sdesc_sw128(smem_u32(smem + SM::kA), 16, 1024);
    const uint64_t d_v = sdesc_sw128(smem_u32(smem + SM::kB), 16, 1024);
    const uint64_t d_ring = sdesc_sw128(smem_u32(smem + SM::kRing), 16, 1024);
    constexpr uint32_t kStageStep = SM::kStage >> 4, kDoOfs = kTileBytes >> 4;
    auto issue_acc = [&](int ii) {
      const int sp = ii % KS;
      #pragma unroll
      for (int k = 0; k < kBlockM / 16; ++k) {
        const uint32_t acc = (ii > 0 || k > 0) ? 1u : 0u;
        umma_ts_w(tbase + 384, tbase + 256 + 8 * k, d_ring + sp * kStageStep + kDoOfs + 128 * k, id_acc, acc);
        umma_ts_w(tbase + 448, tbase + 320 + 8 * k, d_ring + sp * kStageStep + 128 * k, id_acc, acc);
      }
      umma_commit_w(&bars[kBwMmaDone]);
      umma_commit_w(&bars[kBwRingEmpty + sp]);
    };
    bool ok = warp_all(mbar_wait(&bars[kBwQFull], 0, abort_flag, status));
    for (int i = 0; ok && i < n_qt; ++i) {
      const int s = i % KS;
      ok = warp_all(mbar_wait(&bars[kBwRingFull + s], (i / KS) & 1, abort_flag, status));
      if (!ok) break;
      if (i > 0) {
        // the softmax threads hold S^T(i-1) and dP^T(i-1) in registers
        ok = warp_all(mbar_wait(&bars[kBwSFree], (i - 1) & 1, abort_flag, status));
        if (!ok) break;
      }
      tc_fence_after();
      // S^T(i) and dP^T(i) first, so that they run while the softmax threads
      // finish tile i - 1 and start on query tile i while dv and dk take tile i - 1
      #pragma unroll
      for (int k = 0; k < 4; ++k)
        umma_ss_w(tbase + 0, d_k + 2 * k, d_ring + s * kStageStep + 2 * k, id_s, k > 0);
      #pragma unroll
      for (int k = 0; k < 4; ++k)
        umma_ss_w(tbase + 128, d_v + 2 * k, d_ring + s * kStageStep + kDoOfs + 2 * k, id_s, k > 0);
      umma_commit_w(&bars[kBwSFull]);
      if (i > 0) {
        // P^T(i-1) and dZ^T(i-1) are written
        ok = warp_all(mbar_wait(&bars[kBwPFull], (i - 1) & 1, abort_flag, status));
        if (!ok) break;
        tc_fence_after();
        issue_acc(i - 1);
      }
    }
    if (ok && warp_all(mbar_wait(&bars[kBwPFull], (n_qt - 1) & 1, abort_flag, status))) {
      tc_fence_after();
      issue_acc(n_qt - 1);
    }
    umma_commit_w(&bars[kBwQFull]);
    mbar_wait_budget(&bars[kBwQFull], 1, kWaitBudgetCycles);
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- softmax threads
    const int wq = warp & 3;
    const int m = wq * 32 + lane;          // key slot of the tile
    const int part = (warp - 2) >> 2;      // query-column blocks [3 part, 3 part + nb) of every tile
    const int nb = part < 2 ? 3 : 2;       // 16-column blocks of this part
    constexpr int kStg = kColsParts * kBlockM;
    const int t = threadIdx.x - 64;        // index among the kStg staging threads
    const int g = m / WP, kw = m % WP;
    const int kh = j * KHT + g;
    const bool key_valid = m < BN && kw < W && kh < H;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tbase + lane_off, tdP = tS + 128, tP = tS + 256, tdZ = tS + 320, tdV = tS + 384,
                   tdK = tS + 448;
    const float sl2 = args.scale_log2;
    float* stage_base = reinterpret_cast<float*>(smem + SM::kStaging);
    // buffer b: rel_w [n][kw] in query rows of WP floats (the first 128 WP
    // floats), then, by query column so that a thread reads four at once,
    // log2(e) rel_h - lse [g][n] in rows 64..71 and -D in row 72 (rows of
    // kColsStageRow floats; -D holds zeros past N).  rel_w and rel_h entries
    // past N, past W or past H are never written: they reach only masked query
    // columns or key slots without a key.
    constexpr int kBufFloats = kColsStageFloats, RS = kColsStageRow;
    static_assert(kBlockM * WP <= 64 * RS, "rel_w rows fit below the rows by query column");
    auto stage = [&](int i, int b) {
      float* buf = stage_base + b * kBufFloats;
      const int n0 = i * kBlockM;
      const int rows = min(kBlockM, N - n0);
      const size_t base = static_cast<size_t>(bh) * N + n0;
      if (W == WP) {
        // the tile's rel_w rows are one contiguous, 16-byte aligned block
        // (WP is a multiple of 4) copied as it lies
        const float4* src = reinterpret_cast<const float4*>(args.rel_w + base * W);
        for (int e = t; e < rows * (WP / 4); e += kStg) cp_async16(buf + 4 * e, src + e);
      } else {
        // element e = rr W + c of the block goes to row rr, column c; (rr, c)
        // advanced without a division per element
        const int step_r = kStg / W, step_c = kStg - step_r * W;
        int rr = t / W, c = t - (t / W) * W;
        for (int e = t; e < rows * W; e += kStg) {
          cp_async4(buf + rr * WP + c, args.rel_w + base * W + e, 4u);
          rr += step_r;
          c += step_c;
          if (c >= W) {
            c -= W;
            ++rr;
          }
        }
      }
      // whole 128-column rows of the rel_h term (16-byte chunks), one per grid row
      const size_t np = static_cast<size_t>(n_qt) * kBlockM;
      const float* hl = args.hl + (static_cast<size_t>(bh) * H + j * KHT) * np + n0;
      for (int e = t; e < KHT * (kBlockM / 4); e += kStg) {
        const int gg = e / (kBlockM / 4), c = e - gg * (kBlockM / 4);
        if (j * KHT + gg < H) cp_async16(buf + (64 + gg) * RS + 4 * c, hl + gg * np + 4 * c);
      }
      if (t < kBlockM) cp_async4(buf + 72 * RS + t, args.D + (t < rows ? base + t : 0), t < rows ? 4u : 0u);
    };
    uint32_t stg_phase = 0;
    auto group_sync = [&]() -> bool {
      mbar_arrive(&bars[kBwStg]);
      const bool w = mbar_wait(&bars[kBwStg], stg_phase & 1, abort_flag, status);
      ++stg_phase;
      return warp_all(w);
    };
    bool ok = true;
    stage(0, 0);
    for (int i = 0; i < n_qt; ++i) {
      // this tile's staging has landed everywhere, and every thread is done
      // with the previous tile's buffer, which the next prefetch overwrites
      cp_async_wait_all();
      ok = group_sync();
      if (!ok) break;
      if (i + 1 < n_qt) stage(i + 1, (i + 1) & 1);
      const float* buf = stage_base + (i & 1) * kBufFloats;
      const float* rw = buf + 48 * part * WP + kw;   // rel_w of this part's first query column
      const float* rhT = buf + (64 + g) * RS;     // g < 8 for every key slot
      const float* DT = buf + 72 * RS;
      const int rows = min(kBlockM, N - i * kBlockM);
      const bool full = rows == kBlockM;
      ok = warp_all(mbar_wait(&bars[kBwSFull], i & 1, abort_flag, status));
      if (!ok) break;
      tc_fence_after();
      // this part's 16-column blocks; the next block's S^T and dP^T loads are
      // in flight while the current one is computed
      const int c_first = 48 * part;
      const float2 sl2v = make_float2(sl2, sl2), l2ev = make_float2(kLog2e, kLog2e);
      uint32_t us[2][16], up[2][16];
      tmem_ld16(tS + c_first, us[0]);
      tmem_ld16(tdP + c_first, up[0]);
      #pragma unroll
      for (int q = 0; q < 3; ++q) {
        if (q == nb) break;
        const int cb = c_first + 16 * q;
        tmem_wait_ld();
        if (q + 1 < nb) {
          tmem_ld16(tS + cb + 16, us[(q + 1) & 1]);
          tmem_ld16(tdP + cb + 16, up[(q + 1) & 1]);
        } else {
          // all of this thread's S^T(i) and dP^T(i) is in registers
          tc_fence_before();
          mbar_arrive(&bars[kBwSFree]);
        }
        uint32_t pp[8], pz[8];
        #pragma unroll
        for (int k4 = 0; k4 < 16; k4 += 4) {
          const int c4 = cb + k4;
          const int cr = 16 * q + k4;   // query column c4, counted from this part's first
          const float4 w4 = make_float4(rw[cr * WP], rw[(cr + 1) * WP], rw[(cr + 2) * WP], rw[(cr + 3) * WP]);
          const float4 h4 = *reinterpret_cast<const float4*>(rhT + c4);
          const float4 d4 = *reinterpret_cast<const float4*>(DT + c4);
          // Query columns past N must not reach dv or dk; key slots without a key
          // need no mask, since their P^T and dZ^T rows only reach their own
          // (unstored) rows of dv and dk.  Pairs of columns go through the packed
          // fp32x2 units.
          #pragma unroll
          for (int hp = 0; hp < 4; hp += 2) {
            const float2 w2 = hp == 0 ? make_float2(w4.x, w4.y) : make_float2(w4.z, w4.w);
            const float2 h2 = hp == 0 ? make_float2(h4.x, h4.y) : make_float2(h4.z, h4.w);
            const float2 nd2 = hp == 0 ? make_float2(d4.x, d4.y) : make_float2(d4.z, d4.w);   // -D
            const float2 s2 = make_float2(__uint_as_float(us[q & 1][k4 + hp]), __uint_as_float(us[q & 1][k4 + hp + 1]));
            const float2 dp2 =
                make_float2(__uint_as_float(up[q & 1][k4 + hp]), __uint_as_float(up[q & 1][k4 + hp + 1]));
            const float2 x = ffma2(s2, sl2v, ffma2(w2, l2ev, h2));
            float2 p = make_float2(ex2_approx(x.x), ex2_approx(x.y));
            if (!full) {
              if (c4 + hp >= rows) p.x = 0.f;
              if (c4 + hp + 1 >= rows) p.y = 0.f;
            }
            const float2 z = __fmul2_rn(p, fadd2(dp2, nd2));
            pp[(k4 + hp) / 2] = pack_in(p.x, p.y, fmt);
            pz[(k4 + hp) / 2] = pack_in(z.x, z.y, fmt);
          }
        }
        if (q == 0 && i > 0) {
          // P^T(i-1) and dZ^T(i-1) have been read by dv and dk before they are overwritten
          ok = warp_all(mbar_wait(&bars[kBwMmaDone], (i - 1) & 1, abort_flag, status));
          if (!ok) {
            tmem_wait_ld();   // the next block's loads are in flight
            break;
          }
          tc_fence_after();
        }
        tmem_st8(tP + cb / 2, pp);
        tmem_st8(tdZ + cb / 2, pz);
      }
      if (!ok) break;
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars[kBwPFull]);
    }
    cp_async_wait_all();
    if (ok) ok = warp_all(mbar_wait(&bars[kBwMmaDone], (n_qt - 1) & 1, abort_flag, status));
    if (ok && part < 2) {
      tc_fence_after();
      uint32_t a[32];
      const size_t tok = static_cast<size_t>(bh) * N + static_cast<size_t>(kh) * W + kw;
      const float sc = args.scale;
      // tcgen05.ld is warp-collective: every lane loads, lanes with a key store;
      // the warps of part 0 write dv, those of part 1 dk
      const uint32_t tacc = part == 0 ? tdV : tdK;
      void* dst = part == 0 ? args.dv : args.dk;
      const float mul = part == 0 ? 1.0f : sc;
      #pragma unroll
      for (int h = 0; h < 2; ++h) {
        tmem_ld32(tacc + 32 * h, a);
        tmem_wait_ld();
        if (key_valid) {
          #pragma unroll
          for (int c = 0; c < 8; ++c)
            st_grad4(dst, tok * 64 + 32 * h + 4 * c, mul * __uint_as_float(a[4 * c]),
                     mul * __uint_as_float(a[4 * c + 1]), mul * __uint_as_float(a[4 * c + 2]),
                     mul * __uint_as_float(a[4 * c + 3]), args.grad_fmt);
        }
      }
    }
  }
  bwd_teardown(tbase, warp);
}

// Tables kernel: dT = the sum of the per-tile partials.  A CTA of 256 threads
// takes 32 consecutive outputs (coalesced reads); thread (o, c) adds the
// partials of tiles c, c + 8, ..., and the eight chunk sums are added in a
// fixed order, so the result never depends on scheduling.
__global__ void relpos_bwd_tables_kernel(const BwdArgs args, int n_blocks) {
  __shared__ float red[8][32];
  const int LH = 2 * args.H - 1, LW = 2 * args.W - 1;
  const int total = (LH + LW) * 64;
  const int ol = threadIdx.x & 31, chunk = threadIdx.x >> 5;
  const int o = blockIdx.x * 32 + ol;
  float acc = 0.f;
  if (o < total) {
    // eight loads in flight, then added in the same order as one at a time
    int b = chunk;
    for (; b + 56 < n_blocks; b += 64) {
      float v[8];
      #pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = args.parts[static_cast<size_t>(b + 8 * u) * total + o];
      #pragma unroll
      for (int u = 0; u < 8; ++u) acc += v[u];
    }
    for (; b < n_blocks; b += 8) acc += args.parts[static_cast<size_t>(b) * total + o];
  }
  red[chunk][ol] = acc;
  __syncthreads();
  if (chunk == 0 && o < total) {
    float v = red[0][ol];
    #pragma unroll
    for (int c = 1; c < 8; ++c) v += red[c][ol];
    if (o < LH * 64) args.dth[o] = v;
    else args.dtw[o - LH * 64] = v;
  }
}

}  // namespace dera
