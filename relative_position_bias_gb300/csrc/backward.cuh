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
// Four kernels, in stream order (the projection kernel of the forward first
// writes the compact rel_h, rel_w in fp32):
//   relpos_bwd_rows   one CTA per (head, 128-row query tile), key tiles streamed:
//                     S = q k^T and dP = dO v^T on the tensor core, P and dZ on
//                     the softmax warps (one thread per query row), dq_s += dZ k
//                     on the tensor core; writes D, scale * dq_s, drel_h, drel_w.
//   relpos_bwd_cols   one CTA per (head, key tile), query tiles streamed:
//                     S^T = k q^T and dP^T = v dO^T, P^T and dZ^T per key row,
//                     dv += P^T dO and dk += dZ^T q accumulated in TMEM.
//   relpos_bwd_bias   one CTA per (head, query tile): dq = dq_s + the bias part,
//                     and this tile's share of dT_h, dT_w (a partial per CTA).
//   relpos_bwd_tables sums the per-CTA partials in a fixed order.
// Nothing is accumulated with atomics, so the result does not depend on the
// order in which CTAs run.
#pragma once
#include <cfloat>

#include "common.cuh"

namespace dera {

constexpr int kBwdColsThreads = 320;  // warp 0 TMA, warp 1 MMA, warps 2-9 softmax (two per TMEM lane quarter)
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

__device__ __forceinline__ float ld_in(const void* p, size_t i, int fmt) {
  const unsigned short raw = reinterpret_cast<const unsigned short*>(p)[i];
  if (fmt == kBF16) return __uint_as_float(static_cast<uint32_t>(raw) << 16);
  return __half2float(__ushort_as_half(raw));
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
  kBwCount = kBwStg + 1
};
// rows kernel: a two-stage K/V ring; staging holds the rel_h rows and the
// bias-gradient accumulators, 3 x 128 rows of 65 floats
// (one group of softmax threads: a three-stage ring, and only the rel_h rows)
constexpr int kRowsGroupsCfg = 1;
using BwdRowsSmem = BwdSmem<kRowsGroupsCfg == 1 ? 3 : 2, (kRowsGroupsCfg == 1 ? 1 : 3) * 128 * 65 * 4>;
// cols kernel: a three-stage Q/dO ring; staging holds two buffers of one query
// tile's rel_w, rel_h entries, lse and D, transposed (74 rows of 132 floats each)
constexpr int kColsStageRow = 132;
constexpr int kColsStageFloats = 74 * kColsStageRow;
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
// Rows kernel: one CTA per (head, query tile).  From warp 2 on, the softmax
// threads: one per query row (TMEM lane), or, with two groups, two per row
// (warps w and w + 4 share TMEM lane quarter w % 4 and take the first and the
// second half of every key tile's 16-column blocks).  TMEM columns: S [0, 128),
// dP [128, 256), dZ in the input dtype as packed pairs [256, 320), the dZ k
// accumulator [320, 384).  The bias-gradient sums meet in shared memory, with
// at most two addends per entry, so their order does not change the result.
// Softmax thread groups of the rows kernel: 1 (one thread per query row) or 2
// (two per row, each taking half of every key tile's columns).  One measured as
// fast on the 64x64 grid and 5-10 % faster on the 40x40 grid and 14x14 windows.
constexpr int kRowsGroups = kRowsGroupsCfg;
constexpr int kBwdRowsThreads = 64 + 128 * kRowsGroups;

// Which 16-column blocks of a key tile a half of the rows kernel's softmax
// threads takes (see rows_softmax), and their order.
template <int WP, int HALF>
struct RowsSplit {
  static constexpr int kBlocks = KeyTile<WP, 64>::BN / 16, kHalf0 = (kBlocks + 1) / 2;
  __host__ __device__ static constexpr bool mine(int bb) {
    if (HALF == 2) return true;   // one group takes every block
    return WP == 64 ? ((16 * bb) % 64) / 32 == HALF : (HALF == 0 ? bb < kHalf0 : bb >= kHalf0);
  }
  __host__ __device__ static constexpr int next(int bb) {
    for (int x = bb + 1; x < kBlocks; ++x)
      if (mine(x)) return x;
    return kBlocks;
  }
  __host__ __device__ static constexpr int rank(int bb) {
    int c = 0;
    for (int x = 0; x < bb; ++x) c += mine(x) ? 1 : 0;
    return c;
  }
};

// The softmax role of the rows kernel for one group of threads: HALF 2 is the
// single group (every column); with two groups, HALF 0 and 1.  With 64 key
// columns per grid row the halves split every grid row's columns (kw below or
// above 32), so each thread keeps 32 rel_w terms and 32 column sums in
// registers; with narrower rows they split each key tile's 16-column blocks
// into a first and a second half.
template <int WP, bool BF16, int HALF>
__device__ __forceinline__ void rows_softmax(const BwdArgs& args, uint8_t* smem, uint64_t* bars,
                                             volatile int* abort_flag, uint32_t tbase, int warp, int lane, int bh,
                                             int qt) {
  using KT = KeyTile<WP, 64>;
  constexpr int KHT = KT::KHT, BN = KT::BN;
  using SM = BwdRowsSmem;
  constexpr int fmt = BF16 ? kBF16 : kF16;
  constexpr bool kAll = HALF == 2;   // a single group of softmax threads
  constexpr bool kSplitKw = WP == 64 && !kAll;
  constexpr int kLW = kSplitKw ? 32 : WP;              // rel_w terms a thread keeps
  constexpr int kKw0 = kSplitKw ? 32 * HALF : 0;       // first of them
  constexpr int kBlocks = BN / 16;
  int* status = args.status;
  const int n_kv = args.n_kv, H = args.H, W = args.W, N = args.N;
  const int wq = warp & 3;
  const int r = wq * 32 + lane;
  const int t = threadIdx.x - 64;          // index among the softmax threads
  const int n = qt * kBlockM + r;
  const bool row_valid = n < N;
  const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
  const uint32_t tS = tbase + lane_off, tdP = tS + 128, tdZ = tS + 256, tdQ = tS + 320;
  const size_t row = static_cast<size_t>(bh) * N + (row_valid ? n : 0);
  const float NEG_INF = -__int_as_float(0x7f800000);
  const float sl2 = args.scale_log2;
  float* stg = reinterpret_cast<float*>(smem + SM::kStaging);
  float* bh_row = stg + r * 65;                          // rel_h row (base 2)
  float* dRH_sm = stg + 128 * 65 + r * 65;               // per key grid row: sum over its columns
  float* dRW_sm = stg + 2 * 128 * 65 + r * 65;           // per key column: sum over grid rows
  const int Hpad = n_kv * KHT;
  if (HALF != 1) {
    for (int kh = 0; kh < Hpad; ++kh)
      bh_row[kh] = (kh < H) ? (row_valid ? kLog2e * args.rel_h[row * H + kh] : 0.f) : NEG_INF;
  }
  if (!kAll)
    for (int e = t; e < 2 * 128 * 65; e += kRowsGroups * kBlockM) stg[128 * 65 + e] = 0.f;
  float bw[kLW];
  #pragma unroll
  for (int i = 0; i < kLW; ++i) {
    const int kw = kKw0 + i;
    bw[i] = (kw < W) ? (row_valid ? kLog2e * args.rel_w[row * W + kw] : 0.f) : NEG_INF;
  }
  const float lse2 = row_valid ? args.lse[row] : 0.f;
  // D = dO . out for this row (out in fp32 or in the input dtype)
  float Dn = 0.f;
  if (row_valid) {
    for (int c = 0; c < 64; ++c) {
      const float o = args.out_fmt == kF32 ? reinterpret_cast<const float*>(args.out)[row * 64 + c]
                                            : ld_in(args.out, row * 64 + c, fmt);
      Dn = fmaf(ld_in(args.dout, row * 64 + c, fmt), o, Dn);
    }
    if (HALF != 1) args.D[row] = Dn;
  }
  uint32_t stg_phase = 0;
  auto group_sync = [&]() -> bool {
    mbar_arrive(&bars[kBwStg]);
    const bool w = mbar_wait(&bars[kBwStg], stg_phase & 1, abort_flag, status);
    ++stg_phase;
    return warp_all(w);
  };
  bool ok = kAll ? true : group_sync();   // bh_row written, accumulators cleared
  float dRW[kLW];
  #pragma unroll
  for (int i = 0; i < kLW; ++i) dRW[i] = 0.f;
  for (int j = 0; ok && j < n_kv; ++j) {
    float bhv[KHT];
    #pragma unroll
    for (int g = 0; g < KHT; ++g) bhv[g] = bh_row[j * KHT + g];
    ok = warp_all(mbar_wait(&bars[kBwSFull], j & 1, abort_flag, status));
    if (!ok) break;
    tc_fence_after();
    if (j > 0) {
      // dZ(j-1) has been read by its product before dZ(j) is written
      ok = warp_all(mbar_wait(&bars[kBwMmaDone], (j - 1) & 1, abort_flag, status));
      if (!ok) break;
      tc_fence_after();
    }
    float dRH[KHT];
    #pragma unroll
    for (int g = 0; g < KHT; ++g) dRH[g] = 0.f;
    // this half's blocks, the next block's S and dP loads in flight while the
    // current one is computed
    using RS = RowsSplit<WP, HALF>;
    uint32_t us[2][16], up[2][16];
    tmem_ld16(tS + 16 * RS::next(-1), us[0]);
    tmem_ld16(tdP + 16 * RS::next(-1), up[0]);
    #pragma unroll
    for (int bb = 0; bb < kBlocks; ++bb) {
      if (!RS::mine(bb)) continue;
      const int cb = 16 * bb;
      const int cur = RS::rank(bb) & 1;
      tmem_wait_ld();
      if (RS::next(bb) < kBlocks) {
        tmem_ld16(tS + 16 * RS::next(bb), us[cur ^ 1]);
        tmem_ld16(tdP + 16 * RS::next(bb), up[cur ^ 1]);
      }
      uint32_t pk[8];
      #pragma unroll
      for (int k = 0; k < 16; k += 2) {
        const int col = cb + k;
        const int g = col / WP, i = col % WP - kKw0;
        const float x0 = fmaf(__uint_as_float(us[cur][k]), sl2, bw[i] + bhv[g]) - lse2;
        const float x1 = fmaf(__uint_as_float(us[cur][k + 1]), sl2, bw[i + 1] + bhv[g]) - lse2;
        float d0 = ex2_approx(x0) * (__uint_as_float(up[cur][k]) - Dn);
        float d1 = ex2_approx(x1) * (__uint_as_float(up[cur][k + 1]) - Dn);
        if (!row_valid) d0 = d1 = 0.f;
        dRW[i] += d0;
        dRW[i + 1] += d1;
        dRH[g] += d0 + d1;
        pk[k / 2] = pack_in(d0, d1, fmt);
      }
      tmem_st8(tdZ + cb / 2, pk);
    }
    tmem_wait_st();
    tc_fence_before();
    mbar_arrive(&bars[kBwPFull]);
    if (kAll) {
      if (row_valid) {
        #pragma unroll
        for (int g = 0; g < KHT; ++g)
          if (j * KHT + g < H) args.drel_h[row * H + j * KHT + g] = dRH[g];
      }
    } else {
      // two addends per entry (one per half), so their order does not matter
      #pragma unroll
      for (int g = 0; g < KHT; ++g)
        if (j * KHT + g < H) atomicAdd(&dRH_sm[j * KHT + g], dRH[g]);
    }
  }
  if (kAll) {
    if (ok && row_valid) {
      #pragma unroll
      for (int i = 0; i < kLW; ++i)
        if (i < W) args.drel_w[row * W + i] = dRW[i];
    }
  } else if (kSplitKw) {
    // each half owns its columns
    if (ok && row_valid) {
      #pragma unroll
      for (int i = 0; i < kLW; ++i)
        if (kKw0 + i < W) args.drel_w[row * W + kKw0 + i] = dRW[i];
    }
  } else {
    #pragma unroll
    for (int i = 0; i < kLW; ++i)
      if (i < W) atomicAdd(&dRW_sm[i], dRW[i]);
  }
  if (!kAll) {
    if (ok) ok = group_sync();
    if (ok && row_valid) {
      if (HALF == 0)
        for (int kh = 0; kh < H; ++kh) args.drel_h[row * H + kh] = dRH_sm[kh];
      if (HALF == 1 && !kSplitKw)
        for (int kw = 0; kw < W; ++kw) args.drel_w[row * W + kw] = dRW_sm[kw];
    }
  }
  if (ok) ok = warp_all(mbar_wait(&bars[kBwMmaDone], (n_kv - 1) & 1, abort_flag, status));
  if (ok) {
    tc_fence_after();
    #pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      if (!kAll && hh != HALF) continue;
      uint32_t a[32];
      tmem_ld32(tdQ + 32 * hh, a);
      tmem_wait_ld();
      if (row_valid) {
        float4* dst = reinterpret_cast<float4*>(args.dq_s + row * 64 + 32 * hh);
        const float sc = args.scale;
        #pragma unroll
        for (int c = 0; c < 8; ++c)
          dst[c] = make_float4(sc * __uint_as_float(a[4 * c]), sc * __uint_as_float(a[4 * c + 1]),
                               sc * __uint_as_float(a[4 * c + 2]), sc * __uint_as_float(a[4 * c + 3]));
      }
    }
  }
}

template <int WP, bool BF16>
__global__ void __launch_bounds__(kBwdRowsThreads, 1)
relpos_bwd_rows_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                       const BwdArgs args) {
  using KT = KeyTile<WP, 64>;
  constexpr int KHT = KT::KHT, BN = KT::BN, KS = kRowsGroups == 1 ? 3 : 2;
  using SM = BwdRowsSmem;
  constexpr int fmt = BF16 ? kBF16 : kF16;
  extern __shared__ uint8_t smem_raw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const BwdCta cta = bwd_setup<SM>(smem_raw, warp, kRowsGroups * kBlockM);
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
    constexpr uint32_t id_dq = idesc_f16(kBlockM, 64, fmt, fmt, 0, 1);  // dZ k: the k tile N-major
    const uint64_t d_q = sdesc_sw128(smem_u32(smem + SM::kA), 16, 1024);
    const uint64_t d_do = sdesc_sw128(smem_u32(smem + SM::kB), 16, 1024);
    const uint64_t d_ring = sdesc_sw128(smem_u32(smem + SM::kRing), 16, 1024);
    constexpr uint32_t kStageStep = SM::kStage >> 4, kVOfs = kTileBytes >> 4;
    auto issue_dq = [&](int jj) {
      const int sp = jj % KS;
      #pragma unroll
      for (int k = 0; k < BN / 16; ++k)
        umma_ts_w(tbase + 320, tbase + 256 + 8 * k, d_ring + sp * kStageStep + 128 * k, id_dq,
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
        // the softmax threads have read S(j-1), dP(j-1) and written dZ(j-1)
        ok = warp_all(mbar_wait(&bars[kBwPFull], (j - 1) & 1, abort_flag, status));
        if (!ok) break;
        tc_fence_after();
        issue_dq(j - 1);
      }
      tc_fence_after();
      #pragma unroll
      for (int k = 0; k < 4; ++k)
        umma_ss_w(tbase + 0, d_q + 2 * k, d_ring + s * kStageStep + 2 * k, id_s, k > 0);
      #pragma unroll
      for (int k = 0; k < 4; ++k)
        umma_ss_w(tbase + 128, d_do + 2 * k, d_ring + s * kStageStep + kVOfs + 2 * k, id_s, k > 0);
      umma_commit_w(&bars[kBwSFull]);
    }
    if (ok && warp_all(mbar_wait(&bars[kBwPFull], (n_kv - 1) & 1, abort_flag, status))) {
      tc_fence_after();
      issue_dq(n_kv - 1);
    }
    // every product issued above completes before TMEM is released
    umma_commit_w(&bars[kBwQFull]);
    mbar_wait_budget(&bars[kBwQFull], 1, kWaitBudgetCycles);
    __syncwarp();
  } else if (kRowsGroups == 1) {
    rows_softmax<WP, BF16, 2>(args, smem, bars, abort_flag, tbase, warp, lane, bh, qt);
  } else if (((warp - 2) >> 2) == 0) {
    rows_softmax<WP, BF16, 0>(args, smem, bars, abort_flag, tbase, warp, lane, bh, qt);
  } else {
    rows_softmax<WP, BF16, 1>(args, smem, bars, abort_flag, tbase, warp, lane, bh, qt);
  }
  bwd_teardown(tbase, warp);
}

// ---------------------------------------------------------------------------
// Cols kernel: one CTA per (head, key tile of KHT grid rows); thread m of warps
// 2-5 owns key slot m of the tile (TMEM lane m; slots past the tile's BN keys,
// padded columns and padded grid rows compute nothing that is stored).  TMEM
// columns: S^T [0, 128), dP^T [128, 256), P^T and dZ^T in the input dtype as
// packed pairs [256, 320) and [320, 384), dv [384, 448), dk [448, 512).
// Per query tile the softmax threads stage (cp.async, one tile ahead) the
// tile's rel_w rows [128][W], its rel_h entries for this key tile's grid rows
// [128][KHT], lse and D.
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
  const BwdCta cta = bwd_setup<SM>(smem_raw, warp, 2 * kBlockM);
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
        ok = warp_all(mbar_wait(&bars[kBwPFull], (i - 1) & 1, abort_flag, status));
        if (!ok) break;
        tc_fence_after();
        issue_acc(i - 1);
      }
      tc_fence_after();
      #pragma unroll
      for (int k = 0; k < 4; ++k)
        umma_ss_w(tbase + 0, d_k + 2 * k, d_ring + s * kStageStep + 2 * k, id_s, k > 0);
      #pragma unroll
      for (int k = 0; k < 4; ++k)
        umma_ss_w(tbase + 128, d_v + 2 * k, d_ring + s * kStageStep + kDoOfs + 2 * k, id_s, k > 0);
      umma_commit_w(&bars[kBwSFull]);
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
    const int half = (warp - 2) >> 2;      // query columns [64 half, 64 half + 64) of every tile
    const int t = threadIdx.x - 64;        // index among the 256 staging threads
    const int g = m / WP, kw = m % WP;
    const int kh = j * KHT + g;
    const bool key_valid = m < BN && kw < W && kh < H;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tbase + lane_off, tdP = tS + 128, tP = tS + 256, tdZ = tS + 320, tdV = tS + 384,
                   tdK = tS + 448;
    const float sl2 = args.scale_log2;
    float* stage_base = reinterpret_cast<float*>(smem + SM::kStaging);
    // buffer b, transposed so that a thread reads four query columns at once:
    // rel_w [kw][n] in rows 0..63, rel_h [g][n] in rows 64..71, lse in row 72,
    // D in row 73 (rows of kColsStageRow floats; columns past N hold zeros)
    constexpr int kBufFloats = kColsStageFloats, RS = kColsStageRow;
    auto stage = [&](int i, int b) {
      float* buf = stage_base + b * kBufFloats;
      const int n0 = i * kBlockM;
      const int rows = min(kBlockM, N - n0);
      const size_t base = static_cast<size_t>(bh) * N + n0;
      // the tile's rel_w rows are one contiguous block: element e = rr W + c,
      // its (rr, c) advanced without a division per element
      const int step_r = (2 * kBlockM) / W, step_c = (2 * kBlockM) - step_r * W;
      int rr = t / W, c = t - (t / W) * W;
      for (int e = t; e < kBlockM * W; e += 2 * kBlockM) {
        cp_async4(buf + c * RS + rr, args.rel_w + (rr < rows ? base * W + e : 0), rr < rows ? 4u : 0u);
        rr += step_r;
        c += step_c;
        if (c >= W) {
          c -= W;
          ++rr;
        }
      }
      for (int e = t; e < kBlockM * KHT; e += 2 * kBlockM) {
        const int rr = e / KHT, gg = e - rr * KHT, khh = j * KHT + gg;
        const bool v = rr < rows && khh < H;
        cp_async4(buf + (64 + gg) * RS + rr, args.rel_h + (v ? (base + rr) * H + khh : 0), v ? 4u : 0u);
      }
      if (t < kBlockM) {
        cp_async4(buf + 72 * RS + t, args.lse + (t < rows ? base + t : 0), t < rows ? 4u : 0u);
      } else {
        const int u = t - kBlockM;
        cp_async4(buf + 73 * RS + u, args.D + (u < rows ? base + u : 0), u < rows ? 4u : 0u);
      }
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
      const float* rwT = buf + kw * RS;           // kw < WP <= 64
      const float* rhT = buf + (64 + g) * RS;     // g < 8 for every key slot
      const float* lseT = buf + 72 * RS;
      const float* DT = buf + 73 * RS;
      const int rows = min(kBlockM, N - i * kBlockM);
      const bool full = rows == kBlockM;
      ok = warp_all(mbar_wait(&bars[kBwSFull], i & 1, abort_flag, status));
      if (!ok) break;
      tc_fence_after();
      if (i > 0) {
        ok = warp_all(mbar_wait(&bars[kBwMmaDone], (i - 1) & 1, abort_flag, status));
        if (!ok) break;
        tc_fence_after();
      }
      // this half's four 16-column blocks; the next block's S^T and dP^T
      // loads are in flight while the current one is computed
      const int c_first = 64 * half;
      uint32_t us[2][16], up[2][16];
      tmem_ld16(tS + c_first, us[0]);
      tmem_ld16(tdP + c_first, up[0]);
      #pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int cb = c_first + 16 * q;
        tmem_wait_ld();
        if (q < 3) {
          tmem_ld16(tS + cb + 16, us[(q + 1) & 1]);
          tmem_ld16(tdP + cb + 16, up[(q + 1) & 1]);
        }
        uint32_t pp[8], pz[8];
        #pragma unroll
        for (int k4 = 0; k4 < 16; k4 += 4) {
          const int c4 = cb + k4;
          const float4 w4 = *reinterpret_cast<const float4*>(rwT + c4);
          const float4 h4 = *reinterpret_cast<const float4*>(rhT + c4);
          const float4 l4 = *reinterpret_cast<const float4*>(lseT + c4);
          const float4 d4 = *reinterpret_cast<const float4*>(DT + c4);
          const float bw4[4] = {w4.x + h4.x, w4.y + h4.y, w4.z + h4.z, w4.w + h4.w};
          const float ls4[4] = {l4.x, l4.y, l4.z, l4.w};
          const float dd4[4] = {d4.x, d4.y, d4.z, d4.w};
          // Query columns past N must not reach dv or dk; key slots without a key
          // need no mask, since their P^T and dZ^T rows only reach their own
          // (unstored) rows of dv and dk.
          float p4[4], z4[4];
          #pragma unroll
          for (int h = 0; h < 4; ++h) {
            const float x = fmaf(__uint_as_float(us[q & 1][k4 + h]), sl2, fmaf(bw4[h], kLog2e, -ls4[h]));
            const float p = (full || c4 + h < rows) ? ex2_approx(x) : 0.f;
            p4[h] = p;
            z4[h] = p * (__uint_as_float(up[q & 1][k4 + h]) - dd4[h]);
          }
          pp[k4 / 2] = pack_in(p4[0], p4[1], fmt);
          pp[k4 / 2 + 1] = pack_in(p4[2], p4[3], fmt);
          pz[k4 / 2] = pack_in(z4[0], z4[1], fmt);
          pz[k4 / 2 + 1] = pack_in(z4[2], z4[3], fmt);
        }
        tmem_st8(tP + cb / 2, pp);
        tmem_st8(tdZ + cb / 2, pz);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars[kBwPFull]);
    }
    cp_async_wait_all();
    if (ok) ok = warp_all(mbar_wait(&bars[kBwMmaDone], (n_qt - 1) & 1, abort_flag, status));
    if (ok) {
      tc_fence_after();
      uint32_t a[32];
      const size_t tok = static_cast<size_t>(bh) * N + static_cast<size_t>(kh) * W + kw;
      const float sc = args.scale;
      // tcgen05.ld is warp-collective: every lane loads, lanes with a key store;
      // the first half of the warps writes dv, the second dk
      const uint32_t tacc = half == 0 ? tdV : tdK;
      void* dst = half == 0 ? args.dv : args.dk;
      const float mul = half == 0 ? 1.0f : sc;
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

// ---------------------------------------------------------------------------
// Bias kernel: one CTA of 256 threads per (head, query tile).  Adds the bias
// part of dq to dq_s and writes dq; writes this tile's partial table gradients.
// Tables, q rows and the bias gradients of the tile are staged in shared
// memory in fp32; rows of the tables and of q are 16-byte aligned (stride 68
// floats) so that each thread reads them four columns at a time.
constexpr int kBiasThreads = 256;
constexpr int kTStride = 68;

__host__ __device__ constexpr int bias_smem_floats(int H, int W) {
  return (2 * H - 1 + 2 * W - 1) * kTStride + 128 * (H + 1) + 128 * (W + 1) + 128 * kTStride + 2 * 128;
}

// dT partial of one 4 x 4 block: table rows i0..i0+3 of a table of length L
// (2 Lg - 1 rows for grid side Lg), columns c0..c0+3, over the tile's rows:
// acc[u][*] = sum_r [0 <= kk < Lg] dR[r][kk] q[r][c0..c0+3], kk = coord(r) - (i0 + u) + Lg - 1.
__device__ __forceinline__ void table_block(const float* dR, int ld, const int* coord, int Lg, const float* Qf,
                                            int rows, int i0, int c0, float (&acc)[4][4]) {
  #pragma unroll
  for (int u = 0; u < 4; ++u)
    #pragma unroll
    for (int k = 0; k < 4; ++k) acc[u][k] = 0.f;
  #pragma unroll 4
  for (int rr = 0; rr < rows; ++rr) {
    const int kk0 = coord[rr] - i0 + Lg - 1;
    const float4 qv = *reinterpret_cast<const float4*>(Qf + rr * kTStride + c0);
    #pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int kk = kk0 - u;
      const float wv = static_cast<unsigned>(kk) < static_cast<unsigned>(Lg) ? dR[rr * ld + kk] : 0.f;
      acc[u][0] = fmaf(wv, qv.x, acc[u][0]);
      acc[u][1] = fmaf(wv, qv.y, acc[u][1]);
      acc[u][2] = fmaf(wv, qv.z, acc[u][2]);
      acc[u][3] = fmaf(wv, qv.w, acc[u][3]);
    }
  }
}

__global__ void __launch_bounds__(kBiasThreads, 1) relpos_bwd_bias_kernel(const BwdArgs args) {
  extern __shared__ __align__(16) float fsm[];
  const int H = args.H, W = args.W, N = args.N;
  const int bh = blockIdx.x / args.n_qtiles, qt = blockIdx.x - bh * args.n_qtiles;
  const int n0 = qt * kBlockM;
  const int rows = min(kBlockM, N - n0);
  const int LH = 2 * H - 1, LW = 2 * W - 1;
  float* Th = fsm;
  float* Tw = Th + LH * kTStride;
  float* Qf = Tw + LW * kTStride;                  // [128][68]
  float* dRh = Qf + 128 * kTStride;                // [128][H + 1]
  float* dRw = dRh + 128 * (H + 1);                // [128][W + 1]
  int* qhv = reinterpret_cast<int*>(dRw + 128 * (W + 1));
  int* qwv = qhv + 128;
  const int t = threadIdx.x;
  const size_t base = static_cast<size_t>(bh) * N + n0;
  for (int e = t; e < LH * 64; e += kBiasThreads) Th[(e >> 6) * kTStride + (e & 63)] = ld_in(args.th, e, args.in_fmt);
  for (int e = t; e < LW * 64; e += kBiasThreads) Tw[(e >> 6) * kTStride + (e & 63)] = ld_in(args.tw, e, args.in_fmt);
  for (int e = t; e < 128 * H; e += kBiasThreads) {
    const int rr = e / H, c = e - rr * H;
    dRh[rr * (H + 1) + c] = rr < rows ? args.drel_h[base * H + e] : 0.f;
  }
  for (int e = t; e < 128 * W; e += kBiasThreads) {
    const int rr = e / W, c = e - rr * W;
    dRw[rr * (W + 1) + c] = rr < rows ? args.drel_w[base * W + e] : 0.f;
  }
  for (int e = t; e < 128 * 64; e += kBiasThreads) {
    const int rr = e >> 6;
    Qf[rr * kTStride + (e & 63)] = rr < rows ? ld_in(args.q, base * 64 + e, args.in_fmt) : 0.f;
  }
  if (t < 128) {
    const int n = n0 + t;
    qhv[t] = n / W;
    qwv[t] = n - (n / W) * W;
  }
  __syncthreads();
  // dq = dq_s + sum_kh drel_h T_h[qh - kh + H - 1] + sum_kw drel_w T_w[qw - kw + W - 1];
  // a warp holds 32 consecutive rows (mostly one qh, so one T_h row) and one half of the columns
  {
    const int rr = t & 127, c0 = (t >> 7) * 32;
    if (rr < rows) {
      const int qh = qhv[rr], qw = qwv[rr];
      float4 acc[8];
      const float4* src = reinterpret_cast<const float4*>(args.dq_s + (base + rr) * 64 + c0);
      #pragma unroll
      for (int c = 0; c < 8; ++c) acc[c] = src[c];
      for (int kh = 0; kh < H; ++kh) {
        const float wv = dRh[rr * (H + 1) + kh];
        const float4* tr = reinterpret_cast<const float4*>(Th + (qh - kh + H - 1) * kTStride + c0);
        #pragma unroll
        for (int c = 0; c < 8; ++c) {
          const float4 v = tr[c];
          acc[c] = make_float4(fmaf(wv, v.x, acc[c].x), fmaf(wv, v.y, acc[c].y), fmaf(wv, v.z, acc[c].z),
                               fmaf(wv, v.w, acc[c].w));
        }
      }
      for (int kw = 0; kw < W; ++kw) {
        const float wv = dRw[rr * (W + 1) + kw];
        const float4* tr = reinterpret_cast<const float4*>(Tw + (qw - kw + W - 1) * kTStride + c0);
        #pragma unroll
        for (int c = 0; c < 8; ++c) {
          const float4 v = tr[c];
          acc[c] = make_float4(fmaf(wv, v.x, acc[c].x), fmaf(wv, v.y, acc[c].y), fmaf(wv, v.z, acc[c].z),
                               fmaf(wv, v.w, acc[c].w));
        }
      }
      #pragma unroll
      for (int c = 0; c < 8; ++c)
        st_grad4(args.dq, (base + rr) * 64 + c0 + 4 * c, acc[c].x, acc[c].y, acc[c].z, acc[c].w, args.grad_fmt);
    }
  }
  // this tile's partial table gradients, in blocks of 4 table rows x 4 columns
  float* part = args.parts + static_cast<size_t>(blockIdx.x) * (LH + LW) * 64;
  const int hb = (LH + 3) / 4, wb = (LW + 3) / 4;
  for (int b = t; b < (hb + wb) * 16; b += kBiasThreads) {
    const int ib = b >> 4, c0 = (b & 15) * 4;
    const bool is_h = ib < hb;
    const int i0 = 4 * (is_h ? ib : ib - hb);
    const int L = is_h ? LH : LW;
    float acc[4][4];
    if (is_h) table_block(dRh, H + 1, qhv, H, Qf, rows, i0, c0, acc);
    else table_block(dRw, W + 1, qwv, W, Qf, rows, i0, c0, acc);
    float* dst = part + (is_h ? 0 : LH * 64);
    #pragma unroll
    for (int u = 0; u < 4; ++u)
      if (i0 + u < L)
        *reinterpret_cast<float4*>(dst + (i0 + u) * 64 + c0) = make_float4(acc[u][0], acc[u][1], acc[u][2], acc[u][3]);
  }
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
  if (o < total)
    for (int b = chunk; b < n_blocks; b += 8) acc += args.parts[static_cast<size_t>(b) * total + o];
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
