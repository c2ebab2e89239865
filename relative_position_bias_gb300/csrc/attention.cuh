// Global self-attention with decomposed relative-position bias on tcgen05.
//
// Computes, for every (batch*head) b and token n = qh*W + qw,
//   out[b, n] = sum_m softmax_m(scale * q_n.k_m + rel_h[n, kh(m)] + rel_w[n, kw(m)]) v_m
// without materialising the HW x HW bias (vLLM PR #55629 page, sections
// 实现拆解 item 1 and 关键源码片段).  The softmax is online, in base 2, with
// fp32 statistics (section 风险与影响).
//
// Work unit: one 128-row query tile of one head.  The kernel is persistent:
// all but the last one-and-a-fraction waves of units run as data-parallel
// rounds, the rest as a stream-K tail of (unit, key tile) iterations cut into
// one equal-cost range per CTA.  A unit cut between two CTAs: the piece that
// finishes first publishes its partial result (unnormalised O, row max, row
// sum) to the caller's workspace; the piece that finishes second merges.
//
// Every key tile is split by columns into two halves of whole grid rows.  Each
// half is an independent online softmax over its keys, run by its own four
// warps (one thread per row), with its own running maximum, row sum and O
// accumulator in TMEM; the two are merged once, at the end of the segment.  So
// the eight softmax warps share every tile without exchanging anything per tile.
//
// Warp roles (384 threads; warps 0-3 run with 104 registers, the softmax
// warps with 200, set by setmaxnreg):
//   warp 0      TMA producer: Q tile, [tables,] K ring and V ring
//   warp 1      tcgen05.mma issuer (the warp walks the loop, an elected lane issues)
//   warp 2      TMEM allocator; with warp 3, converts bf16 V tiles to fp16
//   warps 4-7   softmax of column half 0 (grid rows 0 .. KHT/2 - 1 of each tile)
//   warps 8-11  softmax of column half 1
// TMEM (512 columns): S0 [0,128) S1 [128,256)   scores of key tiles t (t even / odd)
//                     P0 [256,320) P1 [320,384) fp16 P of tiles t (even / odd), half h at +HALF/2*h
//                     O_0 [384,448) O_1 [448,512) unnormalised output of half 0 / half 1
// S and P are double-buffered, so QK^T of tile t + 2 is issued as soon as both
// halves have read S(t), never behind a P.V product; the fused prologue's
// q.table^T products use S0 and S1 before the segment's first QK^T.
//
// Softmax range: each tile is exponentiated against the half's running
// maximum and P is rounded to fp16.  A segment's first tile starts the maximum
// from a rel_h-aware estimate that may sit up to kStartCap above the exact
// maximum; later tiles are exponentiated at once and redone exactly only if
// their row sum passes kSpecSumLimit.  At the end of a segment the merged row
// sum l (in units of the final maximum) bounds the error that fp16 rounding
// and flushing of P can cause: at most 2^-11 relative, plus 2^-25 per key
// over l.  A segment whose l falls below kMinRowSum on any row is not stored;
// it is run again at the end of the CTA's work with no overshoot (cap 0),
// which keeps l >= 1, and the CTA's later segments use cap 0 as well.
#pragma once
#include <cfloat>

#include "common.cuh"

namespace dera {

constexpr int kTilesPerUnit = 1;  // 128-row query tiles per work unit
constexpr int kRing = 5;          // depth of the K ring and of the V ring
constexpr int kAttnThreads = 384;
// Largest accepted row sum of a speculative tile: with the sum at most this,
// every p rounds to at most 65504, the largest finite fp16.
constexpr float kSpecSumLimit = 65000.0f;
// Starting row maximum of a segment (base 2): at most kStartCap above the
// exact maximum of its first key tile; kStartMargin below the estimate.
constexpr float kStartCap = 12.0f;
constexpr float kStartMargin = 4.0f;
// Smallest accepted merged row sum at the end of a segment (see above).
constexpr float kMinRowSum = 0.25f;
constexpr int kBiasStride = 66;       // floats per row of the bias staging area
// Register split: the producer / MMA / V-conversion warpgroup gives registers
// back and the softmax warps take them.  The block launches with kLaunchRegs
// per thread (the most that 384 threads get); the host checks the compiled
// count before the first launch, since a split larger than the launch pool
// would block forever.
constexpr int kLaunchRegs = 168;
constexpr int kRegsCtl = 104;
constexpr int kRegsSmx = 200;
static_assert(kRegsCtl * 128 + kRegsSmx * 256 <= kLaunchRegs * kAttnThreads, "register split exceeds the launch pool");
static_assert(kRegsCtl % 8 == 0 && kRegsSmx % 8 == 0, "setmaxnreg counts are multiples of 8");

struct AttnSmem {
  static constexpr int kQ = 0;                                    // 16 KB
  static constexpr int kK = kTileBytes;                           // kRing x 16 KB
  static constexpr int kV = kK + kRing * kTileBytes;              // kRing x 16 KB
  static constexpr int kBias = kV + kRing * kTileBytes;           // 128 x 66 floats
  static constexpr int kBiasBytes = kBlockM * kBiasStride * 4;
  static constexpr int kXchg = kBias + kBiasBytes;                // [2 halves][128] float2 (m, l)
  static constexpr int kXchgBytes = 2 * kBlockM * 8;
  static constexpr int kBars = kXchg + kXchgBytes;
  static constexpr int kNumBars = 48;
  static constexpr int kMisc = kBars + kNumBars * 8;              // flags and the replay segment
  static constexpr int kTotal = kMisc + 64;
  static constexpr int kAlloc = kTotal + 1024;                    // slack for 1 KB alignment
};
static_assert(AttnSmem::kAlloc <= 232448, "shared memory budget");

// barrier indices
enum : int {
  kBarQFull = 0,
  kBarQEmpty = 1,
  kBarKFull = 2,                        // + ring slot
  kBarKEmpty = kBarKFull + kRing,
  kBarVFull = kBarKEmpty + kRing,
  kBarVEmpty = kBarVFull + kRing,
  kBarVReady = kBarVEmpty + kRing,
  kBarSFull = kBarVReady + kRing,       // + S buffer
  kBarPFull = kBarSFull + 2,            // + 2 * half + P buffer
  kBarODone = kBarPFull + 4,            // + 2 * half + P buffer
  kBarGFull = kBarODone + 4,
  kBarGFree = kBarGFull + 1,
  kBarEpiDone = kBarGFree + 1,
  kBarXchg = kBarEpiDone + 1,
  kBarMergeGo = kBarXchg + 1,
  kBarPartWritten = kBarMergeGo + 1,
  kBarDecision = kBarPartWritten + 1,
  kBarMmaDone = kBarDecision + 1,
  kBarCount = kBarMmaDone + 1
};
static_assert(kBarCount <= AttnSmem::kNumBars, "barrier slots");

// Work schedule over G persistent CTAs: all but the last one-and-a-fraction
// waves of units run as data-parallel rounds (CTA c takes unit r*G + c in
// round r, so the CTAs active together work on consecutive units, i.e. on the
// same heads, and share those heads' K/V in L2); the remaining G + (U mod G)
// units form a stream-K tail whose (unit, key tile) iterations are cut into G
// contiguous ranges.  With U a multiple of G the tail is one whole unit per
// CTA and nothing is cut.  Iterations are numbered globally:
// t = unit * n_kv + key tile.
//
// The tail ranges are equal in cost rather than in key tiles: each segment
// a CTA starts costs about kSegCost key tiles (prologue, epilogue, pipeline
// refill), so the tail is cut evenly in a virtual space where every unit is
// kSegCost slots of "segment start" followed by its n_kv key tiles.  Each
// range still spans at least n_kv + kSegCost virtual slots, so no unit is cut
// into more than two segments.
struct Schedule {
  static constexpr int kSegCost = 8;
  int G, n_kv, dp_rounds;
  long long sk_base, V;  // first tail iteration; tail length in virtual slots
  __device__ __forceinline__ Schedule(int U, int G_, int n_kv_) : G(G_), n_kv(n_kv_) {
    dp_rounds = max(U / G - 1, 0);
    sk_base = static_cast<long long>(dp_rounds) * G * n_kv;
    V = static_cast<long long>(U - dp_rounds * G) * (n_kv + kSegCost);
  }
  // tail iteration (relative to sk_base) at virtual slot v, 0 <= v <= V
  __device__ __forceinline__ long long real_of(long long v) const {
    const long long per = n_kv + kSegCost;
    const long long u = v / per, o = v - u * per;
    return u * n_kv + max(0LL, o - kSegCost);
  }
  __device__ __forceinline__ long long begin(int c) const {
    return sk_base + real_of(static_cast<long long>(c) * V / G);
  }
  // CTA whose tail range holds iteration t (t >= sk_base)
  __device__ __forceinline__ int cta_of(long long t) const {
    const long long tr = t - sk_base, u = tr / n_kv;
    const long long v = u * (n_kv + kSegCost) + kSegCost + (tr - u * n_kv);
    int c = static_cast<int>(min(static_cast<long long>(G - 1), v * G / V));
    while (c + 1 < G && begin(c + 1) <= t) ++c;
    while (c > 0 && begin(c) > t) --c;
    return c;
  }
};

// One segment of a CTA's work: key tiles [j0, j1) of unit u; tail = index of
// the segment within the CTA's stream-K range (-1 for a data-parallel unit).
struct Segment {
  int u, j0, j1, tail;
  __device__ __forceinline__ bool full(int n_kv) const { return j0 == 0 && j1 == n_kv; }
};

// Walks one CTA's segments in order; every role of the CTA walks the same list.
struct Cursor {
  int c, round, tail;
  long long it, end;
  __device__ __forceinline__ Cursor(const Schedule& s, int c_)
      : c(c_), round(0), tail(0), it(s.begin(c_)), end(s.begin(c_ + 1)) {}
  __device__ __forceinline__ bool next(const Schedule& s, Segment& sg) {
    if (round < s.dp_rounds) {
      sg.u = round * s.G + c;
      sg.j0 = 0;
      sg.j1 = s.n_kv;
      sg.tail = -1;
      ++round;
      return true;
    }
    if (it >= end) return false;
    sg.u = static_cast<int>(it / s.n_kv);
    sg.j0 = static_cast<int>(it - static_cast<long long>(sg.u) * s.n_kv);
    sg.j1 = static_cast<int>(min(static_cast<long long>(s.n_kv), sg.j0 + (end - it)));
    sg.tail = tail++;
    it += sg.j1 - sg.j0;
    return true;
  }
};

// Warp-uniform wait result: tcgen05.ld/st are warp-collective, so a warp
// either proceeds as a whole or stops as a whole.
__device__ __forceinline__ bool warp_all(bool ok) { return __all_sync(0xffffffffu, ok); }

__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
  const float lo = __uint_as_float(w << 16);
  const float hi = __uint_as_float(w & 0xFFFF0000u);
  return pack_f16x2(lo, hi);
}

// Shared-memory record of the segment a CTA has to run again (see the header).
struct ReplayRecord {
  int pending;   // 1 if a segment failed the row-sum check
  Segment sg;
};

template <int WP, bool FUSED, bool BF16>
__global__ void __launch_bounds__(kAttnThreads, 1)
    relpos_attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_th,
                       const __grid_constant__ CUtensorMap tm_tw, const AttnArgs args) {
  using KT = KeyTile<WP>;
  constexpr int KHT = KT::KHT;
  constexpr int BN = KT::BN;
  constexpr int HALF = KT::HALF;
  constexpr int GH = KT::GH;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_u + 1023u) & ~1023u) - raw_u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + AttnSmem::kBars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + AttnSmem::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + AttnSmem::kMisc + 4);
  volatile int* merge_flag = reinterpret_cast<volatile int*>(smem + AttnSmem::kMisc + 8);
  volatile int* bad_flag = reinterpret_cast<volatile int*>(smem + AttnSmem::kMisc + 12);   // [2], by segment parity
  ReplayRecord* replay = reinterpret_cast<ReplayRecord*>(smem + AttnSmem::kMisc + 32);
  int* status = args.status;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_kv = args.n_kv;
  const Schedule sched(args.n_units, static_cast<int>(gridDim.x), n_kv);
  constexpr bool convert_v = BF16;  // P is fp16, so bf16 V tiles are converted to fp16 on chip

  auto sQ = [&]() { return smem + AttnSmem::kQ; };
  auto sK = [&](int s) { return smem + AttnSmem::kK + s * kTileBytes; };
  auto sV = [&](int s) { return smem + AttnSmem::kV + s * kTileBytes; };

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    *merge_flag = 0;
    bad_flag[0] = 0;
    bad_flag[1] = 0;
    replay->pending = 0;
    mbar_init(&bars[kBarQFull], 1);
    mbar_init(&bars[kBarQEmpty], 1);
    for (int s = 0; s < kRing; ++s) {
      mbar_init(&bars[kBarKFull + s], 1);
      mbar_init(&bars[kBarKEmpty + s], 1);
      mbar_init(&bars[kBarVFull + s], 1);
      mbar_init(&bars[kBarVEmpty + s], 1);
      mbar_init(&bars[kBarVReady + s], 64);
    }
    for (int i = 0; i < 2; ++i) mbar_init(&bars[kBarSFull + i], 1);
    // P-ready and P.V-done barriers exist per P buffer: a half may finish tile
    // t + 1 before the MMA warp has looked at tile t, and a parity wait only
    // tolerates one completed phase it has not seen
    for (int i = 0; i < 4; ++i) {
      mbar_init(&bars[kBarPFull + i], kBlockM);
      mbar_init(&bars[kBarODone + i], 1);
    }
    mbar_init(&bars[kBarGFull], 1);
    mbar_init(&bars[kBarGFree], 2 * kBlockM);
    mbar_init(&bars[kBarEpiDone], 2 * kBlockM);
    mbar_init(&bars[kBarXchg], 2 * kBlockM);
    mbar_init(&bars[kBarMergeGo], 1);
    mbar_init(&bars[kBarPartWritten], 2 * kBlockM);
    mbar_init(&bars[kBarDecision], 2 * kBlockM);
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

  // Waits (bounded) until the softmax warps have decided whether a segment
  // must run again, then returns that segment (or false).
  auto replay_decision = [&](bool ok, Segment& sg) -> bool {
    if (!mbar_wait(&bars[kBarDecision], 0, abort_flag, status) || !ok) return false;
    if (!replay->pending) return false;
    sg = replay->sg;
    return true;
  };

  if (warp < 4) {
  regs_release<kRegsCtl>();
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      int rg = 0, seg = 0;
      bool ok = true;
      // ring slot rg % kRing; K and V of one tile share the index
      auto load_kv = [&](bool table, int j, int bh) -> bool {
        const int s = rg % kRing;
        const uint32_t ph = ((rg / kRing) & 1) ^ 1;
        if (!mbar_wait(&bars[kBarKEmpty + s], ph, abort_flag, status)) return false;
        if (table) {
          mbar_arrive_expect_tx(&bars[kBarKFull + s], kTileBytes);
          tma_load_2d(sK(s), &tm_th, &bars[kBarKFull + s], 0, 0);
        } else {
          mbar_arrive_expect_tx(&bars[kBarKFull + s], BN * kRowBytes);
          tma_load_4d(sK(s), &tm_k, &bars[kBarKFull + s], 0, 0, j * KHT, bh);
        }
        if (!mbar_wait(&bars[kBarVEmpty + s], ph, abort_flag, status)) return false;
        if (table) {
          mbar_arrive_expect_tx(&bars[kBarVFull + s], kTileBytes);
          tma_load_2d(sV(s), &tm_tw, &bars[kBarVFull + s], 0, 0);
        } else {
          mbar_arrive_expect_tx(&bars[kBarVFull + s], BN * kRowBytes);
          tma_load_4d(sV(s), &tm_v, &bars[kBarVFull + s], 0, 0, j * KHT, bh);
        }
        ++rg;
        return true;
      };
      auto run_seg = [&](const Segment& sg) -> bool {
        const int bh = sg.u / args.n_qtiles;
        const int qt = sg.u - bh * args.n_qtiles;
        if (seg > 0 && !mbar_wait(&bars[kBarQEmpty], (seg - 1) & 1, abort_flag, status)) return false;
        mbar_arrive_expect_tx(&bars[kBarQFull], kTileBytes);
        tma_load_3d(sQ(), &tm_q, &bars[kBarQFull], 0, qt * kBlockM, bh);
        ++seg;
        if (FUSED && !load_kv(true, 0, 0)) return false;
        for (int j = sg.j0; j < sg.j1; ++j)
          if (!load_kv(false, j, bh)) return false;
        return true;
      };
      Cursor cur(sched, blockIdx.x);
      Segment sg;
      while (ok && cur.next(sched, sg)) ok = run_seg(sg);
      if (replay_decision(ok, sg)) ok = run_seg(sg);
      if (!ok) {
        // Let the copies already in flight land before the CTA exits.
        if (seg > 0) mbar_wait_budget(&bars[kBarQFull], (seg - 1) & 1, kWaitBudgetCycles);
        for (int r = max(0, rg - kRing); r < rg; ++r) {
          mbar_wait_budget(&bars[kBarKFull + r % kRing], (r / kRing) & 1, kWaitBudgetCycles);
          mbar_wait_budget(&bars[kBarVFull + r % kRing], (r / kRing) & 1, kWaitBudgetCycles);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp walks the loop (waits and operand arithmetic are
    // warp-uniform); one elected lane issues each tcgen05 instruction.
    constexpr uint32_t fmt = BF16 ? kBF16 : kF16;
    constexpr uint32_t id_qk = idesc_f16(kBlockM, BN, fmt, fmt, 0, 0);
    constexpr uint32_t id_pv = idesc_f16(kBlockM, kHeadDim, kF16, kF16, 0, 1);
    constexpr uint32_t id_g = idesc_f16(kBlockM, 128, fmt, fmt, 0, 0);
    // Descriptors differ only in their 14-bit start-address field (address / 16),
    // which stays below 2^14 for any shared-memory address, so offsets are
    // added to one base descriptor per operand.
    const uint64_t d_q = sdesc_sw128(smem_u32(sQ()), 16, 1024);
    const uint64_t d_k = sdesc_sw128(smem_u32(sK(0)), 16, 1024);
    const uint64_t d_v = sdesc_sw128(smem_u32(sV(0)), 16, 1024);
    constexpr uint32_t kSlotStep = kTileBytes >> 4;
    int rg = 0, gt = 0, seg = 0;
    bool ok = true;
    // S(t) = Q K(t)^T into S buffer t % 2
    auto issue_qk = [&](int t_local, bool last) -> bool {
      const int s = (rg + t_local) % kRing;
      if (!warp_all(mbar_wait(&bars[kBarKFull + s], ((rg + t_local) / kRing) & 1, abort_flag, status))) return false;
      tc_fence_after();
      const uint32_t d = tbase + 128 * ((gt + t_local) & 1);
      const uint64_t b = d_k + s * kSlotStep;
      #pragma unroll
      for (int k = 0; k < 4; ++k) umma_ss_w(d, d_q + 2 * k, b + 2 * k, id_qk, k > 0);
      umma_commit_w(&bars[kBarSFull + ((gt + t_local) & 1)]);
      umma_commit_w(&bars[kBarKEmpty + s]);
      if (last) umma_commit_w(&bars[kBarQEmpty]);  // no more reads of this segment's Q
      return true;
    };
    // O_h (+)= P_h(t) V_h(t): half h's keys are rows [h*HALF, (h+1)*HALF) of the V tile
    auto issue_pv = [&](int h, int s, int b, bool acc) {
      const uint64_t vb = d_v + s * kSlotStep + ((h * HALF * kRowBytes) >> 4);
      const uint32_t pa = tbase + 256 + 64 * b + h * (HALF / 2);
      #pragma unroll
      for (int k = 0; k < HALF / 16; ++k)
        umma_ts_w(tbase + 384 + 64 * h, pa + 8 * k, vb + 128 * k, id_pv, (acc || k > 0) ? 1u : 0u);
      umma_commit_w(&bars[kBarODone + 2 * h + b]);
    };
    auto run_seg = [&](const Segment& sg) -> bool {
      const int len = sg.j1 - sg.j0;
      if (!warp_all(mbar_wait(&bars[kBarQFull], seg & 1, abort_flag, status))) return false;
      if (FUSED) {
        // G = Q [T_h ; T_w]^T into S0 | S1; both S buffers are free: every
        // earlier QK^T has been read by both halves (their P arrivals came first)
        const int s = rg % kRing;
        const uint32_t ph = (rg / kRing) & 1;
        if (!warp_all(mbar_wait(&bars[kBarKFull + s], ph, abort_flag, status))) return false;
        if (!warp_all(mbar_wait(&bars[kBarVFull + s], ph, abort_flag, status))) return false;
        tc_fence_after();
        #pragma unroll
        for (int k = 0; k < 4; ++k) umma_ss_w(tbase, d_q + 2 * k, d_k + s * kSlotStep + 2 * k, id_g, k > 0);
        #pragma unroll
        for (int k = 0; k < 4; ++k) umma_ss_w(tbase + 128, d_q + 2 * k, d_v + s * kSlotStep + 2 * k, id_g, k > 0);
        umma_commit_w(&bars[kBarGFull]);
        umma_commit_w(&bars[kBarKEmpty + s]);
        umma_commit_w(&bars[kBarVEmpty + s]);
        ++rg;
        if (!warp_all(mbar_wait(&bars[kBarGFree], seg & 1, abort_flag, status))) return false;
        tc_fence_after();
      }
      if (!issue_qk(0, len == 1)) return false;
      if (len > 1 && !issue_qk(1, len == 2)) return false;
      for (int jj = 0; jj < len; ++jj) {
        const int t = gt + jj, s = (rg + jj) % kRing, b = t & 1;
        const uint32_t ph = ((rg + jj) / kRing) & 1;
        if (!warp_all(mbar_wait(&bars[convert_v ? kBarVReady + s : kBarVFull + s], ph, abort_flag, status)))
          return false;
        if (!warp_all(mbar_wait(&bars[kBarPFull + b], (t >> 1) & 1, abort_flag, status))) return false;
        if (jj == 0 && seg > 0) {
          // the first P.V of a segment overwrites O: the previous epilogue must have read it
          if (!warp_all(mbar_wait(&bars[kBarEpiDone], (seg - 1) & 1, abort_flag, status))) return false;
        }
        tc_fence_after();
        issue_pv(0, s, b, jj > 0);
        if (!warp_all(mbar_wait(&bars[kBarPFull + 2 + b], (t >> 1) & 1, abort_flag, status))) return false;
        tc_fence_after();
        // both halves have read S(t): its buffer takes S(t + 2)
        if (jj + 2 < len && !issue_qk(jj + 2, jj + 3 == len)) return false;
        issue_pv(1, s, b, jj > 0);
        umma_commit_w(&bars[kBarVEmpty + s]);
      }
      gt += len;
      rg += len;
      ++seg;
      return true;
    };
    Cursor cur(sched, blockIdx.x);
    Segment sg;
    while (ok && cur.next(sched, sg)) ok = run_seg(sg);
    if (replay_decision(warp_all(ok), sg)) ok = run_seg(sg);
    // Drain: every MMA issued above completes before TMEM is released.
    umma_commit_w(&bars[kBarMmaDone]);
    mbar_wait_budget(&bars[kBarMmaDone], 0, kWaitBudgetCycles);
    __syncwarp();
  } else {
    // ------------------------------------------------------------ bf16 -> fp16 V conversion
    // The fused kernel's table slots are passed through unconverted, so that
    // v_ready completes once per ring index.
    if (convert_v) {
      const int ct = threadIdx.x - 64;
      int rg = 0;
      bool ok = true;
      auto run_seg = [&](const Segment& sg) -> bool {
        for (int j = FUSED ? sg.j0 - 1 : sg.j0; j < sg.j1; ++j, ++rg) {
          const int s = rg % kRing;
          if (!mbar_wait(&bars[kBarVFull + s], (rg / kRing) & 1, abort_flag, status)) return false;
          if (j >= sg.j0) {
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
        return true;
      };
      Cursor cur(sched, blockIdx.x);
      Segment sg;
      while (ok && cur.next(sched, sg)) ok = run_seg(sg);
      if (replay_decision(ok, sg)) run_seg(sg);
    }
  }
  } else {
    regs_claim<kRegsSmx>();
    // ------------------------------------------------------------ softmax / epilogue
    const int h = (warp - 4) >> 2;           // column half of this warp
    const int wq = warp & 3;                 // TMEM lane quarter
    const int r = wq * 32 + lane;            // row inside the query tile
    const int H = args.H, W = args.W, N = args.N;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tO0 = tbase + lane_off + 384;
    float* area = reinterpret_cast<float*>(smem + AttnSmem::kBias);
    float2* xchg = reinterpret_cast<float2*>(smem + AttnSmem::kXchg);   // [2][128] (m, l)
    const int Hpad = n_kv * KHT;
    const int HS = Hpad + 1;
    float* bh_row = area + r * HS;
    const float NEG_INF = -__int_as_float(0x7f800000);
    const float sl2 = args.scale_log2;
    const float2 sl2v = make_float2(sl2, sl2);
    const bool leader = warp == 4 && lane == 0;

    int gt = 0, seg = 0;
    uint32_t xph = 0;   // completed phases of the softmax-wide exchange barrier
    int pmerge = 0;     // completed phases of the merge-go barrier
    int ppub = 0;       // completed phases of the partial-written barrier
    float cap = kStartCap;
    bool ok = true;
    // Barrier of the 256 softmax threads (all arrive, then wait).
    auto sm_sync = [&]() -> bool {
      mbar_arrive(&bars[kBarXchg]);
      const bool w = mbar_wait(&bars[kBarXchg], xph & 1, abort_flag, status);
      ++xph;
      return warp_all(w);
    };

    auto run_seg = [&](const Segment& sg, bool is_replay) -> bool {
      const int bh = sg.u / args.n_qtiles;
      const int qt = sg.u - bh * args.n_qtiles;
      const int n = qt * kBlockM + r;
      const bool row_valid = n < N;
      const int qh = row_valid ? n / W : 0;
      const int qw = row_valid ? n - qh * W : 0;
      const int len = sg.j1 - sg.j0;

      // ---------------------------------------------------------------- prologue
      // every thread has finished with the previous segment's output staging
      // in the bias area before any row is written into it again
      if (seg > 0 && !sm_sync()) return false;
      float bw[WP];
      if (FUSED) {
        if (!warp_all(mbar_wait(&bars[kBarGFull], seg & 1, abort_flag, status))) return false;
        tc_fence_after();
        float* stg = area + r * kBiasStride;
        // rel_w row from G_w (TMEM columns 128..255), skewed into the staging
        // row; the row's two threads take alternate 32-column chunks
        skew_row_to_smem(tbase + lane_off + 128, qw, W, stg, kLog2e, h, 2);
        if (!sm_sync()) return false;
        #pragma unroll
        for (int kw = 0; kw < WP; ++kw) bw[kw] = kw < W ? stg[kw] : NEG_INF;
        // the staging rows (stride kBiasStride) overlap the bias rows (stride HS):
        // every thread has its rel_w row before any rel_h row is written
        if (!sm_sync()) return false;
        skew_row_to_smem(tbase + lane_off, qh, H, bh_row, kLog2e, h, 2);
        if (h == 0)
          for (int kh = H; kh < Hpad; ++kh) bh_row[kh] = NEG_INF;
        tc_fence_before();
        mbar_arrive(&bars[kBarGFree]);
        if (!sm_sync()) return false;
      } else {
        // The tile's rows of rel_w, then of rel_h, are one contiguous block
        // each: each of the eight warps copies every eighth row into the
        // staging area, a row per pass with the lanes along it (coalesced),
        // scaled by log2e.  Rows past N read as 0.
        const size_t row0 = static_cast<size_t>(bh) * N + static_cast<size_t>(qt) * kBlockM;
        const int nrows = min(kBlockM, N - qt * kBlockM);
        const int cw = warp - 4;   // copy warp 0..7
        // Loads for 4 rows go out together before any store (the stores could
        // alias the source as far as the compiler knows).
        auto copy_rows = [&](const void* src, int rlen, int stride) {
          for (int rb = cw; rb < kBlockM; rb += 32) {
            float v[4][2];
            #pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int rr = rb + 8 * u;
              #pragma unroll
              for (int k = 0; k < 2; ++k) {
                const int c = lane + 32 * k;
                v[u][k] = (rr < nrows && c < rlen)
                              ? load_elem(src, (row0 + rr) * static_cast<size_t>(rlen) + c, args.bias_fmt)
                              : 0.f;
              }
            }
            #pragma unroll
            for (int u = 0; u < 4; ++u) {
              #pragma unroll
              for (int k = 0; k < 2; ++k) {
                const int c = lane + 32 * k;
                if (c < rlen) area[(rb + 8 * u) * stride + c] = kLog2e * v[u][k];
              }
            }
          }
        };
        copy_rows(args.rel_w, W, kBiasStride);
        if (!sm_sync()) return false;
        const float* stg = area + r * kBiasStride;
        #pragma unroll
        for (int kw = 0; kw < WP; ++kw) bw[kw] = kw < W ? stg[kw] : NEG_INF;
        // every thread has its rel_w row before the area is reused for rel_h
        if (!sm_sync()) return false;
        copy_rows(args.rel_h, H, HS);
        if (h == 0)
          for (int kh = H; kh < Hpad; ++kh) bh_row[kh] = NEG_INF;
        if (!sm_sync()) return false;
      }

      // S is processed in blocks of 16 columns (one TMEM load and one wait each).
      // Exact maximum over this half of x = s*scale*log2e + rel_w*log2e + rel_h*log2e;
      // base = the same without the rel_h term.
      auto tile_max = [&](uint32_t tS, const float (&bhv)[GH], float& base) -> float {
        float gm[GH];
        #pragma unroll
        for (int g = 0; g < GH; ++g) gm[g] = NEG_INF;
        #pragma unroll
        for (int cb = 0; cb < HALF; cb += 16) {
          uint32_t u[16];
          tmem_ld16(tS + cb, u);
          tmem_wait_ld();
          #pragma unroll
          for (int k = 0; k < 16; k += 2) {
            const int col = cb + k;
            const int g = col / WP, kw = col % WP;
            const float2 t = ffma2(make_float2(__uint_as_float(u[k]), __uint_as_float(u[k + 1])), sl2v,
                                   make_float2(bw[kw], bw[kw + 1]));
            gm[g] = fmax3(gm[g], t.x, t.y);
          }
        }
        float mt = NEG_INF;
        base = NEG_INF;
        #pragma unroll
        for (int g = 0; g < GH; ++g) {
          mt = fmaxf(mt, gm[g] + bhv[g]);
          base = fmaxf(base, gm[g]);
        }
        return mt;
      };
      // p = 2^(x - m) for this half of the tile into P (fp16, TMEM); returns the
      // row sum.  S is read in 16-column blocks with the next block always in
      // flight; four partial sums keep the dependency chains short.  Before the
      // first P store, P.V of tile t - 2 (the last reader of this P buffer) has
      // completed.
      bool pfree_pending = false;
      auto wait_pfree = [&](int t) {
        if (pfree_pending) {
          ok = warp_all(mbar_wait(&bars[kBarODone + 2 * h + (t & 1)], ((t - 2) >> 1) & 1, abort_flag, status)) && ok;
          tc_fence_after();
          pfree_pending = false;
        }
      };
      auto exp_pass = [&](uint32_t tS, uint32_t tP, int t, const float (&bhv)[GH], float m) -> float2 {
        float2 off[GH];
        #pragma unroll
        for (int g = 0; g < GH; ++g) off[g] = make_float2(bhv[g] - m, bhv[g] - m);
        float2 ts[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                        make_float2(0.f, 0.f)};
        uint32_t ua[16], ub[16];
        auto block = [&](int cb, const uint32_t (&u)[16]) {
          uint32_t pk[8];
          #pragma unroll
          for (int k = 0; k < 16; k += 2) {
            const int col = cb + k;
            const int g = col / WP, kw = col % WP;
            float2 x = ffma2(make_float2(__uint_as_float(u[k]), __uint_as_float(u[k + 1])), sl2v,
                             make_float2(bw[kw], bw[kw + 1]));
            x = fadd2(x, off[g]);
            const float2 p = make_float2(ex2_approx(x.x), ex2_approx(x.y));
            ts[(k / 2) & 3] = fadd2(ts[(k / 2) & 3], p);
            pk[k / 2] = pack_f16x2(p.x, p.y);
          }
          if (cb == 0) wait_pfree(t);
          tmem_st8(tP + cb / 2, pk);
        };
        tmem_ld16(tS, ua);
        #pragma unroll
        for (int cb = 0; cb < HALF; cb += 32) {
          tmem_wait_ld();
          if (cb + 16 < HALF) tmem_ld16(tS + cb + 16, ub);
          block(cb, ua);
          if (cb + 16 < HALF) {
            tmem_wait_ld();
            if (cb + 32 < HALF) tmem_ld16(tS + cb + 32, ua);
            block(cb + 16, ub);
          }
        }
        return fadd2(fadd2(ts[0], ts[1]), fadd2(ts[2], ts[3]));
      };

      // Largest rel_h term (base 2) over this half's grid rows of the segment.
      float mbh = NEG_INF;
      for (int j = sg.j0; j < sg.j1; ++j) {
        #pragma unroll
        for (int g = 0; g < GH; ++g) mbh = fmaxf(mbh, bh_row[j * KHT + h * GH + g]);
      }

      // ---------------------------------------------------------------- tiles
      // Online softmax over the segment's key tiles.  The first tile takes the
      // exact maximum (raised by the rel_h estimate, at most `cap` above it);
      // later tiles exponentiate against the running maximum at once and are
      // redone exactly only if their row sum exceeds kSpecSumLimit.  The final
      // O / l uses the same running maximum, so skipping rescales changes nothing.
      float m_used = 0.f;
      float2 lsum = make_float2(0.f, 0.f);
      for (int jj = 0; jj < len; ++jj) {
        const int t = gt + jj;
        const int b = t & 1;
        const uint32_t tS = tbase + lane_off + 128 * b + h * HALF;
        const uint32_t tP = tbase + lane_off + 256 + 64 * b + h * (HALF / 2);
        if (!warp_all(mbar_wait(&bars[kBarSFull + b], (t >> 1) & 1, abort_flag, status))) return false;
        tc_fence_after();
        pfree_pending = t >= 2;
        const int kh0 = (sg.j0 + jj) * KHT + h * GH;
        float bhv[GH];
        #pragma unroll
        for (int g = 0; g < GH; ++g) bhv[g] = bh_row[kh0 + g];

        float2 ts = make_float2(0.f, 0.f);
        bool exact = jj == 0;
        if (!exact) {
          ts = exp_pass(tS, tP, t, bhv, m_used);
          exact = __any_sync(0xffffffffu, !(ts.x + ts.y <= kSpecSumLimit));
        }
        if (exact) {
          float base;
          const float mt = tile_max(tS, bhv, base);
          // rel_h is the term that moves the row maximum most between key
          // tiles, so start from this tile's largest s*scale + rel_w plus the
          // half's largest rel_h (less a margin), at most `cap` above the
          // exact maximum of this tile
          const float est = fminf(mt + cap, base + mbh - kStartMargin);
          if (jj == 0) {
            // A half can hold no valid key at all (the grid rows of a last,
            // partly padded tile); -FLT_MAX instead of -inf keeps x - m at
            // -inf there (p = 0), and the merge then weighs the half with 0.
            m_used = fmaxf(fmaxf(mt, est), -FLT_MAX);
          } else {
            const float m_new = fmaxf(fmaxf(m_used, mt), est);
            const float alpha = ex2_approx(m_used - m_new);
            m_used = m_new;
            lsum.x *= alpha;
            lsum.y *= alpha;
            // P.V of tile t - 1 (the last one into O_h) has completed
            ok = warp_all(mbar_wait(&bars[kBarODone + 2 * h + ((t - 1) & 1)], ((t - 1) >> 1) & 1, abort_flag,
                                    status)) && ok;
            tc_fence_after();
            const uint32_t tOh = tO0 + 64 * h;
            #pragma unroll
            for (int c = 0; c < 2; ++c) {
              uint32_t o[32];
              tmem_ld32(tOh + 32 * c, o);
              tmem_wait_ld();
              #pragma unroll
              for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
              tmem_st32(tOh + 32 * c, o);
            }
          }
          ts = exp_pass(tS, tP, t, bhv, m_used);
        }
        lsum = fadd2(lsum, ts);
        if (!ok) return false;
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bars[kBarPFull + 2 * h + b]);
      }

      // ---------------------------------------------------------------- epilogue
      // Both halves' last P.V products have completed (this thread reads both O halves).
      const int tl = gt + len - 1;
      for (int x = 0; x < 2; ++x)
        if (!warp_all(mbar_wait(&bars[kBarODone + 2 * x + (tl & 1)], (tl >> 1) & 1, abort_flag, status)))
          return false;
      tc_fence_after();
      // merge the halves: m* = max(m_0, m_1), l = f_0 l_0 + f_1 l_1 with f_x = 2^(m_x - m*)
      xchg[h * kBlockM + r] = make_float2(m_used, lsum.x + lsum.y);
      if (!sm_sync()) return false;
      const float2 ml0 = xchg[r], ml1 = xchg[kBlockM + r];
      const float mstar = fmaxf(ml0.x, ml1.x);
      const float f0 = ex2_approx(ml0.x - mstar), f1 = ex2_approx(ml1.x - mstar);
      const float l = f0 * ml0.y + f1 * ml1.y;
      volatile int* bad = bad_flag + (seg & 1);
      if (row_valid && !(l >= kMinRowSum)) *bad = 1;
      // this thread's 32 output columns [32h, 32h + 32) of both O halves
      uint32_t o0[32], o1[32];
      tmem_ld32(tO0 + 32 * h, o0);
      tmem_ld32(tO0 + 64 + 32 * h, o1);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&bars[kBarEpiDone]);
      if (!sm_sync()) return false;
      const bool seg_bad = *bad != 0;
      // every thread has read this segment's flag; the next segment's is cleared
      if (leader) bad_flag[(seg + 1) & 1] = 0;
      gt += len;
      ++seg;
      if (seg_bad && !is_replay) {
        // Too little of the row's mass above the fp16 range: nothing of this
        // segment is stored or published; the CTA runs it again at the end
        // with no overshoot, and its later segments use none either.  (With
        // no overshoot l >= 1 on every row of finite inputs, so the run again
        // always stores.)
        if (leader && !replay->pending) {
          replay->pending = 1;
          replay->sg = sg;
        }
        cap = 0.f;
        return true;
      }
      float v[32];
      #pragma unroll
      for (int k = 0; k < 32; ++k) v[k] = f0 * __uint_as_float(o0[k]) + f1 * __uint_as_float(o1[k]);

      // Output rows leave through the bias area (no thread reads bias rows
      // any more): each lane stages its 32 columns, 16-byte chunks XOR-swizzled
      // by row so neither side has bank conflicts, then the warp stores runs of
      // 512 contiguous bytes.
      const bool out32 = args.out_fmt == kF32;
      const int row_bytes = out32 ? 256 : 128;     // a whole output row in global memory
      const int part_bytes = row_bytes / 2;        // this thread's 32 columns
      uint8_t* ostage = reinterpret_cast<uint8_t*>(area) + (h * 4 + wq) * 32 * 128;
      // 128-byte row parts: chunk k ^ (row & 7); 64-byte row parts (two per 128 bytes): k ^ ((row >> 1) & 3)
      auto chunk_at = [&](int row, int k) {
        const int sw = out32 ? (row & 7) : ((row >> 1) & 3);
        return ostage + row * part_bytes + ((k ^ sw) << 4);
      };
      auto stage_out = [&](const float (&vv)[32], float scale) {
        if (out32) {
          #pragma unroll
          for (int q = 0; q < 8; ++q)
            *reinterpret_cast<float4*>(chunk_at(lane, q)) =
                make_float4(vv[4 * q] * scale, vv[4 * q + 1] * scale, vv[4 * q + 2] * scale, vv[4 * q + 3] * scale);
        } else {
          #pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t w4[4];
            #pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float a = vv[8 * q + 2 * k] * scale, c = vv[8 * q + 2 * k + 1] * scale;
              w4[k] = args.out_fmt == kBF16 ? pack_bf16x2(a, c) : pack_f16x2(a, c);
            }
            *reinterpret_cast<uint4*>(chunk_at(lane, q)) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
          }
        }
      };
      auto flush_rows = [&]() {
        __syncwarp();
        const int n0 = qt * kBlockM + wq * 32;  // this warp's first row
        uint8_t* obase =
            reinterpret_cast<uint8_t*>(args.out) + (static_cast<size_t>(bh) * N + n0) * row_bytes + h * part_bytes;
        const int kc = part_bytes / 16;          // chunks per row part (8 or 4)
        const int per = 32 / kc;                 // row parts per warp instruction
        for (int i = 0; i < 32 / per; ++i) {
          const int row = per * i + lane / kc, k = lane % kc;
          if (n0 + row < N)
            *reinterpret_cast<uint4*>(obase + row * row_bytes + (k << 4)) =
                *reinterpret_cast<const uint4*>(chunk_at(row, k));
        }
        __syncwarp();
      };
      if (sg.full(n_kv)) {
        stage_out(v, 1.0f / l);
        flush_rows();
        return true;
      }
      // Cut unit: the schedule cuts a unit at most once, into two pieces that
      // may run in different CTAs; nothing waits on another CTA.
      //  - If the other piece has already published its (O, m, l), this piece
      //    merges with it straight away (no publish, no atomic).
      //  - Otherwise it publishes, then swaps this launch's tag into the
      //    unit's counter; the piece that finds the tag already there arrived
      //    second and merges both published slots.  Whatever an earlier (or
      //    stopped) launch left holds another tag, so the counters never need
      //    clearing.
      // Both merges combine the pieces in the same order (the unit's first
      // piece, then its second) from the same fp32 values, so the result does
      // not depend on which path ran.
      const int c = blockIdx.x;
      const int slot = (sg.tail == 0) ? 2 * c : 2 * c + 1;
      const long long u0 = static_cast<long long>(sg.u) * n_kv;
      const int c_first = sched.cta_of(u0);
      const int sl0 = (sched.begin(c_first) == u0) ? 2 * c_first : 2 * c_first + 1;
      const int sl1 = 2 * (c_first + 1);
      // a slot holds O as [16 chunks][128 rows] float4 (this thread's chunks
      // are 8h .. 8h + 7), then (m, l) per row as [128] float2
      auto slot_of = [&](int s_) { return args.partials + static_cast<size_t>(s_) * kSlotFloats; };
      auto ld_chunk = [&](const float* sl, int q) { return __ldcg(reinterpret_cast<const float4*>(sl) + q * kBlockM + r); };
      auto ld_ml = [&](const float* sl) { return __ldcg(reinterpret_cast<const float2*>(sl + 64 * kBlockM) + r); };
      // out = (fa O_a + fb O_b) / (fa l_a + fb l_b), rescaled to the larger running max
      auto merge_store = [&](const float4 (&xa)[8], float2 ma, const float4 (&xb)[8], float2 mb) {
        const float ms = fmaxf(ma.x, mb.x);
        const float fa = ex2_approx(ma.x - ms), fb = ex2_approx(mb.x - ms);
        const float inv_l = 1.0f / (fa * ma.y + fb * mb.y);
        float vv[32];
        #pragma unroll
        for (int q = 0; q < 8; ++q) {
          vv[4 * q] = fa * xa[q].x + fb * xb[q].x;
          vv[4 * q + 1] = fa * xa[q].y + fb * xb[q].y;
          vv[4 * q + 2] = fa * xa[q].z + fb * xb[q].z;
          vv[4 * q + 3] = fa * xa[q].w + fb * xb[q].w;
        }
        stage_out(vv, inv_l);
        flush_rows();
      };
      unsigned long long* counter = args.counters + static_cast<size_t>(sg.u);
      const float2 mown = make_float2(mstar, l);
      float4 own[8];
      #pragma unroll
      for (int q = 0; q < 8; ++q) own[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
      if (leader) {
        *merge_flag = ld_acquire_gpu(counter) == args.tag;
        mbar_arrive(&bars[kBarMergeGo]);
      }
      if (!warp_all(mbar_wait(&bars[kBarMergeGo], pmerge & 1, abort_flag, status))) return false;
      ++pmerge;
      const bool first = slot == sl0;  // warp-uniform
      if (*merge_flag) {
        const float* po = slot_of(slot == sl0 ? sl1 : sl0);
        float4 xo[8];
        #pragma unroll
        for (int q = 0; q < 8; ++q) xo[q] = ld_chunk(po, 8 * h + q);
        const float2 mo = ld_ml(po);
        if (first) merge_store(own, mown, xo, mo);
        else merge_store(xo, mo, own, mown);
        return true;
      }
      float* ws = slot_of(slot);
      #pragma unroll
      for (int q = 0; q < 8; ++q) __stcg(reinterpret_cast<float4*>(ws) + (8 * h + q) * kBlockM + r, own[q]);
      if (h == 0) __stcg(reinterpret_cast<float2*>(ws + 64 * kBlockM) + r, mown);
      // mbarrier arrive/wait order these writes before the leader's GPU-scope
      // release below (release is cumulative).  Every thread has read
      // merge_flag above before it arrives here, so the leader may reuse it.
      mbar_arrive(&bars[kBarPartWritten]);
      const int pw = ppub++;
      if (leader) {
        const bool w_ok = mbar_wait(&bars[kBarPartWritten], pw & 1, abort_flag, status);
        *merge_flag = w_ok && atomic_exch_acq_rel_gpu(counter, args.tag) == args.tag;
        mbar_arrive(&bars[kBarMergeGo]);
      }
      if (!warp_all(mbar_wait(&bars[kBarMergeGo], pmerge & 1, abort_flag, status))) return false;
      ++pmerge;
      // the leader writes merge_flag again only in a later segment's epilogue,
      // after the prologue barrier that every thread passes once it has read it here
      if (*merge_flag) {
        const float* pa = slot_of(sl0);
        const float* pb = slot_of(sl1);
        float4 xa[8], xb[8];
        #pragma unroll
        for (int q = 0; q < 8; ++q) {
          xa[q] = ld_chunk(pa, 8 * h + q);
          xb[q] = ld_chunk(pb, 8 * h + q);
        }
        merge_store(xa, ld_ml(pa), xb, ld_ml(pb));
      }
      return true;
    };

    Cursor cur(sched, blockIdx.x);
    Segment sg;
    while (ok && cur.next(sched, sg)) ok = run_seg(sg, false);
    // every softmax thread has finished its segments; tell the other roles
    // whether one must run again
    mbar_arrive(&bars[kBarDecision]);
    if (replay_decision(ok, sg)) run_seg(sg, true);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

}  // namespace dera
