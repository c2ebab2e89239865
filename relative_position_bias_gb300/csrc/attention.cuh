// Global self-attention with decomposed relative-position bias on tcgen05.
//
// Computes, for every (batch*head) b and token n = qh*W + qw,
//   out[b, n] = sum_m softmax_m(scale * q_n.k_m + rel_h[n, kh(m)] + rel_w[n, kw(m)]) v_m
// without materialising the HW x HW bias (vLLM PR #55629 page, sections
// 实现拆解 item 1 and 关键源码片段).  The softmax is online, in base 2, with
// fp32 statistics (section 风险与影响).
//
// Work unit: a pair of 128-row query tiles of one head; both tiles share every
// K/V tile the CTA streams.  The kernel is persistent: CTA c runs the
// contiguous range [c*T/G, (c+1)*T/G) of the T = units x key-tiles iteration
// space (stream-K), so all CTAs get the same number of key tiles whatever the
// unit count.  A unit cut between two CTAs: the piece that finishes first
// publishes its partial results (unnormalised O, row max, row sum) to the
// caller's workspace; the piece that finishes second merges them with its own
// O straight from TMEM (or, if both had to publish, from both slots).  With
// one CTA per unit (no workspace) every segment is a whole unit and nothing
// is written to the workspace.
//
// Warp roles (384 threads; warps 0-3 run with 104 registers, the softmax
// warpgroups with 200, set by setmaxnreg):
//   warp 0      TMA producer: Q pair, [tables,] K/V ring (2 to 4 stages)
//   warp 1      tcgen05.mma issuer (the warp walks the loop, an elected lane issues)
//   warp 2      TMEM allocator; with warp 3, converts bf16 V tiles to fp16
//   warps 4-7   softmax / epilogue of query tile 0 (one thread per row)
//   warps 8-11  softmax / epilogue of query tile 1
// TMEM (512 columns), head_dim 64: S0 [0,128) S1 [128,256) P0 [256,320)
//   P1 [320,384) O0 [384,448) O1 [448,512); head_dim 128 (key tiles of at most
//   80 keys): S_i [128i, 128i+80) P_i [128i+88, 128i+128) O_i [256+128i, 384+128i).
//   The fused prologue uses all 512 columns for G_i = Q_i [T_h ; T_w]^T before
//   each segment.
#pragma once
#include <cfloat>

#include "common.cuh"

namespace dera {

constexpr int kMaxStages = 4;     // deepest K/V ring (head_dim 64)
constexpr int kTilesPerUnit = 2;  // 128-row query tiles per work unit
constexpr int kAttnThreads = 384;
// Largest accepted row sum of a speculative tile: with the sum at most this,
// every p rounds to at most 65504, the largest finite fp16.
constexpr float kSpecSumLimit = 65000.0f;
// Starting row maximum of a segment (base 2): kStartMargin below a rel_h-aware
// estimate, at most kStartCap above the exact maximum of its first key tile.
// A starting maximum that overshoots the row's true maximum leaves the row sum
// small, which the row check at the end of the segment catches (see the
// epilogue); the cap only bounds how often that happens.  24 measured best:
// 12, 16, 20 and 24 gave 786, 799, 824 and 838 TFLOP/s on the 64x64 grid with
// head_dim 128, and 16 and above the same on head_dim 64.
constexpr float kStartCap = 24.0f;
constexpr float kStartMargin = 4.0f;
// Cap used once a row of the CTA has failed the row check: with the starting
// maximum at most 3 above the first tile's exact maximum, l >= 2^-3, which
// passes the check for every segment (n <= 4096 keys), so no later segment
// of the CTA needs a replay.  Inputs whose row maximum moves far between key
// tiles (wide logit ranges) fail early and then run with this cap.
constexpr float kSafeCap = 3.0f;
// A key tile is taken exact at once, without the speculative pass, when on
// some row of the warp the tile's largest rel_h term plus the rel_h-free
// maximum of the row's last exact tile passes the running maximum by more
// than this (base 2): such a tile would almost surely pass kSpecSumLimit and
// be exponentiated twice.  rel_h is known exactly for every key tile, so this
// catches most redos of inputs whose rel_h spreads widely over the grid rows
// (40x40 with fp16 inputs: 365 -> 307 us) and never fires on the 64x64 inputs.
constexpr float kPredictMargin = 14.0f;
// A warp in which at least kWideRows rows start with a rel_h-based estimate
// more than kWideGap (base 2) above their first tile's exact maximum holds
// rows whose rel_h spreads over most of the 40 binades of fp16 P; at
// kStartCap such rows mostly fail the row check (and the segment is run
// again), so the warp starts the segment at kSafeCap instead.  On the 40x40
// fp16 inputs every warp qualifies (307 -> 287 us, the first segment of each
// CTA no longer replayed); on the 64x64 inputs, head_dim 64 or 128, none does.
constexpr float kWideGap = 32.0f;
constexpr int kWideRows = 4;
// Row-sum check at the end of a segment: the row sum l, in units of the
// running maximum, must be at least the segment's valid key count times
// 2^kMinRowSumLog2 (see the epilogue).
constexpr int kMinRowSumLog2 = -16;
// Register split: the producer / MMA / V-conversion warpgroup gives registers
// back and the two softmax warpgroups take them, which removes the softmax's
// spills.  The block launches with kLaunchRegs per thread (the most that 384
// threads get); the host checks the compiled count before the first launch,
// since a split larger than the launch pool would block forever.
constexpr int kLaunchRegs = 168;
constexpr int kRegsCtl = 104;
constexpr int kRegsSmx = 200;
static_assert(kRegsCtl * 128 + kRegsSmx * 256 <= kLaunchRegs * kAttnThreads, "register split exceeds the launch pool");
static_assert(kRegsCtl % 8 == 0 && kRegsSmx % 8 == 0, "setmaxnreg counts are multiples of 8");

// Shapes that depend on the head dimension D (64 or 128) and the key-tile
// width BN.
template <int D, int BN>
struct AttnDims {
  static constexpr int kAtoms = atoms_of<D>();
  static constexpr int kQTile = kBlockM * 2 * D;                 // one 128-row query tile
  // K (and V) region of a ring stage: BN rows of 2D bytes (at most 128 x 128 B
  // for head_dim 64; 64 or 80 x 256 B for head_dim 128)
  static constexpr int kKVBytes = D == 64 ? kTileBytes : BN * 2 * D;
  static constexpr int kStageBytes = 2 * kKVBytes;
  // K/V ring depth, as deep as shared memory allows beside the query tiles and
  // the bias areas: 4 stages for head_dim 64, 3 for head_dim 128 with 64-key
  // tiles, 2 with 80-key tiles
  static constexpr int kStages = D == 64 ? 4 : (kStageBytes <= 32 * 1024 ? 3 : 2);
  // floats per row of a bias staging area (an odd stride: a warp's staged
  // rows start in different banks)
  static constexpr int kBiasStride = 65;
  // ring stages the fused prologue's tables take: [T_h | T_w] in one stage,
  // or T_h and T_w (32 KB each) in one stage apiece
  static constexpr int kTableSlots = D == 64 ? 1 : 2;
  // TMEM columns of query tile i
  static constexpr uint32_t tmS(int i) { return 128u * i; }
  static constexpr uint32_t tmP(int i) { return D == 64 ? 256u + 64u * i : 128u * i + 88u; }
  static constexpr uint32_t tmO(int i) { return D == 64 ? 384u + 64u * i : 256u + 128u * i; }
  static_assert(kMaxStages >= kStages, "barrier slots");
};

template <int D, int BN>
struct AttnSmem {
  using Dm = AttnDims<D, BN>;
  static constexpr int kQ = 0;                                   // 2 query tiles
  static constexpr int kRing = 2 * Dm::kQTile;                   // stages: [K][V]
  static constexpr int kBias = kRing + Dm::kStages * Dm::kStageBytes;  // 2 bias areas of 128 rows
  static constexpr int kBiasBytes = 2 * kBlockM * Dm::kBiasStride * 4;
  static constexpr int kBars = kBias + kBiasBytes;
  static constexpr int kNumBars = 32;
  static constexpr int kMisc = kBars + kNumBars * 8;             // tmem slot, flags, replay records
  static constexpr int kTotal = kMisc + 96;
  static constexpr int kAlloc = kTotal + 1024;                   // slack for 1 KB alignment
  static_assert(kAlloc <= 232448, "shared memory budget");
};

// barrier indices
enum : int {
  kBarQFull = 0,
  kBarQEmpty = 1,
  kBarKVFull = 2,                     // + stage
  kBarKVEmpty = kBarKVFull + kMaxStages,
  kBarVReady = kBarKVEmpty + kMaxStages,
  kBarSFull = kBarVReady + kMaxStages,   // + tile
  kBarPFull = kBarSFull + 2,
  kBarODone = kBarPFull + 2,
  kBarGFull = kBarODone + 2,
  kBarGFree = kBarGFull + 1,
  kBarEpiDone = kBarGFree + 1,
  kBarStg = kBarEpiDone + 1,          // + tile
  kBarPartWritten = kBarStg + 2,     // + tile
  kBarMergeGo = kBarPartWritten + 2,  // + tile
  kBarDecision = kBarMergeGo + 2,
  kBarMmaDone = kBarDecision + 1,
  kBarCount = kBarMmaDone + 1
};
static_assert(kBarCount <= AttnSmem<64, 128>::kNumBars, "barrier slots");

// Work schedule over G persistent CTAs: all but the last one-and-a-fraction
// waves of units run as data-parallel rounds (CTA c takes unit r*G + c in
// round r, so the CTAs active together work on consecutive units, i.e. on the
// same heads, and share those heads' K/V in L2); the remaining G + (U mod G)
// units form a stream-K tail whose (unit, key tile) iterations are cut into G
// equal contiguous ranges.  Every tail range holds at least one unit's worth
// of key tiles, so a unit is cut into at most two segments.  With U a
// multiple of G the tail is one whole unit per CTA and nothing is cut.
// Iterations are numbered globally: t = unit * n_kv + key tile.
//
// The tail ranges are equal in cost rather than in key tiles: each segment
// a CTA starts costs about kSegCost key tiles (prologue, epilogue, pipeline
// refill), so the tail is cut evenly in a virtual space where every unit is
// kSegCost slots of "segment start" followed by its n_kv key tiles.  A range
// then holds fewer key tiles the more unit starts it contains.  Each range
// still spans at least n_kv + kSegCost virtual slots, so no unit is cut into
// more than two segments.
//
// Without cuts (no workspace, or units too short to be worth cutting) the G
// CTAs take whole units round-robin: CTA c runs units c, c + G, c + 2G, ...
// (the last round may hold fewer units than CTAs), so a CTA's later units are
// loaded while it computes the earlier ones.
struct Schedule {
  static constexpr int kSegCost = 8;
  int G, n_kv, dp_rounds, U;
  long long sk_base, V;  // first tail iteration; tail length in virtual slots (0: no tail)
  __device__ __forceinline__ Schedule(int U_, int G_, int n_kv_, bool cut) : G(G_), n_kv(n_kv_), U(U_) {
    if (cut) {
      dp_rounds = max(U / G - 1, 0);
      sk_base = static_cast<long long>(dp_rounds) * G * n_kv;
      V = static_cast<long long>(U - dp_rounds * G) * (n_kv + kSegCost);
    } else {
      dp_rounds = (U + G - 1) / G;
      sk_base = static_cast<long long>(U) * n_kv;
      V = 0;
    }
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
  // CTA whose tail range holds iteration t (t >= sk_base; only with cuts)
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
      if (sg.u < s.U) return true;
      round = s.dp_rounds;  // a last round with fewer units than CTAs
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


__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
  const float lo = __uint_as_float(w << 16);
  const float hi = __uint_as_float(w & 0xFFFF0000u);
  return pack_f16x2(lo, hi);
}

// A segment whose row-sum check failed for one query tile (see the epilogue):
// the CTA runs it again after its other work, storing only that tile.
struct ReplayRecord {
  int pending;
  Segment sg;
};

// Key tiles of the forward: KeyTile's grid rows, except that a grid padded to
// 40 columns (head_dim 64) takes three grid rows, 120 keys, into S and PV
// products 128 keys wide.  Its last 8 columns are padding: their P is 0 and
// their K and V rows are never loaded (V's are kept finite, see the kernel's
// set-up).  Fewer, fuller key tiles than two grid rows of 80 keys.
template <int WP, int D>
struct FwdKeyTile {
  static constexpr int KHT = (D == 64 && WP == 40) ? 3 : KeyTile<WP, D>::KHT;
  static constexpr int BN = KHT * WP;               // keys loaded per tile
  static constexpr int BNP = (BN + 15) / 16 * 16;   // width of the S and PV products
  static_assert(BNP <= 128 && (BNP == BN || D == 64), "padded key tiles need head_dim 64");
};

template <int WP, bool FUSED, bool BF16, int D>
__global__ void __launch_bounds__(kAttnThreads, 1)
    relpos_attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_th,
                       const __grid_constant__ CUtensorMap tm_tw, const AttnArgs args) {
  using KT = FwdKeyTile<WP, D>;
  using Dm = AttnDims<D, KT::BN>;
  using SM = AttnSmem<D, KT::BN>;
  constexpr int kBiasStride = Dm::kBiasStride;
  constexpr int KHT = KT::KHT;
  constexpr int BN = KT::BN;     // keys of a tile
  constexpr int BNP = KT::BNP;   // columns of its S and PV products (BN, or BN padded to 16)
  constexpr int KS = Dm::kStages;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw_u + 1023u) & ~1023u) - raw_u);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + SM::kBars);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + SM::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + SM::kMisc + 4);
  volatile int* merge_flag = reinterpret_cast<volatile int*>(smem + SM::kMisc + 8);  // [2]
  volatile int* bad_flag = reinterpret_cast<volatile int*>(smem + SM::kMisc + 16);   // [2 tiles][2 parities]
  ReplayRecord* replay = reinterpret_cast<ReplayRecord*>(smem + SM::kMisc + 32);     // [2 tiles]
  volatile int* cap_drop = reinterpret_cast<volatile int*>(smem + SM::kMisc + 80);   // a row check failed
  int* status = args.status;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_kv = args.n_kv;
  const Schedule sched(args.n_units, static_cast<int>(gridDim.x), n_kv, args.counters != nullptr);
  constexpr bool convert_v = BF16;  // P is fp16, so bf16 V tiles are converted to fp16 on chip

  auto sQ = [&](int i) { return smem + SM::kQ + i * Dm::kQTile; };
  auto sK = [&](int s) { return smem + SM::kRing + s * Dm::kStageBytes; };
  auto sV = [&](int s) { return smem + SM::kRing + s * Dm::kStageBytes + Dm::kKVBytes; };

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    merge_flag[0] = 0;
    merge_flag[1] = 0;
    for (int i = 0; i < 4; ++i) bad_flag[i] = 0;
    *cap_drop = 0;
    replay[0].pending = 0;
    replay[1].pending = 0;
    mbar_init(&bars[kBarQFull], 1);
    mbar_init(&bars[kBarQEmpty], 1);
    for (int s = 0; s < KS; ++s) {
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
    mbar_init(&bars[kBarEpiDone], 2 * kBlockM);
    mbar_init(&bars[kBarStg + 0], kBlockM);
    mbar_init(&bars[kBarStg + 1], kBlockM);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars[kBarPartWritten + i], kBlockM);
      mbar_init(&bars[kBarMergeGo + i], 1);
    }
    mbar_init(&bars[kBarDecision], 2 * kBlockM);
    mbar_init(&bars[kBarMmaDone], 1);
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  if constexpr (BNP > BN) {
    // Rows BN..BNP-1 of every K and V stage are read by the products but never
    // loaded by TMA (the fused prologue's tables, whose rows there are past the
    // tables' ends for these widths, load zeros).  Their P is 0, and 0 times a
    // finite V is 0, so V (and K, for tidiness) start as zeros.
    constexpr int kPadChunks = (BNP - BN) * 128 / 16;   // 16-byte chunks per region (head_dim 64)
    for (int i = threadIdx.x; i < KS * 2 * kPadChunks; i += kAttnThreads) {
      const int s = i / (2 * kPadChunks), c = i - s * (2 * kPadChunks);
      uint8_t* region = c < kPadChunks ? sK(s) : sV(s);
      *reinterpret_cast<uint4*>(region + BN * 128 + 16 * (c % kPadChunks)) = make_uint4(0u, 0u, 0u, 0u);
    }
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tmem_slot;

  // After the softmax warps have finished their segments (bounded wait), the
  // k-th segment to run again, if any: a failed segment of query tile k, run
  // once for both tiles when both failed in the same segment.  `mask` holds
  // the tiles whose result that run stores.
  auto replay_decision = [&](bool ok, int k, Segment& sg, int& mask) -> bool {
    if (!mbar_wait(&bars[kBarDecision], 0, abort_flag, status) || !ok) return false;
    if (!replay[k].pending) return false;
    const Segment a = replay[k].sg;
    const bool same = replay[0].pending && replay[1].pending && replay[0].sg.u == replay[1].sg.u &&
                      replay[0].sg.j0 == replay[1].sg.j0 && replay[0].sg.j1 == replay[1].sg.j1;
    if (k == 1 && same) return false;   // already run for both tiles
    sg = a;
    mask = same ? 3 : (1 << k);
    return true;
  };
  // The segments of a role, in order: the CTA's own (mask -1), then those to
  // run again.  Every role walks the same list through this one function, so
  // each role's segment body has a single call site.  The softmax warps
  // arrive on the decision barrier when their own segments are done.
  auto next_segment = [&](Cursor& cur, int& phase, bool ok, bool softmax, Segment& sg, int& mask) -> bool {
    if (phase == 0) {
      if (ok && cur.next(sched, sg)) {
        mask = -1;
        return true;
      }
      phase = 1;
      if (softmax) mbar_arrive(&bars[kBarDecision]);
    }
    while (phase <= 2) {
      const int k = phase - 1;
      ++phase;
      if (replay_decision(ok, k, sg, mask)) return true;
    }
    return false;
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
      auto run_seg = [&](const Segment& sg) -> bool {
        const int bh = sg.u / args.n_pairs;
        const int qt0 = 2 * (sg.u - bh * args.n_pairs);
        if (seg > 0 && !mbar_wait(&bars[kBarQEmpty], (seg - 1) & 1, abort_flag, status)) return false;
        mbar_arrive_expect_tx(&bars[kBarQFull], 2 * Dm::kQTile);
        #pragma unroll
        for (int i = 0; i < 2; ++i)
          #pragma unroll
          for (int a = 0; a < Dm::kAtoms; ++a)
            tma_load_3d(sQ(i) + a * kTileBytes, &tm_q, &bars[kBarQFull], 64 * a, (qt0 + i) * kBlockM, bh);
        ++seg;
        if (FUSED) {
          for (int t = 0; t < Dm::kTableSlots; ++t, ++rg) {
            const int s = rg % KS;
            if (!mbar_wait(&bars[kBarKVEmpty + s], ((rg / KS) & 1) ^ 1, abort_flag, status)) return false;
            mbar_arrive_expect_tx(&bars[kBarKVFull + s], 2 * kTileBytes);
            if (D == 64) {
              tma_load_2d(sK(s), &tm_th, &bars[kBarKVFull + s], 0, 0);
              tma_load_2d(sV(s), &tm_tw, &bars[kBarKVFull + s], 0, 0);
            } else {
              // one table per stage, its two atoms back to back
              #pragma unroll
              for (int a = 0; a < Dm::kAtoms; ++a)
                tma_load_2d(sK(s) + a * kTileBytes, t == 0 ? &tm_th : &tm_tw, &bars[kBarKVFull + s], 64 * a, 0);
            }
          }
        }
        for (int j = sg.j0; j < sg.j1; ++j, ++rg) {
          const int s = rg % KS;
          if (!mbar_wait(&bars[kBarKVEmpty + s], ((rg / KS) & 1) ^ 1, abort_flag, status)) return false;
          mbar_arrive_expect_tx(&bars[kBarKVFull + s], 2 * BN * 2 * D);
          #pragma unroll
          for (int a = 0; a < Dm::kAtoms; ++a) {
            tma_load_4d(sK(s) + a * BN * 128, &tm_k, &bars[kBarKVFull + s], 64 * a, 0, j * KHT, bh);
            tma_load_4d(sV(s) + a * BN * 128, &tm_v, &bars[kBarKVFull + s], 64 * a, 0, j * KHT, bh);
          }
        }
        return true;
      };
      Cursor cur(sched, blockIdx.x);
      Segment sg;
      int phase = 0, mask;
      while (next_segment(cur, phase, ok, false, sg, mask)) ok = run_seg(sg) && ok;
      if (!ok) {
        // Let the copies already in flight land before the CTA exits.
        if (seg > 0) mbar_wait_budget(&bars[kBarQFull], (seg - 1) & 1, kWaitBudgetCycles);
        for (int r = max(0, rg - KS); r < rg; ++r)
          mbar_wait_budget(&bars[kBarKVFull + r % KS], (r / KS) & 1, kWaitBudgetCycles);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp walks the loop (waits and operand arithmetic are
    // warp-uniform); one elected lane issues each tcgen05 instruction.
    {
      constexpr uint32_t fmt = BF16 ? kBF16 : kF16;
      constexpr uint32_t id_qk = idesc_f16(kBlockM, BNP, fmt, fmt, 0, 0);
      // PV in 64-column halves of O (one V atom each)
      constexpr uint32_t id_pv = idesc_f16(kBlockM, 64, kF16, kF16, 0, 1);
      // G: [T_h ; T_w] as one N = 256 product (head_dim 64), or T_h and T_w
      // as two N = 128 products from their own stages (head_dim 128)
      constexpr uint32_t id_g = idesc_f16(kBlockM, D == 64 ? 256 : 128, fmt, fmt, 0, 0);
      // Descriptors differ only in their 14-bit start-address field (address / 16),
      // which stays below 2^14 for any shared-memory address, so offsets are
      // added to one base descriptor per operand.
      const uint64_t d_q = sdesc_sw128(smem_u32(sQ(0)), 16, 1024);
      const uint64_t d_k = sdesc_sw128(smem_u32(sK(0)), 16, 1024);
      const uint64_t d_v = sdesc_sw128(smem_u32(sV(0)), 16, 1024);
      constexpr uint32_t kQStep = Dm::kQTile >> 4, kStageStep = Dm::kStageBytes >> 4;
      // atom strides: 128 rows of a query tile or table, BN rows of a K/V tile
      constexpr uint32_t kQAtom = kTileBytes >> 4, kKVAtom = (BN * 128) >> 4;
      // K-step k (16 elements) of a K-major operand: atom k / 4, 32 bytes per step inside it
      auto kstep = [](int k, uint32_t atom) { return static_cast<uint32_t>(k / 4) * atom + 2u * (k % 4); };
      auto issue_qk = [&](int i, int s) {
        const uint64_t a = d_q + i * kQStep, b = d_k + s * kStageStep;
        #pragma unroll
        for (int k = 0; k < D / 16; ++k)
          umma_ss_w(tbase + Dm::tmS(i), a + kstep(k, kQAtom), b + kstep(k, kKVAtom), id_qk, k > 0);
      };
      auto issue_pv = [&](int i, int s, bool acc) {
        #pragma unroll
        for (int h = 0; h < Dm::kAtoms; ++h) {
          const uint64_t b = d_v + s * kStageStep + h * kKVAtom;
          #pragma unroll
          for (int k = 0; k < BNP / 16; ++k)
            umma_ts_w(tbase + Dm::tmO(i) + 64 * h, tbase + Dm::tmP(i) + 8 * k, b + 128 * k, id_pv,
                      (acc || k > 0) ? 1u : 0u);
        }
      };
      int rg = 0, gi = 0, seg = 0;
      bool ok = true;
      auto run_seg = [&](const Segment& sg) -> bool {
        const int len = sg.j1 - sg.j0;
        if (!warp_all(mbar_wait(&bars[kBarQFull], seg & 1, abort_flag, status))) return false;
        if (FUSED) {
          if (seg > 0 && !warp_all(mbar_wait(&bars[kBarEpiDone], (seg - 1) & 1, abort_flag, status))) return false;
          for (int t = 0; t < Dm::kTableSlots; ++t) {
            const int s = (rg + t) % KS;
            if (!warp_all(mbar_wait(&bars[kBarKVFull + s], ((rg + t) / KS) & 1, abort_flag, status))) return false;
          }
          tc_fence_after();
          for (int i = 0; i < 2; ++i) {
            const uint64_t a = d_q + i * kQStep;
            #pragma unroll
            for (int t = 0; t < Dm::kTableSlots; ++t) {
              const uint64_t b = d_k + ((rg + t) % KS) * kStageStep;
              #pragma unroll
              for (int k = 0; k < D / 16; ++k)
                umma_ss_w(tbase + 256 * i + 128 * t, a + kstep(k, kQAtom), b + kstep(k, kQAtom), id_g, k > 0);
            }
          }
          umma_commit_w(&bars[kBarGFull]);
          for (int t = 0; t < Dm::kTableSlots; ++t, ++rg) umma_commit_w(&bars[kBarKVEmpty + rg % KS]);
          if (!warp_all(mbar_wait(&bars[kBarGFree], seg & 1, abort_flag, status))) return false;
          tc_fence_after();
        }
        ++seg;
        {
          const int s = rg % KS;
          if (!warp_all(mbar_wait(&bars[kBarKVFull + s], (rg / KS) & 1, abort_flag, status))) return false;
          tc_fence_after();
          issue_qk(0, s);
          umma_commit_w(&bars[kBarSFull + 0]);
          issue_qk(1, s);
          umma_commit_w(&bars[kBarSFull + 1]);
        }
        for (int jj = 0; jj < len; ++jj, ++rg, ++gi) {
          const int s = rg % KS, ph = (rg / KS) & 1;
          const int sn = (rg + 1) % KS, phn = ((rg + 1) / KS) & 1;
          const bool more = jj + 1 < len;
          if (convert_v && !warp_all(mbar_wait(&bars[kBarVReady + s], ph, abort_flag, status))) return false;
          // Once softmax i has written P_i(j) (and so finished reading S_i),
          // the next S_i goes first: the softmax can start on it while PV_i(j)
          // runs, and waits for PV_i(j) only before it next writes P_i or O_i.
          if (!warp_all(mbar_wait(&bars[kBarPFull + 0], gi & 1, abort_flag, status))) return false;
          tc_fence_after();
          if (more) {
            if (!warp_all(mbar_wait(&bars[kBarKVFull + sn], phn, abort_flag, status))) return false;
            tc_fence_after();
            issue_qk(0, sn);
            umma_commit_w(&bars[kBarSFull + 0]);
          }
          issue_pv(0, s, jj > 0);
          umma_commit_w(&bars[kBarODone + 0]);
          if (!warp_all(mbar_wait(&bars[kBarPFull + 1], gi & 1, abort_flag, status))) return false;
          tc_fence_after();
          if (more) {
            issue_qk(1, sn);
            umma_commit_w(&bars[kBarSFull + 1]);
          } else {
            umma_commit_w(&bars[kBarQEmpty]);  // no more reads of this segment's Q
          }
          issue_pv(1, s, jj > 0);
          umma_commit_w(&bars[kBarODone + 1]);
          umma_commit_w(&bars[kBarKVEmpty + s]);
        }
        return true;
      };
      Cursor cur(sched, blockIdx.x);
      Segment sg;
      int phase = 0, mask;
      while (next_segment(cur, phase, warp_all(ok), false, sg, mask)) ok = run_seg(sg) && ok;
      // Drain: every MMA issued above completes before TMEM is released.
      umma_commit_w(&bars[kBarMmaDone]);
      mbar_wait_budget(&bars[kBarMmaDone], 0, kWaitBudgetCycles);
      __syncwarp();
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------ bf16 -> fp16 V conversion
    // The fused kernel's table slots are passed through unconverted, so that
    // v_ready completes once per ring index.
    if (convert_v) {
      const int ct = threadIdx.x - 64;
      int rg = 0;
      bool ok = true;
      auto run_seg = [&](const Segment& sg) -> bool {
        for (int j = FUSED ? sg.j0 - Dm::kTableSlots : sg.j0; j < sg.j1; ++j, ++rg) {
          const int s = rg % KS;
          if (!mbar_wait(&bars[kBarKVFull + s], (rg / KS) & 1, abort_flag, status)) return false;
          if (j >= sg.j0) {
            uint4* vp = reinterpret_cast<uint4*>(sV(s));
            for (int idx = ct; idx < BN * 2 * D / 16; idx += 64) {
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
      int phase = 0, mask;
      while (next_segment(cur, phase, ok, false, sg, mask)) ok = run_seg(sg) && ok;
    }
  }
  } else {
    regs_claim<kRegsSmx>();
    // ------------------------------------------------------------ softmax / epilogue
    const int wg = (warp - 4) >> 2;          // query tile of this warpgroup
    const int wq = warp & 3;                 // TMEM lane quarter
    const int r = wq * 32 + lane;            // row inside the tile
    const int H = args.H, W = args.W, N = args.N;
    const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tbase + lane_off + Dm::tmS(wg);
    const uint32_t tP = tbase + lane_off + Dm::tmP(wg);
    const uint32_t tO = tbase + lane_off + Dm::tmO(wg);
    float* area = reinterpret_cast<float*>(smem + SM::kBias) + wg * kBlockM * kBiasStride;
    // A thread's rel_h row is its staging row.  Where n_kv KHT grid rows always
    // fit in it, those past H hold -inf; with three grid rows per tile (up to
    // 66 > kBiasStride) the row holds the H grid rows only and a tile's grid
    // rows past H read as -inf.
    constexpr bool kPadRows = (64 + KHT - 1) / KHT * KHT < kBiasStride;
    const int Hpad = n_kv * KHT;
    const int HS = kBiasStride;
    float* bh_row = area + r * HS;
    const float NEG_INF = -__int_as_float(0x7f800000);
    const float sl2 = args.scale_log2;
    const float2 sl2v = make_float2(sl2, sl2);

    int gi = 0, seg = 0;
    // overshoot allowed to the starting maximum: kStartCap until a row check
    // of the CTA fails, kSafeCap after it (and in a segment where the warp's
    // rows are wide, see kWideRows), 0 in replays
    float cap = kStartCap;
    bool own_failed = false;  // this warpgroup has failed a row check (uniform over it)
    int pseg = 0;  // completed phases of this warpgroup's merge-go barrier
    int ppub = 0;  // completed phases of its partial-written barrier
    uint32_t stg_phase = 0;  // completed phases of this warpgroup's staging barrier
    // Warpgroup-wide barrier on the staging mbarrier (all 128 threads arrive, then wait).
    auto wg_sync = [&]() -> bool {
      mbar_arrive(&bars[kBarStg + wg]);
      const bool w = mbar_wait(&bars[kBarStg + wg], stg_phase & 1, abort_flag, status);
      ++stg_phase;
      return warp_all(w);
    };
    bool ok = true;
    auto run_seg = [&](const Segment& sg, int store_mask) -> bool {
      // the other warpgroup's flag may be seen late; either value is safe
      cap = store_mask >= 0 ? 0.f : ((own_failed || *cap_drop) ? kSafeCap : kStartCap);
      const int bh = sg.u / args.n_pairs;
      const int qt = 2 * (sg.u - bh * args.n_pairs) + wg;
      const int n = qt * kBlockM + r;
      const bool row_valid = n < N;
      const int qh = row_valid ? n / W : 0;
      const int qw = row_valid ? n - qh * W : 0;

      float bw[WP];
      if (FUSED) {
        ok = warp_all(mbar_wait(&bars[kBarGFull], seg & 1, abort_flag, status));
        tc_fence_after();
        float* stg = area + r * kBiasStride;
        if (ok) skew_row_to_smem(tbase + lane_off + 256 * wg + 128, qw, W, stg, kLog2e);
        #pragma unroll
        for (int kw = 0; kw < WP; ++kw) bw[kw] = (ok && kw < W) ? stg[kw] : NEG_INF;
        // the staging row and the bias row of a thread are the same row (stride
        // kBiasStride both), read and written by that thread alone
        if (ok) {
          skew_row_to_smem(tbase + lane_off + 256 * wg, qh, H, bh_row, kLog2e);
          if (kPadRows)
            for (int kh = H; kh < Hpad; ++kh) bh_row[kh] = NEG_INF;
        }
        tc_fence_before();
        mbar_arrive(&bars[kBarGFree]);
        if (!ok) return false;
      } else {
        // every warp has stored the previous segment's output rows, which
        // leave through the same area, before any row is copied in
        if (seg > 0) ok = wg_sync() && ok;
        // The tile's rows of rel_w, then of rel_h, are one contiguous block
        // each: every warp copies a quarter of the rows into the staging area,
        // a row per pass with the lanes along it (coalesced), scaled by log2e.
        // Rows past N read as 0.
        const size_t row0 = static_cast<size_t>(bh) * N + static_cast<size_t>(qt) * kBlockM;
        const int nrows = min(kBlockM, N - qt * kBlockM);
        // Loads for 8 rows go out together before any store (the stores could
        // alias the source as far as the compiler knows).
        auto copy_rows = [&](const void* src, int len, int stride) {
          for (int rb = wq; rb < kBlockM; rb += 32) {
            float v[8][2];
            #pragma unroll
            for (int u = 0; u < 8; ++u) {
              const int rr = rb + 4 * u;
              #pragma unroll
              for (int h = 0; h < 2; ++h) {
                const int c = lane + 32 * h;
                v[u][h] = (rr < nrows && c < len)
                              ? load_elem(src, (row0 + rr) * static_cast<size_t>(len) + c, args.bias_fmt)
                              : 0.f;
              }
            }
            #pragma unroll
            for (int u = 0; u < 8; ++u) {
              #pragma unroll
              for (int h = 0; h < 2; ++h) {
                const int c = lane + 32 * h;
                if (c < len) area[(rb + 4 * u) * stride + c] = kLog2e * v[u][h];
              }
            }
          }
        };
        // An fp32 bias is copied as it is with cp.async: every element of
        // the tile's rows goes out at once (element e of the block to thread
        // e mod 128, so a warp reads 128 contiguous bytes), without a round
        // trip through registers per batch of rows; the log2e scaling is
        // applied where the rows are read.  Rows past N are written as 0.
        const bool raw = args.bias_fmt == kF32;
        auto copy_rows_async = [&](const float* src, int len, int stride) {
          const int step_r = kBlockM / len, step_c = kBlockM - step_r * len;
          int rr = r / len, c = r - rr * len;
          for (int e = r; e < kBlockM * len; e += kBlockM) {
            cp_async4(area + rr * stride + c, src + (row0 + (rr < nrows ? rr : 0)) * static_cast<size_t>(len) + c,
                      rr < nrows ? 4u : 0u);
            rr += step_r;
            c += step_c;
            if (c >= len) {
              c -= len;
              ++rr;
            }
          }
          cp_async_wait_all();
        };
        if (raw) copy_rows_async(static_cast<const float*>(args.rel_w), W, kBiasStride);
        else copy_rows(args.rel_w, W, kBiasStride);
        ok = wg_sync() && ok;
        const float* stg = area + r * kBiasStride;
        const float wscale = raw ? kLog2e : 1.0f;
        #pragma unroll
        for (int kw = 0; kw < WP; ++kw) bw[kw] = kw < W ? wscale * stg[kw] : NEG_INF;
        // every thread has its rel_w row before the area is reused for rel_h
        ok = wg_sync() && ok;
        if (raw) copy_rows_async(static_cast<const float*>(args.rel_h), H, HS);
        else copy_rows(args.rel_h, H, HS);
        ok = wg_sync() && ok;
        if (raw)
          for (int kh = 0; kh < H; ++kh) bh_row[kh] *= kLog2e;   // this thread's own row
        if (kPadRows)
          for (int kh = H; kh < Hpad; ++kh) bh_row[kh] = NEG_INF;
        if (!ok) return false;
      }
      ++seg;

      // S is processed in blocks of kBlk columns (one TMEM load and one wait
      // each); narrow grids, with more grid rows per tile, use 16 to keep
      // their per-row bias terms in registers.
      constexpr int kBlk = (WP <= 16 || BNP != BN) ? 16 : 32;
      auto load_block = [&](int cb, uint32_t (&u)[kBlk]) {
        if (kBlk == 32 && BNP - cb >= 32) tmem_ld32(tS + cb, *reinterpret_cast<uint32_t(*)[32]>(&u[0]));
        else tmem_ld16(tS + cb, *reinterpret_cast<uint32_t(*)[16]>(&u[0]));
        tmem_wait_ld();
      };
      // Exact tile maximum of x = s*scale*log2e + rel_w*log2e + rel_h*log2e;
      // base = the same without the rel_h term.
      auto tile_max = [&](const float (&bhv)[KHT], float& base) -> float {
        float gm[KHT];
        #pragma unroll
        for (int g = 0; g < KHT; ++g) gm[g] = NEG_INF;
        #pragma unroll
        for (int cb = 0; cb < BN; cb += kBlk) {
          uint32_t u[kBlk];
          load_block(cb, u);
          #pragma unroll
          for (int k = 0; k < kBlk; k += 2) {
            const int col = cb + k;
            if (col < BN) {
              const int g = col / WP, kw = col % WP;
              const float2 t = ffma2(make_float2(__uint_as_float(u[k]), __uint_as_float(u[k + 1])), sl2v,
                                     make_float2(bw[kw], bw[kw + 1]));
              gm[g] = fmax3(gm[g], t.x, t.y);
            }
          }
        }
        float mt = NEG_INF;
        base = NEG_INF;
        #pragma unroll
        for (int g = 0; g < KHT; ++g) {
          mt = fmaxf(mt, gm[g] + bhv[g]);
          base = fmaxf(base, gm[g]);
        }
        return mt;
      };
      // Waits (once, warp-uniformly) until PV of the previous key tile has
      // read P and written O; needed before P or O is next written.
      bool pv_pending = false;
      auto wait_pv = [&]() {
        if (pv_pending) {
          ok = warp_all(mbar_wait(&bars[kBarODone + wg], (gi - 1) & 1, abort_flag, status)) && ok;
          tc_fence_after();
          pv_pending = false;
        }
      };
      // p = 2^(x - m) for the whole tile into P (fp16, TMEM); returns the row sum.
      // S is read in 16-column blocks with the next block always in flight,
      // so the TMEM load latency overlaps the arithmetic of the current one;
      // four partial sums keep the dependency chains short.
      auto exp_pass = [&](const float (&bhv)[KHT], float m) -> float2 {
        float2 off[KHT];
        #pragma unroll
        for (int g = 0; g < KHT; ++g) off[g] = make_float2(bhv[g] - m, bhv[g] - m);
        float2 ts[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                        make_float2(0.f, 0.f)};
        uint32_t ua[16], ub[16];
        auto block = [&](int cb, const uint32_t (&u)[16]) {
          uint32_t pk[8];
          #pragma unroll
          for (int k = 0; k < 16; k += 2) {
            const int col = cb + k;
            if (col < BN) {
              const int g = col / WP, kw = col % WP;
              float2 t = ffma2(make_float2(__uint_as_float(u[k]), __uint_as_float(u[k + 1])), sl2v,
                               make_float2(bw[kw], bw[kw + 1]));
              t = fadd2(t, off[g]);
              const float2 p = make_float2(ex2_approx(t.x), ex2_approx(t.y));
              ts[(k / 2) & 3] = fadd2(ts[(k / 2) & 3], p);
              pk[k / 2] = pack_f16x2(p.x, p.y);
            } else {
              pk[k / 2] = 0u;   // padding columns of the product: P = 0
            }
          }
          if (cb == 0) wait_pv();
          tmem_st8(tP + cb / 2, pk);
        };
        tmem_ld16(tS, ua);
        #pragma unroll
        for (int cb = 0; cb < BNP; cb += 32) {
          tmem_wait_ld();
          if (cb + 16 < BNP) tmem_ld16(tS + cb + 16, ub);
          block(cb, ua);
          if (cb + 16 < BNP) {
            tmem_wait_ld();
            if (cb + 32 < BNP) tmem_ld16(tS + cb + 32, ua);
            block(cb + 16, ub);
          }
        }
        return fadd2(fadd2(ts[0], ts[1]), fadd2(ts[2], ts[3]));
      };

      // Online softmax over the segment's key tiles.  The first tile takes the
      // exact maximum (raised by the rel_h estimate below); later tiles
      // exponentiate against the running maximum at once and are redone
      // exactly only if their row sum exceeds kSpecSumLimit (so every p stays
      // within fp16), unless their known rel_h predicts that (kPredictMargin),
      // in which case they go exact without the speculative pass.  The final
      // O / l uses the same running maximum, so skipping rescales changes
      // nothing.
      float m_used = 0.f;
      float bref = 0.f;  // rel_h-free maximum of the row's last exact tile
      float2 lsum = make_float2(0.f, 0.f);
      // largest rel_h term (base 2) over the grid rows this segment covers
      float mbh = NEG_INF;
      for (int kh = sg.j0 * KHT; kh < min(sg.j1 * KHT, H); ++kh) mbh = fmaxf(mbh, bh_row[kh]);
      for (int j = sg.j0; j < sg.j1; ++j, ++gi) {
        // the tile's rel_h terms, and whether to take it exact at once, are
        // settled before the wait for its S, which hides their latency
        const int kh0 = j * KHT;
        float bhv[KHT];
        #pragma unroll
        for (int g = 0; g < KHT; ++g) bhv[g] = (kPadRows || kh0 + g < H) ? bh_row[kh0 + g] : NEG_INF;
        bool exact = j == sg.j0;
        if (!exact) {
          float hb = bhv[0];
          #pragma unroll
          for (int g = 1; g < KHT; ++g) hb = fmaxf(hb, bhv[g]);
          exact = __any_sync(0xffffffffu, hb + bref > m_used + kPredictMargin);
        }
        ok = warp_all(mbar_wait(&bars[kBarSFull + wg], gi & 1, abort_flag, status));
        if (!ok) break;
        tc_fence_after();
        pv_pending = j > sg.j0;

        float2 ts = make_float2(0.f, 0.f);
        if (!exact) {
          ts = exp_pass(bhv, m_used);
          exact = __any_sync(0xffffffffu, !(ts.x + ts.y <= kSpecSumLimit));
        }
        if (exact) {
          float base;
          const float mt = tile_max(bhv, base);
          bref = base;
          if (j == sg.j0) {
            // rel_h is the term that moves the row maximum most between key
            // tiles, so start from this tile's largest s*scale + rel_w plus the
            // row's largest rel_h (less a margin), capped above the exact
            // maximum of this tile: later tiles then seldom pass the row-sum
            // bound and need an exact redo
            const float est = base + mbh - kStartMargin;
            if (__popc(__ballot_sync(0xffffffffu, est - mt > kWideGap)) >= kWideRows) cap = fminf(cap, kSafeCap);
            m_used = fmaxf(fmaxf(mt, fminf(mt + cap, est)), -FLT_MAX);
          } else {
            wait_pv();
            // the same estimate, capped above this tile's exact maximum
            const float m_new = fmaxf(fmaxf(m_used, mt), fminf(mt + cap, base + mbh - kStartMargin));
            const float alpha = ex2_approx(m_used - m_new);
            m_used = m_new;
            lsum.x *= alpha;
            lsum.y *= alpha;
            #pragma unroll
            for (int c = 0; c < D / 32; ++c) {
              uint32_t o[32];
              tmem_ld32(tO + 32 * c, o);
              tmem_wait_ld();
              #pragma unroll
              for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
              tmem_st32(tO + 32 * c, o);
            }
          }
          ts = exp_pass(bhv, m_used);
        }
        lsum = fadd2(lsum, ts);
        if (!ok) break;
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bars[kBarPFull + wg]);
      }
      if (!ok) return false;

      // epilogue: O (fp32, unnormalised) streamed out of TMEM 16 columns at a time
      ok = warp_all(mbar_wait(&bars[kBarODone + wg], (gi - 1) & 1, abort_flag, status));
      if (!ok) return false;
      tc_fence_after();
      const float l = lsum.x + lsum.y;
      // Row-sum check.  Rounding P to fp16 moves each p by at most 2^-11 of
      // itself, or by 2^-25 (in units of the running maximum) for the p that
      // fall below the fp16 normal range, so the output moves by at most
      // max|v| (2^-11 + n 2^-25 / l) for the segment's n valid keys.  The
      // estimated starting maximum may overshoot the row's true maximum and
      // leave l small; a tile with l < n 2^-16 on any row (which keeps the
      // second term at most 2^-9) is neither stored nor published but computed
      // again at the end of the CTA's work with no overshoot (cap 0, l >= 1).
      const int n_keys = (min(sg.j1 * KHT, H) - sg.j0 * KHT) * W;
      volatile int* bad = bad_flag + 2 * wg + (seg & 1);
      if (row_valid && !(l >= ldexpf(static_cast<float>(n_keys), kMinRowSumLog2))) *bad = 1;
      if (!wg_sync()) return false;
      const bool tile_bad = *bad != 0;
      if (r == 0) bad_flag[2 * wg + ((seg + 1) & 1)] = 0;   // every thread has read this segment's flag
      const bool store = store_mask < 0 ? !tile_bad : ((store_mask >> wg) & 1) != 0;
      if (store_mask < 0 && tile_bad) {
        if (r == 0) {
          replay[wg].sg = sg;
          replay[wg].pending = 1;
          *cap_drop = 1;
        }
        own_failed = true;
      }
      if (!store) {
        tc_fence_before();
        if (FUSED) mbar_arrive(&bars[kBarEpiDone]);
        return true;
      }
      // Output rows leave through this warp's quarter of the bias area (no
      // warp of the warpgroup reads its bias rows once O is complete), 64
      // columns at a time: each lane stages its row's 64 columns, 16-byte
      // chunks XOR-swizzled by row so neither side has bank conflicts, then the
      // warp stores runs of 512 contiguous staged bytes (4 bf16/f16 rows or 2
      // fp32 rows per instruction; with head_dim 128 each row's half is a run
      // of 128 or 256 bytes).
      const bool out32 = args.out_fmt == kF32;
      const int row_bytes = out32 ? 256 : 128;   // staged bytes of a row's 64 columns
      const int out_row = row_bytes * Dm::kAtoms;  // bytes of an output row
      uint8_t* ostage = reinterpret_cast<uint8_t*>(area + wq * 32 * kBiasStride);
      auto chunk_at = [&](int row, int k) { return ostage + row * row_bytes + ((k ^ (row & 7)) << 4); };
      auto stage16 = [&](int c0, const float (&v)[16], float scale) {
        if (out32) {
          #pragma unroll
          for (int q = 0; q < 4; ++q)
            *reinterpret_cast<float4*>(chunk_at(lane, c0 / 4 + q)) =
                make_float4(v[4 * q] * scale, v[4 * q + 1] * scale, v[4 * q + 2] * scale, v[4 * q + 3] * scale);
        } else {
          uint32_t w[8];
          #pragma unroll
          for (int k = 0; k < 8; ++k)
            w[k] = args.out_fmt == kBF16 ? pack_bf16x2(v[2 * k] * scale, v[2 * k + 1] * scale)
                                         : pack_f16x2(v[2 * k] * scale, v[2 * k + 1] * scale);
          *reinterpret_cast<uint4*>(chunk_at(lane, c0 / 8)) = make_uint4(w[0], w[1], w[2], w[3]);
          *reinterpret_cast<uint4*>(chunk_at(lane, c0 / 8 + 1)) = make_uint4(w[4], w[5], w[6], w[7]);
        }
      };
      // the staged 64 columns of every row go to columns [64h, 64h + 64) of the output
      auto flush_rows = [&](int h) {
        __syncwarp();
        const int n0 = qt * kBlockM + wq * 32;  // this warp's first row
        uint8_t* obase = reinterpret_cast<uint8_t*>(args.out) + (static_cast<size_t>(bh) * N + n0) * out_row +
                         h * row_bytes;
        const int per = out32 ? 2 : 4;           // rows per 512-byte run
        const int kc = out32 ? 16 : 8;           // chunks per row
        for (int i = 0; i < 32 / per; ++i) {
          const int row = per * i + lane / kc, k = lane % kc;
          if (n0 + row < N)
            *reinterpret_cast<uint4*>(obase + row * out_row + (k << 4)) = *reinterpret_cast<const uint4*>(chunk_at(row, k));
        }
        __syncwarp();
      };
      if (sg.full(n_kv)) {
        const float inv_l = 1.0f / l;
        if (args.lse != nullptr && row_valid) args.lse[static_cast<size_t>(bh) * N + n] = m_used + log2f(l);
        #pragma unroll
        for (int h = 0; h < Dm::kAtoms; ++h) {
          #pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t u[16];
            tmem_ld16(tO + 64 * h + 16 * c, u);
            tmem_wait_ld();
            float v[16];
            #pragma unroll
            for (int k = 0; k < 16; ++k) v[k] = __uint_as_float(u[k]);
            stage16(16 * c, v, inv_l);
          }
          if (h == Dm::kAtoms - 1) {
            tc_fence_before();
            if (FUSED) mbar_arrive(&bars[kBarEpiDone]);
          }
          flush_rows(h);
        }
      } else {
        // Cut unit: the schedule cuts a unit at most once, into two pieces
        // that may run in different CTAs.  Each query tile has its own
        // counter, so the two warpgroups never wait for each other, and
        // nothing waits on another CTA.
        //  - If the other piece has already published its (O, m, l), this
        //    piece merges with it straight from TMEM (no publish, no atomic).
        //  - Otherwise it publishes, then swaps this launch's tag into the
        //    counter; the piece that finds the tag already there arrived
        //    second and merges both published slots.  Whatever an earlier
        //    (or stopped) launch left holds another tag, so the counters
        //    never need clearing.
        // Both merges combine the pieces in the same order (the unit's first
        // piece, then its second) from the same fp32 values, so the result
        // does not depend on which path ran.  O is merged and stored 64
        // columns at a time.
        const int c = blockIdx.x;
        const int slot = (sg.tail == 0) ? 2 * c : 2 * c + 1;
        const long long u0 = static_cast<long long>(sg.u) * n_kv;
        const int c_first = sched.cta_of(u0);
        const int sl0 = (sched.begin(c_first) == u0) ? 2 * c_first : 2 * c_first + 1;
        const int sl1 = 2 * (c_first + 1);
        // a slot of this query tile; this thread's row is O chunk q at
        // float4 index q * 128 + r, and (m, l) at float2 index r after the
        // D * 128 floats of O
        auto slot_of = [&](int s_) { return args.partials + (static_cast<size_t>(s_) * 2 + wg) * slot_floats<D>(); };
        auto ld_chunk = [&](const float* sl, int q) { return __ldcg(reinterpret_cast<const float4*>(sl) + q * kBlockM + r); };
        auto ld_ml = [&](const float* sl) { return __ldcg(reinterpret_cast<const float2*>(sl + D * kBlockM) + r); };
        // columns [64h, 64h + 64) of out = (fa O_a + fb O_b) / (fa l_a + fb l_b),
        // rescaled to the larger running max
        auto merge_store = [&](int h, const float4 (&xa)[16], float2 ma, const float4 (&xb)[16], float2 mb) {
          const float mstar = fmaxf(ma.x, mb.x);
          const float fa = ex2_approx(ma.x - mstar), fb = ex2_approx(mb.x - mstar);
          const float inv_l = 1.0f / (fa * ma.y + fb * mb.y);
          if (h == 0 && args.lse != nullptr && row_valid)
            args.lse[static_cast<size_t>(bh) * N + n] = mstar + log2f(fa * ma.y + fb * mb.y);
          #pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            float v[16];
            #pragma unroll
            for (int q = 0; q < 4; ++q) {
              const float4 a = xa[4 * cc + q], b = xb[4 * cc + q];
              v[4 * q] = fa * a.x + fb * b.x;
              v[4 * q + 1] = fa * a.y + fb * b.y;
              v[4 * q + 2] = fa * a.z + fb * b.z;
              v[4 * q + 3] = fa * a.w + fb * b.w;
            }
            stage16(16 * cc, v, inv_l);
          }
          flush_rows(h);
        };
        unsigned long long* counter = args.counters + 2 * static_cast<size_t>(sg.u) + wg;
        if (r == 0) {
          merge_flag[wg] = ld_acquire_gpu(counter) == args.tag;
          mbar_arrive(&bars[kBarMergeGo + wg]);
        }
        ok = warp_all(mbar_wait(&bars[kBarMergeGo + wg], pseg & 1, abort_flag, status));
        ++pseg;
        if (!ok) return false;
        if (merge_flag[wg]) {
          const float* po = slot_of(slot == sl0 ? sl1 : sl0);
          #pragma unroll 1
          for (int h = 0; h < Dm::kAtoms; ++h) {
            float4 xo[16];
            #pragma unroll
            for (int q = 0; q < 16; ++q) xo[q] = ld_chunk(po, 16 * h + q);
            const float2 mo = ld_ml(po);
            uint32_t oa[64];
            tmem_ld32(tO + 64 * h, *reinterpret_cast<uint32_t(*)[32]>(&oa[0]));
            tmem_ld32(tO + 64 * h + 32, *reinterpret_cast<uint32_t(*)[32]>(&oa[32]));
            tmem_wait_ld();
            if (h == Dm::kAtoms - 1) {
              tc_fence_before();
              if (FUSED) mbar_arrive(&bars[kBarEpiDone]);
            }
            const bool first = slot == sl0;  // warp-uniform
            float4 xa[16], xb[16];
            #pragma unroll
            for (int q = 0; q < 16; ++q) {
              const float4 own = make_float4(__uint_as_float(oa[4 * q]), __uint_as_float(oa[4 * q + 1]),
                                             __uint_as_float(oa[4 * q + 2]), __uint_as_float(oa[4 * q + 3]));
              xa[q] = first ? own : xo[q];
              xb[q] = first ? xo[q] : own;
            }
            const float2 mown = make_float2(m_used, l);
            merge_store(h, xa, first ? mown : mo, xb, first ? mo : mown);
          }
        } else {
          float* ws = slot_of(slot);
          #pragma unroll
          for (int cc = 0; cc < D / 16; ++cc) {
            uint32_t u[16];
            tmem_ld16(tO + 16 * cc, u);
            tmem_wait_ld();
            #pragma unroll
            for (int q = 0; q < 4; ++q)
              __stcg(reinterpret_cast<float4*>(ws) + (4 * cc + q) * kBlockM + r,
                     make_float4(__uint_as_float(u[4 * q]), __uint_as_float(u[4 * q + 1]),
                                 __uint_as_float(u[4 * q + 2]), __uint_as_float(u[4 * q + 3])));
          }
          __stcg(reinterpret_cast<float2*>(ws + D * kBlockM) + r, make_float2(m_used, l));
          tc_fence_before();
          if (FUSED) mbar_arrive(&bars[kBarEpiDone]);
          // mbarrier arrive/wait order these writes before the elected thread's
          // GPU-scope release below (release is cumulative).  Every thread has
          // read merge_flag above before it arrives here, so r == 0 may reuse it.
          mbar_arrive(&bars[kBarPartWritten + wg]);
          const int pw = ppub++;
          if (r == 0) {
            const bool w_ok = mbar_wait(&bars[kBarPartWritten + wg], pw & 1, abort_flag, status);
            merge_flag[wg] = w_ok && atomic_exch_acq_rel_gpu(counter, args.tag) == args.tag;
            mbar_arrive(&bars[kBarMergeGo + wg]);
          }
          ok = warp_all(mbar_wait(&bars[kBarMergeGo + wg], pseg & 1, abort_flag, status));
          ++pseg;
          if (!ok) return false;
          if (merge_flag[wg]) {
            const float* pa = slot_of(sl0);
            const float* pb = slot_of(sl1);
            #pragma unroll 1
            for (int h = 0; h < Dm::kAtoms; ++h) {
              float4 xa[16], xb[16];
              #pragma unroll
              for (int q = 0; q < 16; ++q) {
                xa[q] = ld_chunk(pa, 16 * h + q);
                xb[q] = ld_chunk(pb, 16 * h + q);
              }
              merge_store(h, xa, ld_ml(pa), xb, ld_ml(pb));
            }
          }
        }
      }
      return true;
    };
    Cursor cur(sched, blockIdx.x);
    Segment sg;
    int phase = 0, mask;
    while (next_segment(cur, phase, ok, true, sg, mask)) ok = run_seg(sg, mask) && ok;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

}  // namespace dera
