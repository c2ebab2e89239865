// Shared definitions of the rel-pos attention kernels: launch arguments,
// key-tile geometry and the on-chip skew of the q.table^T products.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "ptx.cuh"

namespace dera {

constexpr int kBlockM = 128;      // query rows per tile (one TMEM lane per row)
constexpr int kRowBytes = 128;    // 64 16-bit elements: one swizzle atom of a row
constexpr int kTileBytes = 128 * kRowBytes;  // one atom of a 128-row operand tile (16 KB)
constexpr float kLog2e = 1.4426950408889634f;
// One partial-result slot of a query tile with head_dim D: O as D / 4
// column chunks of 4 floats, chunk-major ([D / 4][128] float4, so a warp's 32
// rows of one chunk are 512 contiguous bytes), then (m, l) per row ([128]
// float2).
template <int D>
constexpr int slot_floats() { return 128 * (D + 2); }

// Key tiles cover KHT whole grid rows of WP (>= W) padded columns, so the
// column of a key inside its tile fixes kw at compile time.  The padded
// columns (kw >= W) and padded rows (kh >= H) are zero-filled by TMA and get
// a -inf bias, which removes them from the softmax.  With head_dim 128 a key
// tile holds about 64 keys (half as many grid rows), so that its K and V fit
// the shared-memory ring and its S, P and O the TMEM budget.
template <int WP, int D = 64>
struct KeyTile {
  static_assert(D == 64 || D == 128, "head_dim 64 or 128");
  static constexpr int KHT = D == 64 ? (WP <= 16 ? 8 : (WP <= 32 ? 4 : 2)) : (WP <= 16 ? 4 : (WP <= 40 ? 2 : 1));
  static constexpr int BN = KHT * WP;
  static_assert(BN % 16 == 0 && BN <= 128, "tcgen05 N constraint");
  static_assert(WP % 2 == 0, "packed pairs must not straddle a grid row");
};

// Operand tiles of head dimension D are D / 64 swizzle atoms: an atom holds
// 64 elements (128 bytes) of every row, and TMA loads each atom as one box.
template <int D>
constexpr int atoms_of() { return D / 64; }

// Element types.
enum : int { kF16 = 0, kBF16 = 1, kF32 = 2 };

struct AttnArgs {
  const void* rel_h;   // [BH, N, H] (compact entry)
  const void* rel_w;   // [BH, N, W]
  void* out;           // [BH, N, head_dim]
  int* status;         // device status word
  float* partials;     // [2 * gridDim.x][2][slot_floats<D>()] partial results (split units only)
  unsigned long long* counters;  // [n_units][2] arrival tags per unit and query tile (split units only)
  unsigned long long tag;        // this launch's arrival tag: no earlier launch of the process used it
  int BH, H, W, N;
  int n_qtiles;        // ceil(N / 128)
  int n_pairs;         // ceil(n_qtiles / 2): query-tile pairs per head
  int n_units;         // BH * n_pairs
  int n_kv;            // ceil(H / KHT)
  float scale_log2;    // scale * log2(e)
  int in_fmt;          // kF16 | kBF16
  int bias_fmt;        // kF32 | kBF16 | kF16 (compact entry)
  int out_fmt;         // kF32 | in_fmt
  float* lse;          // [BH, N] base-2 log-sum-exp of each row's logits, or null
};

struct ProjArgs {
  void* rel_h;         // [BH, N, H]
  void* rel_w;         // [BH, N, W]
  int* status;
  int BH, H, W, N;
  int bias_fmt;        // kF32 | kBF16 | kF16
};

// Arguments of the backward kernels (csrc/backward.cuh).
struct BwdArgs {
  const float* rel_h;   // [BH, N, H] compact bias (fp32, natural units)
  const float* rel_w;   // [BH, N, W]
  const float* lse;     // [BH, N] base-2 log-sum-exp of each row's logits (forward)
  const void* out;      // [BH, N, 64] forward output (input dtype)
  const void* dout;     // [BH, N, 64] upstream gradient (input dtype)
  float* D;             // [BH, N] -(dO . out) per row (rows kernel writes, cols kernel reads)
  float* hl;            // [BH, H, n_qtiles * 128] log2(e) rel_h - lse, key grid row major
                        // (rows kernel writes, cols kernel reads)
  void* dq;             // [BH, N, 64] grad dtype (rows kernel)
  void* dk;             // [BH, N, 64] grad dtype (cols kernel)
  void* dv;             // [BH, N, 64]
  float* parts;         // [BH * n_qtiles][(2H-1) + (2W-1)][64] per-query-tile table-gradient partials
  float* dth;           // [2H-1, 64] fp32
  float* dtw;           // [2W-1, 64] fp32
  int* status;
  int BH, H, W, N;
  int n_qtiles, n_kv;
  float scale, scale_log2;
  int in_fmt, out_fmt, grad_fmt;
};

// Warp-uniform wait result: tcgen05.ld/st are warp-collective, so a warp
// either proceeds as a whole or stops as a whole.
__device__ __forceinline__ bool warp_all(bool ok) { return __all_sync(0xffffffffu, ok); }

__device__ __forceinline__ float load_elem(const void* p, size_t i, int fmt) {
  if (fmt == kF32) return __ldg(reinterpret_cast<const float*>(p) + i);
  const unsigned short raw = __ldg(reinterpret_cast<const unsigned short*>(p) + i);
  if (fmt == kBF16) return __uint_as_float(static_cast<uint32_t>(raw) << 16);
  return __half2float(__ushort_as_half(raw));
}

// ---------------------------------------------------------------------------
// On-chip skew of the tensor-core products G = Q_tile . [T_h ; T_w]^T.
//
// The thread owning query row r (token n, grid coordinates qh, qw) holds
// G[r, c] = q_n . table[c] in TMEM lane r.  The decomposed bias needs
//   rel_h[n, kh] = G_h[r, qh - kh + H - 1],  rel_w[n, kw] = G_w[r, qw - kw + W - 1],
// a per-row shift.  Each TMEM chunk is written to shared memory at an offset
// that depends on the row (dynamic address, static register index), so the
// shifted row can then be read back with static indices.
//
// dst[r * stride + (len - 1 - j)] = scale * G[r, first + j] for j in [0, len),
// i.e. dst[r][k] = scale * G[r, first + len - 1 - k].  With first = qh and
// len = H this gives dst[r][kh] = scale * rel_h[n, kh].
__device__ __forceinline__ void skew_row_to_smem(uint32_t tmem_row_base, int first, int len, float* dst_row,
                                                 float scale) {
  // Columns [first, first + len) of this row; chunks of 32 are loaded
  // warp-wide (every lane must take part in tcgen05.ld), so the chunk range
  // is the warp's union.
  int lo = first, hi = first + len;
  #pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, off));
    hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, off));
  }
  for (int cb = lo & ~31; cb < hi; cb += 32) {
    uint32_t u[32];
    tmem_ld32(tmem_row_base + static_cast<uint32_t>(cb), u);
    tmem_wait_ld();
    #pragma unroll
    for (int k = 0; k < 32; ++k) {
      const int j = cb + k - first;
      if (j >= 0 && j < len) dst_row[len - 1 - j] = scale * __uint_as_float(u[k]);
    }
  }
}

}  // namespace dera
