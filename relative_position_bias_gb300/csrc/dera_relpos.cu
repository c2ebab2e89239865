// C-ABI of libdera_relpos: argument validation, TMA descriptors and kernel
// dispatch for the decomposed rel-pos attention path.  Declarations and the
// contract of every entry point are in include/dera_relpos.h.
#include <algorithm>
#include <atomic>
#include <chrono>
#include <random>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstring>
#include <initializer_list>
#include <mutex>

#include "../../include/dera_relpos.h"
#include "launch.cuh"
#include "project.cuh"

namespace dera {

// Device status word: 0, or DERA_ERR_TIMEOUT once a bounded wait expired.
__device__ int g_status_word = 0;

template <int D>
cudaError_t launch_project_d(const CUtensorMap& q, const CUtensorMap& th, const CUtensorMap& tw,
                             const ProjArgs& args, int in_fmt, int max_ctas, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(relpos_project_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       ProjSmem<D>::kAlloc);
  if (e != cudaSuccess) return e;
  const int n_qtiles = (args.N + kBlockM - 1) / kBlockM;
  // persistent: at most max_ctas CTAs (one per SM), each walking a strided list of tiles
  const unsigned tiles = static_cast<unsigned>(n_qtiles) * static_cast<unsigned>(args.BH);
  const unsigned grid = max_ctas > 0 ? std::min(tiles, static_cast<unsigned>(max_ctas)) : tiles;
  relpos_project_kernel<D><<<grid, kProjThreads, ProjSmem<D>::kAlloc, stream>>>(q, th, tw, args, in_fmt, n_qtiles);
  return cudaGetLastError();
}

cudaError_t launch_project(const CUtensorMap& q, const CUtensorMap& th, const CUtensorMap& tw,
                           const ProjArgs& args, int in_fmt, int head_dim, int max_ctas, cudaStream_t stream) {
  return head_dim == 128 ? launch_project_d<128>(q, th, tw, args, in_fmt, max_ctas, stream)
                         : launch_project_d<64>(q, th, tw, args, in_fmt, max_ctas, stream);
}

// One thread waits on an mbarrier that nothing arrives on; the bounded wait
// gives up after `budget` cycles and records DERA_ERR_TIMEOUT.
__global__ void wait_selftest_kernel(int* status, long long budget) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    if (!mbar_wait_budget(&bar, 0, budget)) atomicCAS(status, 0, DERA_ERR_TIMEOUT);
  }
}

cudaError_t launch_wait_selftest(int* status, long long budget, cudaStream_t stream) {
  wait_selftest_kernel<<<1, 32, 0, stream>>>(status, budget);
  return cudaGetLastError();
}

}  // namespace dera

using namespace dera;

namespace {

constexpr int kMaxDevices = 64;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Device address of the status word on the current device (looked up once per device).
int* status_ptr(int dev) {
  static int* ptrs[kMaxDevices] = {};
  static std::mutex mu;
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<int*>(p);
  }
  return ptrs[dev];
}

bool is16(dera_dtype t) { return t == DERA_F16 || t == DERA_BF16; }
bool is_float(dera_dtype t) { return t == DERA_F16 || t == DERA_BF16 || t == DERA_F32; }
int fmt_of(dera_dtype t) { return t == DERA_F16 ? kF16 : (t == DERA_BF16 ? kBF16 : kF32); }

dera_status check_shape(int BH, int H, int W, int head_dim) {
  if (head_dim != 64 && head_dim != 128) return DERA_ERR_HEAD_DIM;
  if (BH < 0 || H < 1 || W < 1 || H > 64 || W > 64) return DERA_ERR_SHAPE;
  // grid size: ceil(N/256) CTAs per head must fit 2^31 - 1 in total
  const long long pairs = (static_cast<long long>(H) * W + 255) / 256;
  if (pairs * BH > 0x7fffffffLL) return DERA_ERR_SHAPE;
  return DERA_OK;
}

// Host-only checks: non-null and 16-byte aligned (TMA operands).
dera_status check_host(std::initializer_list<const void*> ptrs) {
  for (const void* p : ptrs)
    if (!p) return DERA_ERR_NULL;
  for (const void* p : ptrs)
    if (reinterpret_cast<uintptr_t>(p) % 16 != 0) return DERA_ERR_ALIGN;
  return DERA_OK;
}

// Device memory of device `dev` (the launcher's same-device rule).
dera_status check_ptr(const void* p, int dev) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return DERA_ERR_DEVICE;
  }
  if ((a.type != cudaMemoryTypeDevice && a.type != cudaMemoryTypeManaged) || a.device != dev)
    return DERA_ERR_DEVICE;
  return DERA_OK;
}

bool make_map(CUtensorMap* m, const void* base, CUtensorMapDataType dt, int rank, const cuuint64_t* dims,
              const cuuint64_t* strides_bytes, const cuuint32_t* box) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint32_t es[5] = {1, 1, 1, 1, 1};
  std::memset(m, 0, sizeof(*m));
  return fn(m, dt, rank, const_cast<void*>(base), dims, strides_bytes, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

CUtensorMapDataType tma_type(dera_dtype t) {
  return t == DERA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
}

// Every box is 64 elements (128 bytes, one swizzle atom) wide; a row of
// head_dim d is d / 64 boxes, loaded at element offsets 0 and 64.

// q / out-like tensor [BH, N, d] read in 128-row tiles
bool map_rows(CUtensorMap* m, const void* p, dera_dtype t, int BH, int N, int d) {
  const cuuint64_t row = 2 * static_cast<cuuint64_t>(d);
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {row, static_cast<cuuint64_t>(N) * row};
  const cuuint32_t box[3] = {64, 128, 1};
  return make_map(m, p, tma_type(t), 3, dims, strides, box);
}

// k / v viewed as [BH, H, W, d], read in tiles of KHT grid rows x WP columns
bool map_keys(CUtensorMap* m, const void* p, dera_dtype t, int BH, int H, int W, int d, int WP, int KHT) {
  const cuuint64_t row = 2 * static_cast<cuuint64_t>(d);
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(W), static_cast<cuuint64_t>(H),
                              static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[3] = {row, static_cast<cuuint64_t>(W) * row, static_cast<cuuint64_t>(H) * W * row};
  const cuuint32_t box[4] = {64, static_cast<cuuint32_t>(WP), static_cast<cuuint32_t>(KHT), 1};
  return make_map(m, p, tma_type(t), 4, dims, strides, box);
}

// table [2L-1, d], one 128-row box per 64 columns (rows past 2L-1 read as zero)
bool map_table(CUtensorMap* m, const void* p, dera_dtype t, int L, int d) {
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(2 * L - 1)};
  const cuuint64_t strides[1] = {2 * static_cast<cuuint64_t>(d)};
  const cuuint32_t box[2] = {64, 128};
  return make_map(m, p, tma_type(t), 2, dims, strides, box);
}

int padded_width(int W) { return W <= 16 ? 16 : (W <= 32 ? 32 : (W <= 40 ? 40 : 64)); }
// grid rows per key tile (KeyTile<WP, d>::KHT), and the forward's
// (FwdKeyTile<WP, d>::KHT: three for a 40-column grid with head_dim 64)
int rows_per_tile(int WP, int d) {
  if (d == 64) return WP <= 16 ? 8 : (WP <= 32 ? 4 : 2);
  return WP <= 16 ? 4 : (WP <= 40 ? 2 : 1);
}
int fwd_rows_per_tile(int WP, int d) { return (d == 64 && WP == 40) ? 3 : rows_per_tile(WP, d); }

// Streaming-multiprocessor count of a device (cached; 0 if the query fails).
int sm_count(int dev) {
  static int counts[kMaxDevices] = {};
  static std::mutex mu;
  if (dev < 0 || dev >= kMaxDevices) return 0;
  std::lock_guard<std::mutex> lock(mu);
  if (counts[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    counts[dev] = n;
  }
  return counts[dev];
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Arrival tags of the split schedule's per-unit counters: a 64-bit sequence
// from a random start, so no two launches of this process share a tag and
// counters left by any earlier launch (finished or stopped) never match.
unsigned long long next_launch_tag() {
  static std::atomic<unsigned long long> next{[] {
    unsigned long long seed = 0x9e3779b97f4a7c15ull ^ static_cast<unsigned long long>(
        std::chrono::steady_clock::now().time_since_epoch().count());
    try {
      std::random_device rd;
      seed ^= (static_cast<unsigned long long>(rd()) << 32) ^ rd();
    } catch (...) {
      // no entropy source: the clock alone seeds the sequence
    }
    return seed;
  }()};
  return next.fetch_add(1, std::memory_order_relaxed);
}

// Work decomposition of one call: units are pairs of 128-row query tiles.
constexpr int kMinSplitKeyTiles = 4;
struct Plan {
  int n_qtiles, n_pairs, n_units, n_kv, ctas;
  bool split;              // stream-K over `ctas` persistent CTAs (needs the workspace)
  size_t counters_bytes, partial_bytes;
};

// CTAs of a schedule without cuts: one per SM, taking whole units
// round-robin, or one per unit when there are fewer units (or the SM count
// is unknown).
int uncut_ctas(int n_units, int sms) { return sms > 0 && n_units > sms ? sms : n_units; }

Plan make_plan(int BH, int H, int W, int d, int sms) {
  Plan p;
  const int N = H * W;
  const int KHT = fwd_rows_per_tile(padded_width(W), d);
  p.n_qtiles = (N + kBlockM - 1) / kBlockM;
  p.n_pairs = (p.n_qtiles + 1) / 2;
  p.n_units = BH * p.n_pairs;
  p.n_kv = (H + KHT - 1) / KHT;
  // Split only when the units do not fill whole waves of one CTA per SM; with
  // more units than CTAs every CTA range spans at least one unit's key tiles,
  // so a unit is cut into at most two segments.  Units of fewer than
  // kMinSplitKeyTiles key tiles (small grids such as 14x14 windows) are not
  // split: the merge of a cut unit costs more than the imbalance it removes
  // (measured on 25 windows x 12 heads of 14x14: 28 us whole, 32 us split).
  p.split = sms > 0 && p.n_kv >= kMinSplitKeyTiles && p.n_units > sms && p.n_units % sms != 0;
  p.ctas = p.split ? sms : uncut_ctas(p.n_units, sms);
  p.counters_bytes = align256(static_cast<size_t>(p.n_units) * 2 * sizeof(unsigned long long));  // one per query tile
  p.partial_bytes = static_cast<size_t>(2) * sms * 2 * (d == 128 ? slot_floats<128>() : slot_floats<64>()) *
                    sizeof(float);
  return p;
}

size_t workspace_bytes_for(const Plan& p) { return p.split ? p.counters_bytes + p.partial_bytes : 0; }
dera_status current_device(int* dev) {
  if (cudaGetDevice(dev) != cudaSuccess) {
    cudaGetLastError();
    return DERA_ERR_CUDA;
  }
  return DERA_OK;
}

#define DERA_TRY(expr)              \
  do {                              \
    const dera_status s_ = (expr);  \
    if (s_ != DERA_OK) return s_;   \
  } while (0)

// Workspace of the backward: fp32 regions, each 256-byte aligned.
struct BwdLayout {
  size_t rel_h, rel_w, D, hl, parts, total;
  int n_qtiles;
  BwdLayout(int BH, int H, int W) {
    const size_t rows = static_cast<size_t>(BH) * H * W;
    n_qtiles = (H * W + kBlockM - 1) / kBlockM;
    size_t o = 0;
    auto take = [&](size_t floats) {
      const size_t at = o;
      o += align256(floats * sizeof(float));
      return at;
    };
    rel_h = take(rows * H);
    rel_w = take(rows * W);
    D = take(rows);
    hl = take(static_cast<size_t>(BH) * H * n_qtiles * kBlockM);
    parts = take(static_cast<size_t>(BH) * n_qtiles * (2 * H - 1 + 2 * W - 1) * 64);
    total = o;
  }
};

dera_status run_attention(const void* q, const void* k, const void* v, const void* a, const void* b, void* out,
                          int BH, int H, int W, int d, float scale, dera_dtype in_dtype, dera_dtype bias_dtype,
                          dera_dtype out_dtype, bool fused, void* workspace, size_t workspace_bytes,
                          void* stream, float* lse = nullptr) {
  int dev = 0;
  DERA_TRY(current_device(&dev));
  const int N = H * W;
  Plan plan = make_plan(BH, H, W, d, sm_count(dev));
  if (plan.split && (workspace == nullptr || workspace_bytes < workspace_bytes_for(plan))) {
    plan.split = false;  // no (or too small a) workspace: whole units, round-robin
    plan.ctas = uncut_ctas(plan.n_units, sm_count(dev));
  }
  const int WP = padded_width(W), KHT = fwd_rows_per_tile(WP, d);
  AttnMaps maps;
  if (!map_rows(&maps.q, q, in_dtype, BH, N, d) || !map_keys(&maps.k, k, in_dtype, BH, H, W, d, WP, KHT) ||
      !map_keys(&maps.v, v, in_dtype, BH, H, W, d, WP, KHT))
    return DERA_ERR_CUDA;
  if (fused) {
    if (!map_table(&maps.th, a, in_dtype, H, d) || !map_table(&maps.tw, b, in_dtype, W, d)) return DERA_ERR_CUDA;
  } else {
    maps.th = maps.q;  // unused by the compact-bias kernel
    maps.tw = maps.q;
  }
  AttnArgs args;
  args.rel_h = fused ? nullptr : a;
  args.rel_w = fused ? nullptr : b;
  args.out = out;
  args.status = status_ptr(dev);
  if (!args.status) return DERA_ERR_CUDA;
  args.BH = BH;
  args.H = H;
  args.W = W;
  args.N = N;
  args.n_qtiles = plan.n_qtiles;
  args.n_pairs = plan.n_pairs;
  args.n_units = plan.n_units;
  args.n_kv = plan.n_kv;
  args.partials = nullptr;
  args.counters = nullptr;
  args.tag = 0;
  args.scale_log2 = scale * kLog2e;
  args.in_fmt = fmt_of(in_dtype);
  args.bias_fmt = fmt_of(bias_dtype);
  args.out_fmt = fmt_of(out_dtype);
  args.lse = lse;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (plan.split) {
    args.counters = static_cast<unsigned long long*>(workspace);
    args.tag = next_launch_tag();
    args.partials = reinterpret_cast<float*>(static_cast<char*>(workspace) + plan.counters_bytes);
  }
  cudaError_t e;
  switch (WP) {
    case 16: e = launch_attention<16>(maps, args, plan.ctas, fused, d, s); break;
    case 32: e = launch_attention<32>(maps, args, plan.ctas, fused, d, s); break;
    case 40: e = launch_attention<40>(maps, args, plan.ctas, fused, d, s); break;
    default: e = launch_attention<64>(maps, args, plan.ctas, fused, d, s); break;
  }
  return e == cudaSuccess ? DERA_OK : DERA_ERR_CUDA;
}

// Scratch of dera_relpos_fused_noalloc: a buffer compiled into the library,
// for callers that cannot allocate device memory.  In host code the array's
// name only stands in for the symbol; its device address is looked up once
// per device (with that device current) and passed to the kernel.
static __device__ __align__(256) unsigned char g_noalloc_scratch[DERA_NOALLOC_SCRATCH_BYTES];

void* noalloc_scratch(int dev) {
  static void* ptrs[kMaxDevices] = {};
  static std::mutex mu;
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    ptrs[dev] = p;
  }
  return ptrs[dev];
}

}  // namespace

extern "C" {

const char* dera_status_string(dera_status status) {
  switch (status) {
    case DERA_OK: return "DERA_OK";
    case DERA_ERR_NULL: return "DERA_ERR_NULL: a required pointer is NULL";
    case DERA_ERR_SHAPE: return "DERA_ERR_SHAPE: H, W or BH out of range";
    case DERA_ERR_DTYPE: return "DERA_ERR_DTYPE: unsupported dtype for this argument";
    case DERA_ERR_HEAD_DIM: return "DERA_ERR_HEAD_DIM: head_dim must be 64 or 128";
    case DERA_ERR_ALIGN: return "DERA_ERR_ALIGN: pointer not 16-byte aligned";
    case DERA_ERR_DEVICE: return "DERA_ERR_DEVICE: pointer is not device memory of the current device";
    case DERA_ERR_TIMEOUT: return "DERA_ERR_TIMEOUT: a bounded wait expired inside a kernel";
    case DERA_ERR_CUDA: return "DERA_ERR_CUDA: a CUDA call failed";
    case DERA_ERR_SCRATCH: return "DERA_ERR_SCRATCH: the problem needs more scratch than the static buffer holds";
  }
  return "DERA_ERR_UNKNOWN";
}

int dera_relpos_abi_version(void) { return DERA_RELPOS_ABI_VERSION; }

dera_status dera_relpos_project(const void* q, const void* rel_pos_h, const void* rel_pos_w, void* rel_h,
                                void* rel_w, int BH, int H, int W, int head_dim, dera_dtype in_dtype,
                                dera_dtype bias_dtype, void* stream) {
  DERA_TRY(check_shape(BH, H, W, head_dim));
  if (!is16(in_dtype) || !is_float(bias_dtype)) return DERA_ERR_DTYPE;
  if (BH == 0) return DERA_OK;  // empty batch: nothing to read or write
  DERA_TRY(check_host({q, rel_pos_h, rel_pos_w, rel_h, rel_w}));
  int dev = 0;
  DERA_TRY(current_device(&dev));
  for (const void* p : {q, rel_pos_h, rel_pos_w, static_cast<const void*>(rel_h), static_cast<const void*>(rel_w)})
    DERA_TRY(check_ptr(p, dev));
  const int N = H * W;
  CUtensorMap mq, mh, mw;
  if (!map_rows(&mq, q, in_dtype, BH, N, head_dim) || !map_table(&mh, rel_pos_h, in_dtype, H, head_dim) ||
      !map_table(&mw, rel_pos_w, in_dtype, W, head_dim))
    return DERA_ERR_CUDA;
  ProjArgs args;
  args.rel_h = rel_h;
  args.rel_w = rel_w;
  args.status = status_ptr(dev);
  if (!args.status) return DERA_ERR_CUDA;
  args.BH = BH;
  args.H = H;
  args.W = W;
  args.N = N;
  args.bias_fmt = fmt_of(bias_dtype);
  const cudaError_t e =
      launch_project(mq, mh, mw, args, fmt_of(in_dtype), head_dim, sm_count(dev), static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? DERA_OK : DERA_ERR_CUDA;
}

dera_status dera_relpos_workspace_size(int BH, int H, int W, int head_dim, size_t* bytes) {
  if (!bytes) return DERA_ERR_NULL;
  DERA_TRY(check_shape(BH, H, W, head_dim));
  *bytes = 0;
  if (BH == 0) return DERA_OK;
  int dev = 0;
  DERA_TRY(current_device(&dev));
  *bytes = workspace_bytes_for(make_plan(BH, H, W, head_dim, sm_count(dev)));
  return DERA_OK;
}

dera_status dera_relpos_attention(const void* q, const void* k, const void* v, const void* rel_h,
                                  const void* rel_w, void* out, int BH, int H, int W, int head_dim, float scale,
                                  dera_dtype in_dtype, dera_dtype bias_dtype, dera_dtype out_dtype,
                                  void* workspace, size_t workspace_bytes, void* stream) {
  DERA_TRY(check_shape(BH, H, W, head_dim));
  if (!is16(in_dtype) || !is_float(bias_dtype) || !(out_dtype == DERA_F32 || out_dtype == in_dtype))
    return DERA_ERR_DTYPE;
  if (BH == 0) return DERA_OK;  // empty batch: nothing to read or write
  DERA_TRY(check_host({q, k, v, rel_h, rel_w, out}));
  int dev = 0;
  DERA_TRY(current_device(&dev));
  for (const void* p : {q, k, v, rel_h, rel_w, static_cast<const void*>(out)}) DERA_TRY(check_ptr(p, dev));
  if (workspace) {
    if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return DERA_ERR_ALIGN;
    DERA_TRY(check_ptr(workspace, dev));
  }
  return run_attention(q, k, v, rel_h, rel_w, out, BH, H, W, head_dim, scale, in_dtype, bias_dtype, out_dtype, false,
                       workspace, workspace_bytes, stream);
}

dera_status dera_relpos_fused(const void* q, const void* k, const void* v, const void* rel_pos_h,
                              const void* rel_pos_w, void* out, int BH, int H, int W, int head_dim, float scale,
                              dera_dtype in_dtype, dera_dtype out_dtype, void* workspace, size_t workspace_bytes,
                              void* stream) {
  DERA_TRY(check_shape(BH, H, W, head_dim));
  if (!is16(in_dtype) || !(out_dtype == DERA_F32 || out_dtype == in_dtype)) return DERA_ERR_DTYPE;
  if (BH == 0) return DERA_OK;  // empty batch: nothing to read or write
  DERA_TRY(check_host({q, k, v, rel_pos_h, rel_pos_w, out}));
  int dev = 0;
  DERA_TRY(current_device(&dev));
  for (const void* p : {q, k, v, rel_pos_h, rel_pos_w, static_cast<const void*>(out)})
    DERA_TRY(check_ptr(p, dev));
  if (workspace) {
    if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return DERA_ERR_ALIGN;
    DERA_TRY(check_ptr(workspace, dev));
  }
  return run_attention(q, k, v, rel_pos_h, rel_pos_w, out, BH, H, W, head_dim, scale, in_dtype, in_dtype, out_dtype, true,
                       workspace, workspace_bytes, stream);
}

dera_status dera_relpos_fused_lse(const void* q, const void* k, const void* v, const void* rel_pos_h,
                                  const void* rel_pos_w, void* out, float* lse, int BH, int H, int W,
                                  int head_dim, float scale, dera_dtype in_dtype, dera_dtype out_dtype,
                                  void* workspace, size_t workspace_bytes, void* stream) {
  DERA_TRY(check_shape(BH, H, W, head_dim));
  if (!is16(in_dtype) || !(out_dtype == DERA_F32 || out_dtype == in_dtype)) return DERA_ERR_DTYPE;
  if (BH == 0) return DERA_OK;
  DERA_TRY(check_host({q, k, v, rel_pos_h, rel_pos_w, out, lse}));
  int dev = 0;
  DERA_TRY(current_device(&dev));
  for (const void* p : {q, k, v, rel_pos_h, rel_pos_w, static_cast<const void*>(out), static_cast<const void*>(lse)})
    DERA_TRY(check_ptr(p, dev));
  if (workspace) {
    if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return DERA_ERR_ALIGN;
    DERA_TRY(check_ptr(workspace, dev));
  }
  return run_attention(q, k, v, rel_pos_h, rel_pos_w, out, BH, H, W, head_dim, scale, in_dtype, in_dtype, out_dtype, true,
                       workspace, workspace_bytes, stream, lse);
}

dera_status dera_relpos_backward_workspace_size(int BH, int H, int W, int head_dim, size_t* bytes) {
  if (!bytes) return DERA_ERR_NULL;
  DERA_TRY(check_shape(BH, H, W, head_dim));
  if (head_dim != 64) return DERA_ERR_HEAD_DIM;
  *bytes = BwdLayout(BH, H, W).total;
  return DERA_OK;
}

dera_status dera_relpos_fused_backward(const void* q, const void* k, const void* v, const void* rel_pos_h,
                                       const void* rel_pos_w, const void* out, const float* lse,
                                       const void* dout, void* dq, void* dk, void* dv, float* drel_pos_h,
                                       float* drel_pos_w, int BH, int H, int W, int head_dim, float scale,
                                       dera_dtype in_dtype, dera_dtype out_dtype, dera_dtype grad_dtype,
                                       void* workspace, size_t workspace_bytes, void* stream) {
  DERA_TRY(check_shape(BH, H, W, head_dim));
  if (head_dim != 64) return DERA_ERR_HEAD_DIM;
  if (!is16(in_dtype) || !(out_dtype == DERA_F32 || out_dtype == in_dtype) ||
      !(grad_dtype == DERA_F32 || grad_dtype == in_dtype))
    return DERA_ERR_DTYPE;
  int dev = 0;
  if (BH == 0) {
    // no rows: only the table gradients are written, as zeros
    DERA_TRY(check_host({drel_pos_h, drel_pos_w}));
    DERA_TRY(current_device(&dev));
    for (const void* p : {static_cast<const void*>(drel_pos_h), static_cast<const void*>(drel_pos_w)})
      DERA_TRY(check_ptr(p, dev));
    const size_t th_bytes = static_cast<size_t>(2 * H - 1) * 64 * sizeof(float);
    const size_t tw_bytes = static_cast<size_t>(2 * W - 1) * 64 * sizeof(float);
    cudaStream_t s0 = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(drel_pos_h, 0, th_bytes, s0) != cudaSuccess ||
        cudaMemsetAsync(drel_pos_w, 0, tw_bytes, s0) != cudaSuccess)
      return DERA_ERR_CUDA;
    return DERA_OK;
  }
  DERA_TRY(check_host({q, k, v, rel_pos_h, rel_pos_w, out, lse, dout, dq, dk, dv, drel_pos_h, drel_pos_w}));
  DERA_TRY(current_device(&dev));
  const BwdLayout L(BH, H, W);
  if (!workspace || workspace_bytes < L.total) return DERA_ERR_SCRATCH;
  if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return DERA_ERR_ALIGN;
  for (const void* p : {q, k, v, rel_pos_h, rel_pos_w, out, static_cast<const void*>(lse), dout,
                        static_cast<const void*>(dq), static_cast<const void*>(dk), static_cast<const void*>(dv),
                        static_cast<const void*>(drel_pos_h), static_cast<const void*>(drel_pos_w),
                        static_cast<const void*>(workspace)})
    DERA_TRY(check_ptr(p, dev));
  const int N = H * W;
  char* ws = static_cast<char*>(workspace);
  float* rel_h = reinterpret_cast<float*>(ws + L.rel_h);
  float* rel_w = reinterpret_cast<float*>(ws + L.rel_w);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int* st = status_ptr(dev);
  if (!st) return DERA_ERR_CUDA;
  // the compact bias, fp32, by the forward's projection kernel
  {
    CUtensorMap mq, mh, mw;
    if (!map_rows(&mq, q, in_dtype, BH, N, 64) || !map_table(&mh, rel_pos_h, in_dtype, H, 64) ||
        !map_table(&mw, rel_pos_w, in_dtype, W, 64))
      return DERA_ERR_CUDA;
    ProjArgs pa;
    pa.rel_h = rel_h;
    pa.rel_w = rel_w;
    pa.status = st;
    pa.BH = BH;
    pa.H = H;
    pa.W = W;
    pa.N = N;
    pa.bias_fmt = kF32;
    if (launch_project(mq, mh, mw, pa, fmt_of(in_dtype), 64, sm_count(dev), s) != cudaSuccess) return DERA_ERR_CUDA;
  }
  const int WP = padded_width(W), KHT = rows_per_tile(WP, 64);
  BwdMaps maps;
  if (!map_rows(&maps.q, q, in_dtype, BH, N, 64) || !map_rows(&maps.dout, dout, in_dtype, BH, N, 64) ||
      !map_keys(&maps.k, k, in_dtype, BH, H, W, 64, WP, KHT) || !map_keys(&maps.v, v, in_dtype, BH, H, W, 64, WP, KHT) ||
      !map_table(&maps.th, rel_pos_h, in_dtype, H, 64) || !map_table(&maps.tw, rel_pos_w, in_dtype, W, 64))
    return DERA_ERR_CUDA;
  BwdArgs a;
  a.rel_h = rel_h;
  a.rel_w = rel_w;
  a.lse = lse;
  a.out = out;
  a.dout = dout;
  a.D = reinterpret_cast<float*>(ws + L.D);
  a.hl = reinterpret_cast<float*>(ws + L.hl);
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.parts = reinterpret_cast<float*>(ws + L.parts);
  a.dth = drel_pos_h;
  a.dtw = drel_pos_w;
  a.status = st;
  a.BH = BH;
  a.H = H;
  a.W = W;
  a.N = N;
  a.n_qtiles = L.n_qtiles;
  a.n_kv = (H + KHT - 1) / KHT;
  a.scale = scale;
  a.scale_log2 = scale * kLog2e;
  a.in_fmt = fmt_of(in_dtype);
  a.out_fmt = fmt_of(out_dtype);
  a.grad_fmt = fmt_of(grad_dtype);
  return launch_backward(maps, a, WP, s) == cudaSuccess ? DERA_OK : DERA_ERR_CUDA;
}

dera_status dera_relpos_device_status(int* status, int reset) {
  if (!status) return DERA_ERR_NULL;
  if (cudaDeviceSynchronize() != cudaSuccess) return DERA_ERR_CUDA;
  if (cudaMemcpyFromSymbol(status, g_status_word, sizeof(int)) != cudaSuccess) return DERA_ERR_CUDA;
  if (reset) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_status_word, &zero, sizeof(int)) != cudaSuccess) return DERA_ERR_CUDA;
  }
  return DERA_OK;
}

dera_status dera_relpos_selftest_wait_timeout(long long budget_cycles, void* stream) {
  int dev = 0;
  DERA_TRY(current_device(&dev));
  int* st = status_ptr(dev);
  if (!st) return DERA_ERR_CUDA;
  if (budget_cycles < 1000) budget_cycles = 1000;
  if (budget_cycles > 4000000000LL) budget_cycles = 4000000000LL;
  return launch_wait_selftest(st, budget_cycles, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? DERA_OK
             : DERA_ERR_CUDA;
}

dera_status dera_relpos_fused_noalloc(const void* q, const void* k, const void* v, const void* rel_pos_h,
                                      const void* rel_pos_w, void* out, int BH, int H, int W, int head_dim,
                                      float scale, dera_dtype in_dtype, dera_dtype out_dtype, void* stream) {
  DERA_TRY(check_shape(BH, H, W, head_dim));
  if (!is16(in_dtype) || !(out_dtype == DERA_F32 || out_dtype == in_dtype)) return DERA_ERR_DTYPE;
  if (BH == 0) return DERA_OK;  // empty batch: nothing to read or write
  DERA_TRY(check_host({q, k, v, rel_pos_h, rel_pos_w, out}));
  int dev = 0;
  DERA_TRY(current_device(&dev));
  // The size limit is decided before any pointer is examined, and a device whose SM count
  // cannot be read is refused (that count sizes the schedule and its scratch).
  const int sms = sm_count(dev);
  if (sms <= 0) return DERA_ERR_CUDA;
  const size_t need = workspace_bytes_for(make_plan(BH, H, W, head_dim, sms));
  if (need > DERA_NOALLOC_SCRATCH_BYTES) return DERA_ERR_SCRATCH;
  for (const void* p : {q, k, v, rel_pos_h, rel_pos_w, static_cast<const void*>(out)})
    DERA_TRY(check_ptr(p, dev));
  void* scratch = nullptr;
  if (need > 0) {
    scratch = noalloc_scratch(dev);
    if (!scratch) return DERA_ERR_CUDA;
  }
  return run_attention(q, k, v, rel_pos_h, rel_pos_w, out, BH, H, W, head_dim, scale, in_dtype, in_dtype, out_dtype, true,
                       scratch, need, stream);
}

}  // extern "C"
