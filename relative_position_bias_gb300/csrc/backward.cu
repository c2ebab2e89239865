// Launchers of the backward kernels (csrc/backward.cuh): the two attention
// kernels for every padded width and input dtype, then the table reduction.
#include "backward.cuh"
#include "launch.cuh"

namespace dera {

namespace {

template <int WP, bool BF16>
cudaError_t launch_bwd_attn(const BwdMaps& maps, const BwdArgs& args, cudaStream_t stream) {
  auto rows = relpos_bwd_rows_kernel<WP, BF16>;
  auto cols = relpos_bwd_cols_kernel<WP, BF16>;
  cudaError_t e = cudaFuncSetAttribute(rows, cudaFuncAttributeMaxDynamicSharedMemorySize, BwdRowsSmem::kAlloc);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(cols, cudaFuncAttributeMaxDynamicSharedMemorySize, BwdColsSmem::kAlloc);
  if (e != cudaSuccess) return e;
  const unsigned grid_rows = static_cast<unsigned>(args.BH) * static_cast<unsigned>(args.n_qtiles);
  rows<<<grid_rows, kBwdRowsThreads, BwdRowsSmem::kAlloc, stream>>>(maps.q, maps.dout, maps.k, maps.v, maps.th,
                                                                     maps.tw, args);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const unsigned grid_cols = static_cast<unsigned>(args.BH) * static_cast<unsigned>(args.n_kv);
  cols<<<grid_cols, kBwdColsThreads, BwdColsSmem::kAlloc, stream>>>(maps.q, maps.dout, maps.k, maps.v, args);
  return cudaGetLastError();
}

template <int WP>
cudaError_t launch_bwd_attn_w(const BwdMaps& maps, const BwdArgs& args, cudaStream_t stream) {
  return args.in_fmt == kBF16 ? launch_bwd_attn<WP, true>(maps, args, stream)
                              : launch_bwd_attn<WP, false>(maps, args, stream);
}

}  // namespace

cudaError_t launch_backward(const BwdMaps& maps, const BwdArgs& args, int WP, cudaStream_t stream) {
  cudaError_t e;
  switch (WP) {
    case 16: e = launch_bwd_attn_w<16>(maps, args, stream); break;
    case 32: e = launch_bwd_attn_w<32>(maps, args, stream); break;
    case 40: e = launch_bwd_attn_w<40>(maps, args, stream); break;
    default: e = launch_bwd_attn_w<64>(maps, args, stream); break;
  }
  if (e != cudaSuccess) return e;
  const unsigned blocks = static_cast<unsigned>(args.BH) * static_cast<unsigned>(args.n_qtiles);
  const int total = (2 * args.H - 1 + 2 * args.W - 1) * 64;
  relpos_bwd_tables_kernel<<<(total + 31) / 32, 256, 0, stream>>>(args, static_cast<int>(blocks));
  return cudaGetLastError();
}

}  // namespace dera
