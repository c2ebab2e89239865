// Definition of launch_attention<WP>; included by one .cu per padded width.
#pragma once
#include "attention.cuh"
#include "launch.cuh"

namespace dera {

template <int WP>
cudaError_t launch_attention(const AttnMaps& maps, const AttnArgs& args, int ctas, bool fused, cudaStream_t stream) {
  const bool bf16 = args.in_fmt == kBF16;
  auto kern = fused ? (bf16 ? relpos_attn_kernel<WP, true, true> : relpos_attn_kernel<WP, true, false>)
                    : (bf16 ? relpos_attn_kernel<WP, false, true> : relpos_attn_kernel<WP, false, false>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, AttnSmem::kAlloc);
  if (e != cudaSuccess) return e;
  const unsigned grid = static_cast<unsigned>(ctas);
  kern<<<grid, kAttnThreads, AttnSmem::kAlloc, stream>>>(maps.q, maps.k, maps.v, maps.th, maps.tw, args);
  return cudaGetLastError();
}

}  // namespace dera
