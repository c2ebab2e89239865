// Definition of launch_attention<WP>; included by one .cu per padded width.
#pragma once
#include <atomic>

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
  // The kernel's setmaxnreg split needs the block to launch with at least
  // kLaunchRegs registers per thread; a build that compiled to fewer is
  // refused rather than launched into a wait that never ends.
  static std::atomic<int> regs_ok[2][2];  // 0 unknown, 1 fits, -1 refused
  std::atomic<int>& ok = regs_ok[fused][bf16];
  if (ok.load(std::memory_order_relaxed) == 0) {
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, kern);
    if (e != cudaSuccess) return e;
    ok.store(fa.numRegs * kAttnThreads >= kRegsCtl * 128 + kRegsSmx * 256 ? 1 : -1, std::memory_order_relaxed);
  }
  if (ok.load(std::memory_order_relaxed) < 0) return cudaErrorInvalidKernelImage;
  const unsigned grid = static_cast<unsigned>(ctas);
  kern<<<grid, kAttnThreads, AttnSmem::kAlloc, stream>>>(maps.q, maps.k, maps.v, maps.th, maps.tw, args);
  return cudaGetLastError();
}

}  // namespace dera
