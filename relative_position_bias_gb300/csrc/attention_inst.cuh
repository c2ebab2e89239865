// Definition of launch_attention<WP>; included by one .cu per padded width.
// Each width instantiates the kernel for head_dim 64 and 128, fused or not,
// bf16 or fp16 inputs.
#pragma once
#include <atomic>

#include "attention.cuh"
#include "launch.cuh"

namespace dera {

template <int WP, int D>
cudaError_t launch_attention_d(const AttnMaps& maps, const AttnArgs& args, int ctas, bool fused,
                               cudaStream_t stream) {
  using SM = AttnSmem<D, FwdKeyTile<WP, D>::BN>;
  const bool bf16 = args.in_fmt == kBF16;
  auto kern = fused ? (bf16 ? relpos_attn_kernel<WP, true, true, D> : relpos_attn_kernel<WP, true, false, D>)
                    : (bf16 ? relpos_attn_kernel<WP, false, true, D> : relpos_attn_kernel<WP, false, false, D>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SM::kAlloc);
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
  kern<<<grid, kAttnThreads, SM::kAlloc, stream>>>(maps.q, maps.k, maps.v, maps.th, maps.tw, args);
  return cudaGetLastError();
}

template <int WP>
cudaError_t launch_attention(const AttnMaps& maps, const AttnArgs& args, int ctas, bool fused, int head_dim,
                             cudaStream_t stream) {
  return head_dim == 128 ? launch_attention_d<WP, 128>(maps, args, ctas, fused, stream)
                         : launch_attention_d<WP, 64>(maps, args, ctas, fused, stream);
}

}  // namespace dera
