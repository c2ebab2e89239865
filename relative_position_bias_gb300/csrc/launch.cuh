// Host-side launchers of the kernel templates; each padded width WP is
// instantiated in its own translation unit so the build compiles in parallel.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace dera {

struct AttnMaps {
  CUtensorMap q, k, v, th, tw;
};

template <int WP>
cudaError_t launch_attention(const AttnMaps& maps, const AttnArgs& args, int ctas, bool fused, int head_dim,
                             cudaStream_t stream);

cudaError_t launch_project(const CUtensorMap& q, const CUtensorMap& th, const CUtensorMap& tw,
                           const ProjArgs& args, int in_fmt, int head_dim, int max_ctas, cudaStream_t stream);

cudaError_t launch_wait_selftest(int* status, long long budget, cudaStream_t stream);

struct BwdMaps {
  CUtensorMap q, dout, k, v, th, tw;
};

// The backward's attention kernels and its table reduction for head_dim 64, in
// stream order; the compact rel_h, rel_w in args must already be written.
cudaError_t launch_backward(const BwdMaps& maps, const BwdArgs& args, int WP, cudaStream_t stream);

}  // namespace dera
