// Attention kernels for key tiles padded to 64 grid columns.
#include "attention_inst.cuh"

namespace dera {
template cudaError_t launch_attention<64>(const AttnMaps&, const AttnArgs&, int, bool, int, cudaStream_t);
}  // namespace dera
