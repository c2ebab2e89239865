// Attention kernels for key tiles padded to 16 grid columns.
#include "attention_inst.cuh"

namespace dera {
template cudaError_t launch_attention<16>(const AttnMaps&, const AttnArgs&, int, bool, int, cudaStream_t);
}  // namespace dera
