// Attention kernels for key tiles padded to 48 grid columns.
#include "attention_inst.cuh"

namespace dera {
template cudaError_t launch_attention<48>(const AttnMaps&, const AttnArgs&, int, bool, cudaStream_t);
}  // namespace dera
