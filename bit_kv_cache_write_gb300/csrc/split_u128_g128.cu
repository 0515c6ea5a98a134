// Split-kernel instantiations for D = 128, uniform codebook, group 128 (the bs1 and mixed-batch shapes): the INT2 split-K decode of
// decode_device.cuh, launched by decode_kernels.cu through the functions below.

#include "decode_device.cuh"

namespace oscar {

cudaError_t split_launch_u128_g128(int gq, const SplitArgs& a, int batch, cudaStream_t st) {
    return dispatch_gq<128, 128, OSCAR_CODEBOOK_UNIFORM>(gq, a, batch, st);
}
int split_occupancy_u128_g128(int gq) { return occupancy_gq<128, 128, OSCAR_CODEBOOK_UNIFORM>(gq); }

}  // namespace oscar
