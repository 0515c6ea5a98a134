// Split-kernel instantiations for D = 128, uniform codebook, groups 32 and 64: the INT2 split-K decode of
// decode_device.cuh, launched by decode_kernels.cu through the functions below.

#include "decode_device.cuh"

namespace oscar {

cudaError_t split_launch_u128_small_g(int group, int gq, const SplitArgs& a, int batch, cudaStream_t st) {
    if (group == 32) return dispatch_gq<128, 32, OSCAR_CODEBOOK_UNIFORM>(gq, a, batch, st);
    if (group == 64) return dispatch_gq<128, 64, OSCAR_CODEBOOK_UNIFORM>(gq, a, batch, st);
    return cudaErrorInvalidValue;
}
int split_occupancy_u128_small_g(int group, int gq) {
    return group == 32 ? occupancy_gq<128, 32, OSCAR_CODEBOOK_UNIFORM>(gq) : occupancy_gq<128, 64, OSCAR_CODEBOOK_UNIFORM>(gq);
}

}  // namespace oscar
