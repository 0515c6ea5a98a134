// Split-kernel instantiations for D = 128, Lloyd-Max codebook, groups 32, 64 and 128: the INT2 split-K decode of
// decode_device.cuh, launched by decode_kernels.cu through the functions below.

#include "decode_device.cuh"

namespace oscar {

cudaError_t split_launch_lm128(int group, int gq, const SplitArgs& a, int batch, cudaStream_t st) {
    if (group == 32) return dispatch_gq<128, 32, OSCAR_CODEBOOK_LLOYD_MAX>(gq, a, batch, st);
    if (group == 64) return dispatch_gq<128, 64, OSCAR_CODEBOOK_LLOYD_MAX>(gq, a, batch, st);
    if (group == 128) return dispatch_gq<128, 128, OSCAR_CODEBOOK_LLOYD_MAX>(gq, a, batch, st);
    return cudaErrorInvalidValue;
}
int split_occupancy_lm128(int group, int gq) {
    if (group == 32) return occupancy_gq<128, 32, OSCAR_CODEBOOK_LLOYD_MAX>(gq);
    if (group == 64) return occupancy_gq<128, 64, OSCAR_CODEBOOK_LLOYD_MAX>(gq);
    return occupancy_gq<128, 128, OSCAR_CODEBOOK_LLOYD_MAX>(gq);
}

}  // namespace oscar
