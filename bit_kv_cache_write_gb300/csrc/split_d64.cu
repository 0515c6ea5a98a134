// Split-kernel instantiations for D = 64, both codebooks, groups 32 and 64: the INT2 split-K decode of
// decode_device.cuh, launched by decode_kernels.cu through the functions below.

#include "decode_device.cuh"

namespace oscar {

cudaError_t split_launch_d64(int group, int codebook, int gq, const SplitArgs& a, int batch, cudaStream_t st) {
    const bool lm = codebook == OSCAR_CODEBOOK_LLOYD_MAX;
    if (group == 32)
        return lm ? dispatch_gq<64, 32, OSCAR_CODEBOOK_LLOYD_MAX>(gq, a, batch, st)
                  : dispatch_gq<64, 32, OSCAR_CODEBOOK_UNIFORM>(gq, a, batch, st);
    if (group == 64)
        return lm ? dispatch_gq<64, 64, OSCAR_CODEBOOK_LLOYD_MAX>(gq, a, batch, st)
                  : dispatch_gq<64, 64, OSCAR_CODEBOOK_UNIFORM>(gq, a, batch, st);
    return cudaErrorInvalidValue;
}
int split_occupancy_d64(int group, int codebook, int gq) {
    const bool lm = codebook == OSCAR_CODEBOOK_LLOYD_MAX;
    if (group == 32) return lm ? occupancy_gq<64, 32, OSCAR_CODEBOOK_LLOYD_MAX>(gq) : occupancy_gq<64, 32, OSCAR_CODEBOOK_UNIFORM>(gq);
    return lm ? occupancy_gq<64, 64, OSCAR_CODEBOOK_LLOYD_MAX>(gq) : occupancy_gq<64, 64, OSCAR_CODEBOOK_UNIFORM>(gq);
}

}  // namespace oscar
