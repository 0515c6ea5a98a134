// Write / demote with the Lloyd-Max codebook: rotate -> clip -> group mean and standard deviation
// -> nearest of four levels -> pack into the paged INT2 cache.
//
// Method: QbitAI article on OSCAR. Rotation and clipping as in the serving pipeline (the oldest
// recent token is rotated, clipped, quantized and packed, four codes per byte); the closing part of
// the article pairs the rotation with "a stronger Lloyd-Max codebook". The stored codebook is the
// Gaussian Lloyd-Max quantizer with its levels rounded to delta * (-27, -8, 8, 27), delta = y_1 / 8,
// y_1 the inner level: each group is normalised by its own mean mu and standard deviation sigma, the
// code is the nearest level (midpoints delta * (-17.5, 0, 17.5), ties to the lower level), and the
// (scale, zero) pair holds (fp16(sigma * delta), fp16(mu)). A group with sigma = 0 stores scale 0 and
// codes 0. Dequant: zero + scale * l(code).
//
// Precision: the stored mu and sigma must round to the same fp16 values as the exact statistics
// (within one ulp) even where mu is far smaller than the row's norm, so the rotation is summed as a
// double-float (error ~2^-44 relative) and rounded once to fp32, and the statistics and the code
// decision are fp64.
//
// One warp per (token, KV head, K|V): lane l owns rotated channels [CPL*l, CPL*l + CPL); a group is an
// aligned run of G/CPL lanes, reduced with butterfly shuffles.

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cfloat>

#include "layout.cuh"
#include "oscar_internal.h"

namespace oscar {
namespace {

constexpr int kWarpsLm = 4;
constexpr long long kWaitCyclesLm = 2000000000LL;   // give up on the R copy after ~1 s
// delta = y_1 / 8 for the 4-level Gaussian Lloyd-Max quantizer (y_1 = 0.45278...), as a double
constexpr double kDelta = 0.05659750432956155;

__device__ __forceinline__ void two_sum_lm(float a, float b, float& s, float& e) {
    s = __fadd_rn(a, b);
    const float bp = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bp)), __fsub_rn(b, bp));
}

__device__ __forceinline__ bool mbar_wait_lm(uint32_t bar, uint32_t phase) {
    const long long t0 = clock64();
    while (true) {
        uint32_t ok;
        asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
                     : "=r"(ok) : "r"(bar), "r"(phase) : "memory");
        if (ok) return true;
        if (clock64() - t0 > kWaitCyclesLm) return false;
    }
}

template <int D, int G>
__global__ void __launch_bounds__(kWarpsLm * 32)
write_lm_kernel(const float* __restrict__ r_all, const float* __restrict__ t_all,
                const __nv_bfloat16* __restrict__ k_in, const __nv_bfloat16* __restrict__ v_in,
                const int64_t* __restrict__ dst_slots, int n, int h_kv,
                const __nv_bfloat16* __restrict__ bf16_pool, int64_t bf16_pages,
                const int64_t* __restrict__ src_slots,
                uint8_t* __restrict__ int2_pool, int64_t int2_pages, int debug, DebugWord* dbg) {
    constexpr int CPL = D / 32;             // rotated channels per lane
    constexpr int LPG = G / CPL;            // lanes per group
    constexpr int WORDS = D / 16;           // 32-bit words per code row
    using GE = Geo<D, G>;

    extern __shared__ __align__(16) float smem[];
    float* r_s = smem;                                  // [D][D]
    float* x_s = smem + D * D;                          // [kWarpsLm][D]

    const int head = blockIdx.y;
    const int kind = blockIdx.z;                        // 0 = K, 1 = V
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    __shared__ __align__(8) uint64_t rbar;
    const float* r_g = r_all + ((size_t)kind * h_kv + head) * D * D;
    const uint32_t rbar_s = (uint32_t)__cvta_generic_to_shared(&rbar);
    if (threadIdx.x == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" :: "r"(rbar_s) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(rbar_s), "r"(D * D * 4) : "memory");
        asm volatile("cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                     :: "r"((uint32_t)__cvta_generic_to_shared(r_s)), "l"(r_g), "r"(D * D * 4), "r"(rbar_s) : "memory");
    }
    __syncthreads();
    float thr[CPL];
    const float* t_g = t_all + ((size_t)kind * h_kv + head) * D;
#pragma unroll
    for (int j = 0; j < CPL; ++j) thr[j] = __ldg(t_g + CPL * lane + j);
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    int off[CPL];
#pragma unroll
    for (int j = 0; j < CPL; ++j) {
        const int c = CPL * lane + j;
        off[j] = kind == 0 ? k_bit_offset(c, D) : v_bit_offset(c, D);
    }
    if (!__all_sync(0xffffffffu, mbar_wait_lm(rbar_s, 0))) {
        if (lane == 0) record_error(&dbg->kind, &dbg->index, 4, -1);
        (void)mbar_wait_lm(rbar_s, 0);      // bounded again: the copy may still be in flight
        return;
    }
    // code decision cuts: midpoints of the levels delta * (-27, -8, 8, 27), formed level by level
    const double l0 = kDelta * -27.0, l1 = kDelta * -8.0, l2 = kDelta * 8.0, l3 = kDelta * 27.0;
    const double cut0 = 0.5 * (l0 + l1), cut1 = 0.5 * (l1 + l2), cut2 = 0.5 * (l2 + l3);
    float* xw = x_s + warp * D;

    for (int tok = blockIdx.x * kWarpsLm + warp; tok < n; tok += gridDim.x * kWarpsLm) {
        const __nv_bfloat16* src = nullptr;
        if (src_slots) {
            const int64_t s = src_slots[tok];
            const int64_t pg = s / kPage;
            if (s < 0 || pg >= bf16_pages) {
                if (debug && lane == 0) record_error(&dbg->kind, &dbg->index, 1, s);
            } else {
                src = bf16_pool + ((((size_t)pg * h_kv + head) * 2 + kind) * kPage + (s % kPage)) * D;
            }
        } else {
            src = (kind == 0 ? k_in : v_in) + ((size_t)tok * h_kv + head) * D;
        }
        const int64_t slot = dst_slots[tok];
        const int64_t pg = slot / kPage;
        const bool slot_ok = !(slot < 0 || pg >= int2_pages);
        if (!slot_ok && debug && lane == 0) record_error(&dbg->kind, &dbg->index, 1, slot);
        if (!src || !slot_ok) continue;      // warp-uniform
#pragma unroll
        for (int j = 0; j < CPL; ++j) xw[lane + 32 * j] = __bfloat162float(src[lane + 32 * j]);
        __syncwarp();
        // x . R[:, c] for this lane's channels as a double-float, rounded once to fp32
        float hi[CPL], lo[CPL];
#pragma unroll
        for (int j = 0; j < CPL; ++j) { hi[j] = 0.0f; lo[j] = 0.0f; }
#pragma unroll 2
        for (int i = 0; i < D; ++i) {
            const float xv = xw[i];
            float rv[CPL];
            if constexpr (CPL == 4) {
                const float4 r4 = *reinterpret_cast<const float4*>(r_s + i * D + 4 * lane);
                rv[0] = r4.x; rv[1] = r4.y; rv[2] = r4.z; rv[3] = r4.w;
            } else {
                const float2 r2 = *reinterpret_cast<const float2*>(r_s + i * D + 2 * lane);
                rv[0] = r2.x; rv[1] = r2.y;
            }
#pragma unroll
            for (int j = 0; j < CPL; ++j) {
                const float p = __fmul_rn(xv, rv[j]);
                const float pe = __fmaf_rn(xv, rv[j], -p);
                float s, e;
                two_sum_lm(hi[j], p, s, e);
                hi[j] = s;
                lo[j] = __fadd_rn(lo[j], __fadd_rn(pe, e));
            }
        }
        double xh[CPL];
        double s1 = 0.0;
#pragma unroll
        for (int j = 0; j < CPL; ++j) {
            const float xr = __fadd_rn(hi[j], lo[j]);
            xh[j] = (double)fminf(fmaxf(xr, -thr[j]), thr[j]);
            s1 += xh[j];
        }
#pragma unroll
        for (int o = 1; o < LPG; o <<= 1) s1 += __shfl_xor_sync(0xffffffffu, s1, o);
        const double mu = s1 / (double)G;
        double s2 = 0.0;
#pragma unroll
        for (int j = 0; j < CPL; ++j) s2 += (xh[j] - mu) * (xh[j] - mu);
#pragma unroll
        for (int o = 1; o < LPG; o <<= 1) s2 += __shfl_xor_sync(0xffffffffu, s2, o);
        const double sigma = sqrt(s2 / (double)G);
        const bool flat = !(sigma > 0.0);

        uint32_t contrib[WORDS];
#pragma unroll
        for (int w = 0; w < WORDS; ++w) contrib[w] = 0u;
#pragma unroll
        for (int j = 0; j < CPL; ++j) {
            const double z = (xh[j] - mu) / (flat ? 1.0 : sigma);
            const int code = flat ? 0 : (int)(z > cut0) + (int)(z > cut1) + (int)(z > cut2);
#pragma unroll
            for (int w = 0; w < WORDS; ++w)
                if ((off[j] >> 5) == w) contrib[w] |= (uint32_t)code << (off[j] & 31);
        }
        uint32_t mine = 0u;
#pragma unroll
        for (int w = 0; w < WORDS; ++w) {
            const uint32_t r = __reduce_or_sync(0xffffffffu, contrib[w]);
            if (lane == w) mine = r;
        }
        uint8_t* seg = int2_pool + ((size_t)pg * h_kv + head) * GE::kBlock + (size_t)kind * GE::kSeg;
        const int row = (int)(slot % kPage);
        if (lane < WORDS) reinterpret_cast<uint32_t*>(seg + row * GE::kCodeRow)[lane] = mine;
        if (lane % LPG == 0) {
            __half2 sz;
            sz.x = __double2half(flat ? 0.0 : sigma * kDelta);
            sz.y = __double2half(mu);
            reinterpret_cast<__half2*>(seg + GE::kCodeBytes)[row * GE::kGroups + lane / LPG] = sz;
        }
        __syncwarp();
    }
}

template <int D, int G>
cudaError_t launch_lm(const Shape& s, const LayerParams& p, int num_sms, const void* k, const void* v,
                      const int64_t* slots, int n, const void* bf16_pool, int64_t bf16_pages,
                      const int64_t* src_slots, void* int2_pool, int64_t int2_pages, DebugWord* dbg,
                      Profiler* prof, cudaStream_t st) {
    const size_t smem = (size_t)(D * D + kWarpsLm * D) * sizeof(float);
    const cudaError_t attr = smem_opt_in<write_lm_kernel<D, G>>(smem);
    if (attr != cudaSuccess) return attr;
    const int max_gx = (n + kWarpsLm - 1) / kWarpsLm;
    int gx = (4 * num_sms + 2 * s.h_kv - 1) / (2 * s.h_kv);
    gx = gx < 1 ? 1 : (gx > max_gx ? max_gx : gx);
    ProfScope ps(prof, OSCAR_KERNEL_WRITE, st);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(gx, s.h_kv, 2);
    cfg.blockDim = dim3(kWarpsLm * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute la[1];
    la[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    la[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = la;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, write_lm_kernel<D, G>, p.r_k, p.t_k, static_cast<const __nv_bfloat16*>(k),
                              static_cast<const __nv_bfloat16*>(v), slots, n, s.h_kv,
                              static_cast<const __nv_bfloat16*>(bf16_pool), bf16_pages, src_slots,
                              static_cast<uint8_t*>(int2_pool), int2_pages, s.debug, dbg);
}

}  // namespace

cudaError_t launch_write_lm(const Shape& s, const LayerParams& p, int num_sms, const void* k, const void* v,
                            const int64_t* slots, int n, const void* bf16_pool, int64_t bf16_pages,
                            const int64_t* src_slots, void* int2_pool, int64_t int2_pages, DebugWord* dbg,
                            Profiler* prof, cudaStream_t st) {
#define OSCAR_LM_CASE(D_, G_)                                                                      \
    if (s.d == D_ && s.group == G_)                                                                \
        return launch_lm<D_, G_>(s, p, num_sms, k, v, slots, n, bf16_pool, bf16_pages, src_slots,  \
                                 int2_pool, int2_pages, dbg, prof, st);
    OSCAR_LM_CASE(64, 32)
    OSCAR_LM_CASE(64, 64)
    OSCAR_LM_CASE(128, 32)
    OSCAR_LM_CASE(128, 64)
    OSCAR_LM_CASE(128, 128)
#undef OSCAR_LM_CASE
    return cudaErrorInvalidValue;
}

}  // namespace oscar
