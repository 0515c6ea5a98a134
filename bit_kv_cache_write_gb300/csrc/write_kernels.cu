// Write / demote kernel on CUDA cores: rotate -> clip -> group scale/zero ->
// 2-bit quantize -> pack into the paged INT2 cache.
//
// Method: QbitAI article on OSCAR, serving-pipeline part. The demoted token is
// rotated, clipped, quantized and packed, four codes per byte, with a scale and
// zero point per group. R and the clip thresholds are the fixed per-layer
// calibration (section "OSCAR aligns the rotation with attention"; arXiv
// 2605.17757 abstracts).
//
// One CTA owns one (KV head, K|V) pair and a contiguous range of tokens, and
// keeps that pair's R (d x d fp32) in shared memory. Each warp rotates kTok
// tokens at a time: lane l produces rotated channels [CPL*l, CPL*l + CPL). That
// keeps a quantization group on an aligned run of G/CPL lanes, so group min/max
// is a butterfly shuffle. Codes are packed with one warp OR-reduction per 32-bit
// word of the row. For a handful of tokens (the demote of a few sequences) each
// CTA takes one token and its four warps each sum a quarter of the d terms.

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cfloat>
#include <cstdlib>
#include <cstring>

#include "layout.cuh"
#include "oscar_internal.h"

namespace oscar {
namespace {

constexpr int kWarps = 4;
constexpr long long kWaitCycles = 2000000000LL;   // give up on the R copy after ~1 s
constexpr int kSplitTokens = 8;                    // up to this many tokens: one CTA per token

// Error-free transformations on fp32 (explicit _rn intrinsics: no contraction).
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
    s = __fadd_rn(a, b);
    const float bp = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bp)), __fsub_rn(b, bp));
}

// x . R[:, c] rounded once to fp32 (double-float accumulation, ~48-bit), computed by the
// whole warp: lane l takes terms l, l+32, ...; the result is lane 0's, broadcast.
template <int D>
__device__ float exact_dot_warp(const float* x, const float* r, int c, int lane) {
    float hi = 0.0f, lo = 0.0f;
#pragma unroll
    for (int k = 0; k < D / 32; ++k) {
        const int i = lane + 32 * k;
        const float a = x[i], b = r[i * D + c];
        const float p = __fmul_rn(a, b);
        const float pe = __fmaf_rn(a, b, -p);
        float s, e;
        two_sum(hi, p, s, e);
        hi = s;
        lo = __fadd_rn(lo, __fadd_rn(pe, e));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float h2 = __shfl_xor_sync(0xffffffffu, hi, o);
        const float l2 = __shfl_xor_sync(0xffffffffu, lo, o);
        float s, e;
        two_sum(hi, h2, s, e);
        hi = s;
        lo = __fadd_rn(__fadd_rn(lo, l2), e);
    }
    return __shfl_sync(0xffffffffu, __fadd_rn(hi, lo), 0);
}

__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t phase) {
    uint32_t ok;
    asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
                 : "=r"(ok) : "r"(bar), "r"(phase) : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t phase) {
    if (mbar_test(bar, phase)) return true;
    const long long t0 = clock64();
    while (!mbar_test(bar, phase))
        if (clock64() - t0 > kWaitCycles) return false;
    return true;
}

// Clip, group scale/zero (exact recompute of the candidate channels where the fp32 rotation error could
// move the stored zero or scale by more than one fp16 step), 2-bit codes and the packed row of token tok,
// whose fp32 rotation a[j] (channels CPL * lane + j) this warp holds; x is the token's row and r_s its R.
template <int D, int G>
__device__ __forceinline__ void finish_row(const float (&a)[D / 32], int tok, const float* x, const float* r_s,
                                           const float (&thr)[D / 32], const int (&off)[D / 32], int kind, int head,
                                           int h_kv, const int64_t* __restrict__ dst_slots, int64_t bf16_pages,
                                           const int64_t* __restrict__ src_slots, uint8_t* __restrict__ int2_pool,
                                           int64_t int2_pages, int debug, DebugWord* dbg, int lane) {
    constexpr int CPL = D / 32;             // rotated channels per lane
    constexpr int LPG = G / CPL;            // lanes per group
    constexpr int WORDS = D / 16;           // 32-bit words per code row
    using GE = Geo<D, G>;
    const int64_t slot = dst_slots[tok];
    const int64_t pg = slot / kPage;
    bool ok = !(slot < 0 || pg >= int2_pages);
    if (!ok && debug && lane == 0) record_error(&dbg->kind, &dbg->index, 1, slot);
    if (src_slots && debug) {
        const int64_t s = src_slots[tok];
        if (s < 0 || s / kPage >= bf16_pages) ok = false;
    }
    if (!ok) return;     // warp-uniform

    // rigorous bound on the fp32 rotation error of every channel of this token:
    // |fl(x.R_c) - x.R_c| <= gamma_D * sum_i |x_i R_ic| <= gamma_D * ||x||_2 (R orthogonal)
    float sq = 0.0f;
#pragma unroll
    for (int j = 0; j < CPL; ++j) sq = fmaf(x[lane + 32 * j], x[lane + 32 * j], sq);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
    const float err = 1.01f * (float)(D + 1) * 0x1p-24f * sqrtf(sq * 1.001f);

    float xh[CPL];
    float mn = FLT_MAX, mx = -FLT_MAX;
#pragma unroll
    for (int j = 0; j < CPL; ++j) {
        xh[j] = fminf(fmaxf(a[j], -thr[j]), thr[j]);
        mn = fminf(mn, xh[j]);
        mx = fmaxf(mx, xh[j]);
    }
#pragma unroll
    for (int o = 1; o < LPG; o <<= 1) {
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    // The stored zero (fp16 mn) and scale (fp16 (mx-mn)/3) can only be off by more than
    // one fp16 ulp when |mn| or the range is within ~2^12 error bounds. Then every channel
    // that may hold the group min (max) is recomputed exactly and the stats are redone.
    {
        const float r0 = mx - mn;
        const bool need_min = fabsf(mn) < 4096.0f * err || r0 < 8192.0f * err;
        const bool need_max = r0 < 8192.0f * err;
        uint32_t cand = 0u;
#pragma unroll
        for (int j = 0; j < CPL; ++j)
            if ((need_min && xh[j] <= mn + 2.0f * err) || (need_max && xh[j] >= mx - 2.0f * err))
                cand |= 1u << j;
        uint32_t lanes = __ballot_sync(0xffffffffu, cand != 0u);
        if (lanes) {
            while (lanes) {
                const int src = __ffs(lanes) - 1;
                lanes &= lanes - 1;
                uint32_t cm = __shfl_sync(0xffffffffu, cand, src);
                while (cm) {
                    const int j = __ffs(cm) - 1;
                    cm &= cm - 1;
                    const float ex = exact_dot_warp<D>(x, r_s, CPL * src + j, lane);
#pragma unroll
                    for (int jj = 0; jj < CPL; ++jj)
                        if (lane == src && jj == j) xh[jj] = fminf(fmaxf(ex, -thr[jj]), thr[jj]);
                }
            }
            mn = FLT_MAX;
            mx = -FLT_MAX;
#pragma unroll
            for (int j = 0; j < CPL; ++j) { mn = fminf(mn, xh[j]); mx = fmaxf(mx, xh[j]); }
#pragma unroll
            for (int o = 1; o < LPG; o <<= 1) {
                mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            }
        }
    }
    const float rng = __fsub_rn(mx, mn);
    const bool degenerate = !(rng >= FLT_MIN);
    const float inv = __fdiv_rn(3.0f, degenerate ? 1.0f : rng);

    uint32_t contrib[WORDS];
#pragma unroll
    for (int w = 0; w < WORDS; ++w) contrib[w] = 0u;
#pragma unroll
    for (int j = 0; j < CPL; ++j) {
        const float u = __fmul_rn(__fsub_rn(xh[j], mn), inv);
        int code = degenerate ? 0 : (int)rintf(u);
        code = min(max(code, 0), 3);
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
    if (lane < WORDS)
        reinterpret_cast<uint32_t*>(seg + row * GE::kCodeRow)[lane] = mine;
    if (lane % LPG == 0) {
        const int grp = lane / LPG;
        __half2 sz;
        sz.x = __float2half_rn(__fdiv_rn(rng, 3.0f));
        sz.y = __float2half_rn(mn);
        reinterpret_cast<__half2*>(seg + GE::kCodeBytes)[row * GE::kGroups + grp] = sz;
    }
}

// kTok: tokens each warp rotates per iteration (register blocking over R); 8 for bulk writes,
// 1 when there are few tokens (demotes of a batch). kTok = 0: one token per CTA, its d-term sums split
// over the four warps (a quarter of R's rows each), then warp 0 finishes the row: the latency-bound
// demote of a handful of sequences.
template <int D, int G, int kTok>
__global__ void __launch_bounds__(kWarps * 32)
write_kernel(const float* __restrict__ r_all, const float* __restrict__ t_all,
             const __nv_bfloat16* __restrict__ k_in, const __nv_bfloat16* __restrict__ v_in,
             const int64_t* __restrict__ dst_slots, int n, int h_kv,
             const __nv_bfloat16* __restrict__ bf16_pool, int64_t bf16_pages,
             const int64_t* __restrict__ src_slots,
             uint8_t* __restrict__ int2_pool, int64_t int2_pages,
             int debug, DebugWord* dbg) {
    constexpr int CPL = D / 32;             // rotated channels per lane

    extern __shared__ __align__(16) float smem[];
    float* r_s = smem;                                  // [D][D]
    float* x_s = smem + D * D;                          // [kWarps][kTok][D]; kTok = 0: x [D], partials [kWarps][D]

    const int head = blockIdx.y;
    const int kind = blockIdx.z;                        // 0 = K, 1 = V
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

    // R of this (head, K|V) -> shared memory with one bulk async copy (bounded wait)
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

    // programmatic dependent launch: R and T are calibration data, staged above while the preceding
    // grid may still run; wait for it before touching token data or the pools (a no-op without the
    // launch attribute), then let the next grid start its prologue
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    // bit offset of each of this lane's channels inside the packed row
    int off[CPL];
#pragma unroll
    for (int j = 0; j < CPL; ++j) {
        const int c = CPL * lane + j;
        off[j] = kind == 0 ? k_bit_offset(c, D) : v_bit_offset(c, D);
    }
    if (!__all_sync(0xffffffffu, mbar_wait(rbar_s, 0))) {
        if (lane == 0) record_error(&dbg->kind, &dbg->index, 4, -1);
        (void)mbar_wait(rbar_s, 0);      // bounded again: the copy may still be in flight
        return;
    }

    if constexpr (kTok == 0) {
        // one token per CTA (blockIdx.x < n): stage it, four partial rotations, warp 0 finishes
        const int tok = blockIdx.x;
        float* xr = x_s;
        float* part = x_s + D;
        const __nv_bfloat16* src = nullptr;
        if (src_slots) {
            const int64_t sl = src_slots[tok];
            const int64_t pg = sl / kPage;
            if (debug && (sl < 0 || pg >= bf16_pages)) {
                if (threadIdx.x == 0) record_error(&dbg->kind, &dbg->index, 1, sl);
            } else {
                src = bf16_pool + ((((size_t)pg * h_kv + head) * 2 + kind) * kPage + (sl % kPage)) * D;
            }
        } else {
            src = (kind == 0 ? k_in : v_in) + ((size_t)tok * h_kv + head) * D;
        }
        for (int c = threadIdx.x; c < D; c += blockDim.x) xr[c] = src ? __bfloat162float(src[c]) : 0.0f;
        __syncthreads();
        constexpr int QD = D / kWarps;
        float a[CPL];
#pragma unroll
        for (int j = 0; j < CPL; ++j) a[j] = 0.0f;
#pragma unroll 4
        for (int i = warp * QD; i < (warp + 1) * QD; ++i) {
            float rv[CPL];
            if constexpr (CPL == 4) {
                const float4 r4 = *reinterpret_cast<const float4*>(r_s + i * D + 4 * lane);
                rv[0] = r4.x; rv[1] = r4.y; rv[2] = r4.z; rv[3] = r4.w;
            } else {
                const float2 r2 = *reinterpret_cast<const float2*>(r_s + i * D + 2 * lane);
                rv[0] = r2.x; rv[1] = r2.y;
            }
            const float xv = xr[i];
#pragma unroll
            for (int j = 0; j < CPL; ++j) a[j] = fmaf(xv, rv[j], a[j]);
        }
#pragma unroll
        for (int j = 0; j < CPL; ++j) part[warp * D + CPL * lane + j] = a[j];
        __syncthreads();
        if (warp == 0) {
#pragma unroll
            for (int j = 0; j < CPL; ++j) {
                const int c = CPL * lane + j;
                a[j] = __fadd_rn(__fadd_rn(part[c], part[D + c]), __fadd_rn(part[2 * D + c], part[3 * D + c]));
            }
            finish_row<D, G>(a, tok, xr, r_s, thr, off, kind, head, h_kv, dst_slots, bf16_pages, src_slots,
                             int2_pool, int2_pages, debug, dbg, lane);
        }
        return;
    }

    const int per_cta = (n + gridDim.x - 1) / gridDim.x;
    const int t_begin = blockIdx.x * per_cta;
    const int t_end = min(n, t_begin + per_cta);
    constexpr int KT = kTok > 0 ? kTok : 1;       // the one-token path returned above
    float* xw = x_s + warp * KT * D;

    for (int base = t_begin + warp * KT; base < t_end; base += kWarps * KT) {
        const int cnt = min(KT, t_end - base);
        // stage the kTok input rows (bf16 -> fp32) in this warp's smem tile
        for (int t = 0; t < KT; ++t) {
            const __nv_bfloat16* src = nullptr;
            if (t < cnt) {
                const int tok = base + t;
                if (src_slots) {
                    const int64_t s = src_slots[tok];
                    const int64_t pg = s / kPage;
                    if (debug && (s < 0 || pg >= bf16_pages)) {
                        if (lane == 0) record_error(&dbg->kind, &dbg->index, 1, s);
                    } else {
                        src = bf16_pool + ((((size_t)pg * h_kv + head) * 2 + kind) * kPage + (s % kPage)) * D;
                    }
                } else {
                    src = (kind == 0 ? k_in : v_in) + ((size_t)tok * h_kv + head) * D;
                }
            }
#pragma unroll
            for (int j = 0; j < CPL; ++j)
                xw[t * D + lane + 32 * j] = src ? __bfloat162float(src[lane + 32 * j]) : 0.0f;
        }
        __syncwarp();

        float acc[KT][CPL];
#pragma unroll
        for (int t = 0; t < KT; ++t)
#pragma unroll
            for (int j = 0; j < CPL; ++j) acc[t][j] = 0.0f;

#pragma unroll 4
        for (int i = 0; i < D; ++i) {
            float rv[CPL];
            if constexpr (CPL == 4) {
                const float4 r4 = *reinterpret_cast<const float4*>(r_s + i * D + 4 * lane);
                rv[0] = r4.x; rv[1] = r4.y; rv[2] = r4.z; rv[3] = r4.w;
            } else {
                const float2 r2 = *reinterpret_cast<const float2*>(r_s + i * D + 2 * lane);
                rv[0] = r2.x; rv[1] = r2.y;
            }
#pragma unroll
            for (int t = 0; t < KT; ++t) {
                const float xv = xw[t * D + i];
#pragma unroll
                for (int j = 0; j < CPL; ++j) acc[t][j] = fmaf(xv, rv[j], acc[t][j]);
            }
        }

#pragma unroll
        for (int t = 0; t < KT; ++t) {
            if (t >= cnt) break;
            finish_row<D, G>(acc[t], base + t, xw + t * D, r_s, thr, off, kind, head, h_kv, dst_slots, bf16_pages,
                             src_slots, int2_pool, int2_pages, debug, dbg, lane);
        }
        __syncwarp();
    }
}

template <int D, int G, int kTok>
cudaError_t launch_write_tok(const Shape& s, const LayerParams& p, int num_sms,
                             const void* k, const void* v, const int64_t* slots, int n,
                             const void* bf16_pool, int64_t bf16_pages, const int64_t* src_slots,
                             void* int2_pool, int64_t int2_pages, DebugWord* dbg, Profiler* prof,
                             cudaStream_t st) {
    const size_t smem = (size_t)(D * D + (kTok == 0 ? (kWarps + 1) * D : kWarps * kTok * D)) * sizeof(float);
    auto kern = write_kernel<D, G, kTok>;
    // Opt in to the large dynamic shared memory once per device (outside any stream capture: the
    // first call of a shape on a device happens before a caller can capture it).
    const cudaError_t attr = smem_opt_in<write_kernel<D, G, kTok>>(smem);
    if (attr != cudaSuccess) return attr;
    // K and V rotations/thresholds sit back to back: r_k then r_v, t_k then t_v.
    const int pairs = s.h_kv * 2;
    const int per_cta = kTok == 0 ? 1 : kWarps * kTok;
    const int max_gx = (n + per_cta - 1) / per_cta;
    int gx = kTok <= 1 ? max_gx : (2 * num_sms + pairs - 1) / pairs;
    gx = gx < 1 ? 1 : (gx > max_gx ? max_gx : gx);
    dim3 grid(gx, s.h_kv, 2);
    ProfScope ps(prof, OSCAR_KERNEL_WRITE, st);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kWarps * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute la[1];
    la[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    la[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = la;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, p.r_k, p.t_k, static_cast<const __nv_bfloat16*>(k),
                              static_cast<const __nv_bfloat16*>(v), slots, n, s.h_kv,
                              static_cast<const __nv_bfloat16*>(bf16_pool), bf16_pages, src_slots,
                              static_cast<uint8_t*>(int2_pool), int2_pages, s.debug, dbg);
}

template <int D, int G>
cudaError_t launch_write_t(const Shape& s, const LayerParams& p, int num_sms,
                           const void* k, const void* v, const int64_t* slots, int n,
                           const void* bf16_pool, int64_t bf16_pages, const int64_t* src_slots,
                           void* int2_pool, int64_t int2_pages, DebugWord* dbg, Profiler* prof,
                           cudaStream_t st) {
    // a handful of tokens: one per CTA over four warps; few: one per warp, one CTA per 4 tokens
    // (latency); many: 8 per warp (R reuse)
    if (n <= kSplitTokens)
        return launch_write_tok<D, G, 0>(s, p, num_sms, k, v, slots, n, bf16_pool, bf16_pages, src_slots,
                                         int2_pool, int2_pages, dbg, prof, st);
    if (n <= 64 * num_sms)
        return launch_write_tok<D, G, 1>(s, p, num_sms, k, v, slots, n, bf16_pool, bf16_pages, src_slots,
                                         int2_pool, int2_pages, dbg, prof, st);
    return launch_write_tok<D, G, 8>(s, p, num_sms, k, v, slots, n, bf16_pool, bf16_pages, src_slots,
                                     int2_pool, int2_pages, dbg, prof, st);
}

__global__ void transpose_kernel(const float* __restrict__ src, float* __restrict__ dst, int d) {
    __shared__ float tile[32][33];
    const size_t mat = (size_t)blockIdx.z * d * d;
    const int bx = blockIdx.x * 32, by = blockIdx.y * 32;
    for (int j = threadIdx.y; j < 32; j += blockDim.y)
        tile[j][threadIdx.x] = src[mat + (size_t)(by + j) * d + bx + threadIdx.x];
    __syncthreads();
    for (int j = threadIdx.y; j < 32; j += blockDim.y)
        dst[mat + (size_t)(bx + j) * d + by + threadIdx.x] = tile[threadIdx.x][j];
}

}  // namespace

cudaError_t launch_write(const Shape& s, const LayerParams& p, int num_sms,
                         const void* k, const void* v, const int64_t* slots, int n,
                         const void* bf16_pool, int64_t bf16_pages, const int64_t* src_slots,
                         void* int2_pool, int64_t int2_pages, DebugWord* dbg, Profiler* prof,
                         cudaStream_t st) {
    // many tokens straight from K/V rows: the tcgen05 kernel (OSCAR_WRITE_PATH=cuda keeps the
    // CUDA-core kernel, for comparisons)
    if (s.codebook == OSCAR_CODEBOOK_LLOYD_MAX)
        return launch_write_lm(s, p, num_sms, k, v, slots, n, bf16_pool, bf16_pages, src_slots, int2_pool,
                               int2_pages, dbg, prof, st);
    const char* path = std::getenv("OSCAR_WRITE_PATH");
    const bool force_cuda = path && std::strcmp(path, "cuda") == 0;
    if (!src_slots && !force_cuda && write_tc_eligible(s, k, v, int2_pool, n))
        return launch_write_tc(s, p, num_sms, k, v, slots, n, int2_pool, int2_pages, dbg, prof, st);
#define OSCAR_WRITE_CASE(D_, G_)                                                              \
    if (s.d == D_ && s.group == G_)                                                           \
        return launch_write_t<D_, G_>(s, p, num_sms, k, v, slots, n, bf16_pool, bf16_pages,   \
                                      src_slots, int2_pool, int2_pages, dbg, prof, st);
    OSCAR_WRITE_CASE(64, 32)
    OSCAR_WRITE_CASE(64, 64)
    OSCAR_WRITE_CASE(128, 32)
    OSCAR_WRITE_CASE(128, 64)
    OSCAR_WRITE_CASE(128, 128)
#undef OSCAR_WRITE_CASE
    return cudaErrorInvalidValue;
}

cudaError_t launch_transpose(const float* src, float* dst, int h, int d, cudaStream_t st) {
    dim3 grid(d / 32, d / 32, h);
    transpose_kernel<<<grid, dim3(32, 8), 0, st>>>(src, dst, d);
    return cudaGetLastError();
}

}  // namespace oscar
