// Paged decode attention over the three-segment cache: INT2 history and BF16 sink/recent.
//
// Method: QbitAI article on OSCAR, serving-pipeline part. At decode, the INT2
// part unpacks codes, dequantizes with scale/zero point and accumulates in
// floating point; a BF16 part covers sink and recent; an online-softmax merge
// combines the two. arXiv 2605.17757 abstracts: the kernels keep the paged
// KV-cache layout and prefix caching (block tables may share pages).
//
// Three launches per layer:
//   1. q_rotate:   q_rot = q @ R_k for every query head (fp32).
//   2. split:      one CTA per (split, KV head, sequence). INT2 splits stream
//                  pages of the history; BF16 splits cover sink + recent. Each
//                  writes a partial (m, l, acc[d]) per query head of the group,
//                  with m in log2 units.
//   3. merge:      combines the splits of each query head, un-rotates the INT2
//                  accumulator by R_v^T and normalises.
//
// Inside an INT2 split, the scale/zero identity
//   q . (code*s + z) = s * (q . code) + z * sum(q)
// keeps the dequant out of the inner product, per group.

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cfloat>
#include <cmath>

#include "layout.cuh"
#include "oscar_internal.h"

namespace oscar {
namespace {

constexpr int kWarps = 4;

__device__ __forceinline__ float fast_exp2(float x) { return exp2f(x); }

// Error-free transformations on fp32 (no contraction: explicit _rn intrinsics).
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
    s = __fadd_rn(a, b);
    const float bp = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bp)), __fsub_rn(b, bp));
}

__device__ __forceinline__ void two_prod(float a, float b, float& p, float& e) {
    p = __fmul_rn(a, b);
    e = __fmaf_rn(a, b, -p);
}

// Rotated query prepared for exact INT2 logits. Per query head:
//   q_rot = q @ R_k accumulated as an unevaluated sum hi + lo of two fp32 (about 48 bits);
//   qg = hi rounded to a grid of 2^(E-12) where max|hi| < 2^E, so sum_c code_c * qg_c over
//        d <= 128 channels (codes <= 3) is an integer multiple of the grid below 2^24: exact in fp32;
//   qr = (hi - qg) + lo, the residual (|qr| <= 2^(E-13));
//   qsum[g] = sum over group g of q_rot, as hi/lo fp32 from an fp64 reduction.
template <int D, int G>
__global__ void q_prep_kernel(const __nv_bfloat16* __restrict__ q, const float* __restrict__ r_k,
                              float* __restrict__ qg, float* __restrict__ qr, float* __restrict__ qsum,
                              int h_q, int g) {
    constexpr int NG = D / G;
    __shared__ float qs[D];
    __shared__ float wmax[D / 32];
    __shared__ double part[D];
    const int bh = blockIdx.x;
    const int kv = (bh % h_q) / g;
    const int c = threadIdx.x;
    qs[c] = __bfloat162float(q[(size_t)bh * D + c]);
    __syncthreads();
    const float* r = r_k + (size_t)kv * D * D;
    float hi = 0.0f, lo = 0.0f;
#pragma unroll 4
    for (int i = 0; i < D; ++i) {
        float p, e, s2, e2;
        two_prod(qs[i], __ldg(r + i * D + c), p, e);
        two_sum(hi, p, s2, e2);
        hi = s2;
        lo = __fadd_rn(lo, __fadd_rn(e, e2));
    }
    {
        float s2, e2;
        two_sum(hi, lo, s2, e2);
        hi = s2;
        lo = e2;
    }
    float m = fabsf(hi);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (c % 32 == 0) wmax[c / 32] = m;
    part[c] = (double)hi + (double)lo;
    __syncthreads();
    m = 0.0f;
#pragma unroll
    for (int w = 0; w < D / 32; ++w) m = fmaxf(m, wmax[w]);
    int ex = 0;
    frexpf(m, &ex);                                  // m < 2^ex
    const float grid_hi = m > 0.0f ? rintf(ldexpf(hi, 12 - ex)) : 0.0f;
    const float gq = ldexpf(grid_hi, ex - 12);
    qg[(size_t)bh * D + c] = gq;
    qr[(size_t)bh * D + c] = __fadd_rn(__fsub_rn(hi, gq), lo);
    if (c < NG) {
        double sum = 0.0;
        for (int j = 0; j < G; ++j) sum += part[c * G + j];
        const float sh = (float)sum;
        qsum[((size_t)bh * NG + c) * 2 + 0] = sh;
        qsum[((size_t)bh * NG + c) * 2 + 1] = (float)(sum - (double)sh);
    }
}

struct SplitArgs {
    const float* qg;              // [B][H_q][D] grid part of q_rot
    const float* qr;              // [B][H_q][D] residual of q_rot
    const float* qsum;            // [B][H_q][D/G][2] group sums of q_rot (hi, lo)
    const __nv_bfloat16* q;       // [B][H_q][D]
    const uint8_t* int2_pool; int64_t int2_pages;
    const int32_t* int2_tables; int int2_stride;
    const int32_t* hist_len; int max_hist;
    const __nv_bfloat16* bf16_pool; int64_t bf16_pages;
    const int32_t* bf16_tables; int bf16_stride;
    const int32_t* bf16_len; int max_bf16;
    float* partials;              // [B][H_q][S][D+2]
    int h_kv, int2_splits, pages_per_split, bf16_splits, bf16_pages_per_split, total_splits;
    float scale_log2, scale_log2_lo;   // sm_scale * log2(e) as hi + lo
    int debug; DebugWord* dbg;
};

template <int D, int GQ>
struct WarpState {
    float m[GQ], l[GQ];
};

// Online-softmax update for one page of 16 tokens held one token per lane
// (lanes t and t+16 carry the same logit). Returns p for this lane's token.
// Logits arrive as hi + lo (lo = 0 for the BF16 segment); m tracks the max of hi.
template <int GQ>
__device__ __forceinline__ void softmax_page(float (&lg)[GQ], float (&lgl)[GQ], float (&m)[GQ], float (&l)[GQ],
                                             float (&alpha)[GQ], float (&p)[GQ]) {
#pragma unroll
    for (int h = 0; h < GQ; ++h) {
        float mp = lg[h];
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) mp = fmaxf(mp, __shfl_xor_sync(0xffffffffu, mp, o));
        const float mn = fmaxf(m[h], mp);
        if (mn == -INFINITY) {          // nothing valid yet
            alpha[h] = 1.0f;
            p[h] = 0.0f;
            continue;
        }
        alpha[h] = fast_exp2(m[h] - mn);
        p[h] = fast_exp2(__fadd_rn(__fsub_rn(lg[h], mn), lgl[h]));
        float ps = p[h];
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
        l[h] = l[h] * alpha[h] + ps;
        m[h] = mn;
    }
}

template <int D, int G, int GQ>
__global__ void __launch_bounds__(kWarps * 32)
split_kernel(SplitArgs a) {
    constexpr int n = D / 16;
    constexpr int MPL = n / 2;          // V m-steps owned per lane (INT2)
    constexpr int CPL = D / 32;         // channels per lane (BF16 PV)
    constexpr int NG = D / G;
    using GE = Geo<D, G>;

    __shared__ __align__(16) float qs[GQ * D];     // INT2: grid part of q_rot; BF16: q
    __shared__ __align__(16) float qrs[GQ * D];    // INT2: residual of q_rot
    __shared__ float qsum_s[GQ][NG][2];
    __shared__ float p_s[kWarps][16][GQ];
    __shared__ float acc_s[GQ * D];
    __shared__ float ml_s[kWarps][GQ][2];

    const int split = blockIdx.x, kv = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int h_q = a.h_kv * GQ;
    const bool is_int2 = split < a.int2_splits;

    for (int i = threadIdx.x; i < GQ * D; i += blockDim.x) {
        const size_t qi = ((size_t)b * h_q + kv * GQ) * D + i;
        qs[i] = is_int2 ? a.qg[qi] : __bfloat162float(a.q[qi]);
        qrs[i] = is_int2 ? a.qr[qi] : 0.0f;
        acc_s[i] = 0.0f;
    }
    if (threadIdx.x < GQ * NG * 2)
        (&qsum_s[0][0][0])[threadIdx.x] = a.qsum[((size_t)b * h_q + kv * GQ) * NG * 2 + threadIdx.x];
    __syncthreads();

    float m[GQ], l[GQ];
#pragma unroll
    for (int h = 0; h < GQ; ++h) { m[h] = -INFINITY; l[h] = 0.0f; }

    const int t = lane & 15, hf = lane >> 4;

    if (is_int2) {
        int len = a.hist_len[b];
        const int cap = min(a.max_hist, a.int2_stride * kPage);
        if (len < 0 || len > cap) {
            if (a.debug && threadIdx.x == 0) record_error(&a.dbg->kind, &a.dbg->index, 3, len);
            len = len < 0 ? 0 : cap;
        }
        const int n_pages = (len + kPage - 1) / kPage;
        const int pg0 = split * a.pages_per_split;
        const int pg1 = min(n_pages, pg0 + a.pages_per_split);

        float acc[GQ][MPL];
#pragma unroll
        for (int h = 0; h < GQ; ++h)
#pragma unroll
            for (int j = 0; j < MPL; ++j) acc[h][j] = 0.0f;

        const int r = lane & 15, mh = lane >> 4;
        const int vbase = 4 * n * (r % 8) + 2 * n * (r / 8) + 2 * MPL * mh;   // bit offset of this lane's V codes

        for (int pg = pg0 + warp; pg < pg1; pg += kWarps) {
            const int32_t phys = a.int2_tables[(size_t)b * a.int2_stride + pg];
            if (phys < 0 || phys >= a.int2_pages) {
                if (a.debug && lane == 0) record_error(&a.dbg->kind, &a.dbg->index, 2, phys);
                continue;
            }
            const uint8_t* blk = a.int2_pool + ((size_t)phys * a.h_kv + kv) * GE::kBlock;
            const uint8_t* kseg = blk;
            const uint8_t* vseg = blk + GE::kSeg;
            const bool valid = pg * kPage + t < len;

            // ---- QK: lane = (token t, half hf of the K bit runs)
            uint32_t w[n / 2];
            if constexpr (D == 128) {
                const uint4 u = *reinterpret_cast<const uint4*>(kseg + t * GE::kCodeRow + 16 * hf);
                w[0] = u.x; w[1] = u.y; w[2] = u.z; w[3] = u.w;
            } else {
                const uint2 u = *reinterpret_cast<const uint2*>(kseg + t * GE::kCodeRow + 8 * hf);
                w[0] = u.x; w[1] = u.y;
            }
            // S = sum_c code_c * q_rot_c per group: grid part exact, residual in fp32
            float shi[GQ][NG], slo[GQ][NG];
#pragma unroll
            for (int h = 0; h < GQ; ++h)
#pragma unroll
                for (int gg = 0; gg < NG; ++gg) { shi[h][gg] = 0.0f; slo[h][gg] = 0.0f; }
#pragma unroll
            for (int tl = 0; tl < 2; ++tl)
#pragma unroll
                for (int kk = 0; kk < n; ++kk)
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int word = tl * (n / 4) + kk / 4;
                        const int bit = 16 * (i % 2) + 2 * (2 * (kk % 4) + i / 2);
                        const float cf = (float)((w[word] >> bit) & 3u);
                        const int c = 16 * kk + 4 * (2 * hf + tl) + i;
#pragma unroll
                        for (int h = 0; h < GQ; ++h) {
                            shi[h][(16 * kk) / G] = __fmaf_rn(qs[h * D + c], cf, shi[h][(16 * kk) / G]);
                            slo[h][(16 * kk) / G] = __fmaf_rn(qrs[h * D + c], cf, slo[h][(16 * kk) / G]);
                        }
                    }
            const __half2* ksz = reinterpret_cast<const __half2*>(kseg + GE::kCodeBytes) + t * NG;
            float lg[GQ], lgl[GQ];
#pragma unroll
            for (int h = 0; h < GQ; ++h) {
                // logit = sm2 * sum_g (s_g * S_g + z_g * Q_g), carried as hi + lo
                float dh = 0.0f, dl = 0.0f;
#pragma unroll
                for (int gg = 0; gg < NG; ++gg) {
                    const float sh = __fadd_rn(shi[h][gg], __shfl_xor_sync(0xffffffffu, shi[h][gg], 16));
                    const float sl = __fadd_rn(slo[h][gg], __shfl_xor_sync(0xffffffffu, slo[h][gg], 16));
                    const float2 sz = __half22float2(ksz[gg]);
                    float p1, e1, p2, e2, t1, e3, t2, e4;
                    two_prod(sz.x, sh, p1, e1);
                    two_prod(sz.y, qsum_s[h][gg][0], p2, e2);
                    two_sum(p1, p2, t1, e3);
                    const float low = __fadd_rn(__fadd_rn(e1, e2), __fadd_rn(e3,
                                      __fmaf_rn(sz.x, sl, __fmul_rn(sz.y, qsum_s[h][gg][1]))));
                    two_sum(dh, t1, t2, e4);
                    dh = t2;
                    dl = __fadd_rn(dl, __fadd_rn(low, e4));
                }
                float lh, ll;
                two_prod(dh, a.scale_log2, lh, ll);
                ll = __fadd_rn(ll, __fmaf_rn(dl, a.scale_log2, __fmul_rn(dh, a.scale_log2_lo)));
                lg[h] = valid ? lh : -INFINITY;
                lgl[h] = valid ? ll : 0.0f;
            }
            float alpha[GQ], p[GQ];
            softmax_page<GQ>(lg, lgl, m, l, alpha, p);
            if (hf == 0) {
#pragma unroll
                for (int h = 0; h < GQ; ++h) p_s[warp][t][h] = p[h];
            }
            __syncwarp();

            // ---- PV: lane = (row r, m-steps [MPL*mh, MPL*mh+MPL)) in the rotated basis
#pragma unroll
            for (int h = 0; h < GQ; ++h)
#pragma unroll
                for (int j = 0; j < MPL; ++j) acc[h][j] *= alpha[h];
            const __half2* vsz = reinterpret_cast<const __half2*>(vseg + GE::kCodeBytes);
            const int tmax = min(kPage, len - pg * kPage);
            for (int tt = 0; tt < tmax; ++tt) {
                const uint32_t byte = vseg[tt * GE::kCodeRow + vbase / 8];
                const uint32_t bits = byte >> (vbase % 8);
#pragma unroll
                for (int j = 0; j < MPL; ++j) {
                    const int grp = (16 * (MPL * mh + j) + r) / G;
                    const float2 sz = __half22float2(vsz[tt * NG + grp]);
                    const float cf = (float)((bits >> (2 * j)) & 3u);
                    const float v = fmaf(cf, sz.x, sz.y);
#pragma unroll
                    for (int h = 0; h < GQ; ++h) acc[h][j] = fmaf(p_s[warp][tt][h], v, acc[h][j]);
                }
            }
            __syncwarp();
        }
        // ---- combine the warps
#pragma unroll
        for (int h = 0; h < GQ; ++h)
            if (lane == 0) { ml_s[warp][h][0] = m[h]; ml_s[warp][h][1] = l[h]; }
        __syncthreads();
#pragma unroll
        for (int h = 0; h < GQ; ++h) {
            float mm = -INFINITY;
            for (int w2 = 0; w2 < kWarps; ++w2) mm = fmaxf(mm, ml_s[w2][h][0]);
            const float f = (m[h] == -INFINITY) ? 0.0f : fast_exp2(m[h] - mm);
#pragma unroll
            for (int j = 0; j < MPL; ++j)
                atomicAdd(&acc_s[h * D + 16 * (MPL * mh + j) + r], acc[h][j] * f);
        }
    } else {
        // ---------------- BF16 sink/recent split
        const int bs = split - a.int2_splits;
        int len = a.bf16_len[b];
        const int cap = min(a.max_bf16, a.bf16_stride * kPage);
        if (len < 0 || len > cap) {
            if (a.debug && threadIdx.x == 0) record_error(&a.dbg->kind, &a.dbg->index, 3, len);
            len = len < 0 ? 0 : cap;
        }
        const int n_pages = (len + kPage - 1) / kPage;
        const int pg0 = bs * a.bf16_pages_per_split;
        const int pg1 = min(n_pages, pg0 + a.bf16_pages_per_split);
        float acc[GQ][CPL];
#pragma unroll
        for (int h = 0; h < GQ; ++h)
#pragma unroll
            for (int j = 0; j < CPL; ++j) acc[h][j] = 0.0f;

        for (int pg = pg0 + warp; pg < pg1; pg += kWarps) {
            const int32_t phys = a.bf16_tables[(size_t)b * a.bf16_stride + pg];
            if (phys < 0 || phys >= a.bf16_pages) {
                if (a.debug && lane == 0) record_error(&a.dbg->kind, &a.dbg->index, 2, phys);
                continue;
            }
            const __nv_bfloat16* kp = a.bf16_pool + (((size_t)phys * a.h_kv + kv) * 2 + 0) * kPage * D;
            const __nv_bfloat16* vp = kp + kPage * D;
            const bool valid = pg * kPage + t < len;
            float lg[GQ];
#pragma unroll
            for (int h = 0; h < GQ; ++h) lg[h] = 0.0f;
            const __nv_bfloat16* krow = kp + t * D + hf * (D / 2);
#pragma unroll
            for (int c8 = 0; c8 < D / 2; c8 += 8) {
                const uint4 u = *reinterpret_cast<const uint4*>(krow + c8);
                const __nv_bfloat162* k2 = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 kf = __bfloat1622float2(k2[e]);
                    const int c = hf * (D / 2) + c8 + 2 * e;
#pragma unroll
                    for (int h = 0; h < GQ; ++h)
                        lg[h] = fmaf(qs[h * D + c], kf.x, fmaf(qs[h * D + c + 1], kf.y, lg[h]));
                }
            }
            float lgl[GQ];
#pragma unroll
            for (int h = 0; h < GQ; ++h) {
                lg[h] += __shfl_xor_sync(0xffffffffu, lg[h], 16);
                float lh, ll;
                two_prod(lg[h], a.scale_log2, lh, ll);
                ll = __fmaf_rn(lg[h], a.scale_log2_lo, ll);
                lg[h] = valid ? lh : -INFINITY;
                lgl[h] = valid ? ll : 0.0f;
            }
            float alpha[GQ], p[GQ];
            softmax_page<GQ>(lg, lgl, m, l, alpha, p);
            if (hf == 0) {
#pragma unroll
                for (int h = 0; h < GQ; ++h) p_s[warp][t][h] = p[h];
            }
            __syncwarp();
#pragma unroll
            for (int h = 0; h < GQ; ++h)
#pragma unroll
                for (int j = 0; j < CPL; ++j) acc[h][j] *= alpha[h];
            const int tmax = min(kPage, len - pg * kPage);
            for (int tt = 0; tt < tmax; ++tt) {
                float v[CPL];
                if constexpr (CPL == 4) {
                    const uint2 u = *reinterpret_cast<const uint2*>(vp + tt * D + 4 * lane);
                    const float2 a0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
                    const float2 a1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
                    v[0] = a0.x; v[1] = a0.y; v[2] = a1.x; v[3] = a1.y;
                } else {
                    const float2 a0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(vp + tt * D + 2 * lane));
                    v[0] = a0.x; v[1] = a0.y;
                }
#pragma unroll
                for (int h = 0; h < GQ; ++h)
#pragma unroll
                    for (int j = 0; j < CPL; ++j) acc[h][j] = fmaf(p_s[warp][tt][h], v[j], acc[h][j]);
            }
            __syncwarp();
        }
#pragma unroll
        for (int h = 0; h < GQ; ++h)
            if (lane == 0) { ml_s[warp][h][0] = m[h]; ml_s[warp][h][1] = l[h]; }
        __syncthreads();
#pragma unroll
        for (int h = 0; h < GQ; ++h) {
            float mm = -INFINITY;
            for (int w2 = 0; w2 < kWarps; ++w2) mm = fmaxf(mm, ml_s[w2][h][0]);
            const float f = (m[h] == -INFINITY) ? 0.0f : fast_exp2(m[h] - mm);
#pragma unroll
            for (int j = 0; j < CPL; ++j) atomicAdd(&acc_s[h * D + CPL * lane + j], acc[h][j] * f);
        }
    }
    __syncthreads();

    // ---- write the partial of each query head of the group
    for (int h = 0; h < GQ; ++h) {
        float mm = -INFINITY;
        for (int w2 = 0; w2 < kWarps; ++w2) mm = fmaxf(mm, ml_s[w2][h][0]);
        float ll = 0.0f;
        for (int w2 = 0; w2 < kWarps; ++w2) {
            const float mw = ml_s[w2][h][0];
            if (mw != -INFINITY) ll += ml_s[w2][h][1] * fast_exp2(mw - mm);
        }
        float* dst = a.partials + (((size_t)b * h_q + kv * GQ + h) * a.total_splits + split) * (D + 2);
        for (int c = threadIdx.x; c < D; c += blockDim.x) dst[2 + c] = acc_s[h * D + c];
        if (threadIdx.x == 0) { dst[0] = mm; dst[1] = ll; }
    }
}

template <int D>
__global__ void merge_kernel(const float* __restrict__ partials, const float* __restrict__ r_vt,
                             float* __restrict__ out, int h_q, int g, int int2_splits, int total_splits) {
    __shared__ float acc_rot[D];
    const int bh = blockIdx.x;
    const int kv = (bh % h_q) / g;
    const int c = threadIdx.x;
    const float* part = partials + (size_t)bh * total_splits * (D + 2);
    float mm = -INFINITY;
    for (int s = 0; s < total_splits; ++s) mm = fmaxf(mm, part[(size_t)s * (D + 2)]);
    float L = 0.0f, ai = 0.0f, ab = 0.0f;
    if (mm != -INFINITY) {
        for (int s = 0; s < total_splits; ++s) {
            const float* ps = part + (size_t)s * (D + 2);
            if (ps[0] == -INFINITY) continue;
            const float w = fast_exp2(ps[0] - mm);
            L = fmaf(ps[1], w, L);
            if (s < int2_splits) ai = fmaf(ps[2 + c], w, ai);
            else ab = fmaf(ps[2 + c], w, ab);
        }
    }
    acc_rot[c] = ai;
    __syncthreads();
    const float* rt = r_vt + (size_t)kv * D * D;
    float o = 0.0f;
#pragma unroll 8
    for (int i = 0; i < D; ++i) o = fmaf(acc_rot[i], __ldg(rt + i * D + c), o);
    out[(size_t)bh * D + c] = L > 0.0f ? (o + ab) / L : 0.0f;
}

template <int D, int G, int GQ>
cudaError_t launch_split(const SplitArgs& a, int batch, cudaStream_t st) {
    dim3 grid(a.total_splits, a.h_kv, batch);
    split_kernel<D, G, GQ><<<grid, kWarps * 32, 0, st>>>(a);
    return cudaGetLastError();
}

template <int D, int G>
cudaError_t dispatch_gq(int gq, const SplitArgs& a, int batch, cudaStream_t st) {
    switch (gq) {
        case 1: return launch_split<D, G, 1>(a, batch, st);
        case 2: return launch_split<D, G, 2>(a, batch, st);
        case 4: return launch_split<D, G, 4>(a, batch, st);
        case 8: return launch_split<D, G, 8>(a, batch, st);
    }
    return cudaErrorInvalidValue;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

DecodePlan plan_decode(const Shape& s, int num_sms, int batch, int max_hist) {
    DecodePlan p{};
    const int max_pages = (max_hist + kPage - 1) / kPage;
    const int units = batch * s.h_kv;
    int splits = units > 0 ? (4 * num_sms + units - 1) / units : 1;
    if (splits < 1) splits = 1;
    if (max_pages > 0 && splits > max_pages) splits = max_pages;
    if (max_pages == 0) splits = 1;
    p.pages_per_split = max_pages > 0 ? (max_pages + splits - 1) / splits : 1;
    p.int2_splits = max_pages > 0 ? (max_pages + p.pages_per_split - 1) / p.pages_per_split : 1;
    p.bf16_splits = 1;
    p.total_splits = p.int2_splits + p.bf16_splits;
    p.ws_partials = align256((size_t)batch * s.h_q * p.total_splits * (s.d + 2) * sizeof(float));
    p.ws_qrot = align256((size_t)batch * s.h_q * (2 * s.d + 2 * (s.d / s.group)) * sizeof(float));
    p.ws_total = p.ws_partials + p.ws_qrot;
    return p;
}

cudaError_t launch_decode(const Shape& s, const LayerParams& prm, const DecodePlan& plan,
                          const DecodeArgs& a, DebugWord* dbg, Profiler* prof, cudaStream_t st) {
    const int g = s.h_q / s.h_kv;
    float* partials = static_cast<float*>(a.ws);
    float* qg = reinterpret_cast<float*>(static_cast<char*>(a.ws) + plan.ws_partials);
    float* qr = qg + (size_t)a.batch * s.h_q * s.d;
    float* qsum = qr + (size_t)a.batch * s.h_q * s.d;
    const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q);

    {
        ProfScope ps(prof, OSCAR_KERNEL_QROT, st);
#define OSCAR_QPREP_CASE(D_, G_) \
        if (s.d == D_ && s.group == G_) \
            q_prep_kernel<D_, G_><<<a.batch * s.h_q, D_, 0, st>>>(q, prm.r_k, qg, qr, qsum, s.h_q, g);
        OSCAR_QPREP_CASE(64, 32)
        OSCAR_QPREP_CASE(64, 64)
        OSCAR_QPREP_CASE(128, 32)
        OSCAR_QPREP_CASE(128, 64)
        OSCAR_QPREP_CASE(128, 128)
#undef OSCAR_QPREP_CASE
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;

    SplitArgs sa{};
    sa.qg = qg; sa.qr = qr; sa.qsum = qsum; sa.q = q;
    sa.int2_pool = a.int2_pool; sa.int2_pages = a.int2_pages;
    sa.int2_tables = a.int2_tables; sa.int2_stride = a.int2_stride;
    sa.hist_len = a.hist_len; sa.max_hist = a.max_hist;
    sa.bf16_pool = reinterpret_cast<const __nv_bfloat16*>(a.bf16_pool); sa.bf16_pages = a.bf16_pages;
    sa.bf16_tables = a.bf16_tables; sa.bf16_stride = a.bf16_stride;
    sa.bf16_len = a.bf16_len; sa.max_bf16 = s.sink + s.recent;
    sa.partials = partials;
    sa.h_kv = s.h_kv; sa.int2_splits = plan.int2_splits; sa.pages_per_split = plan.pages_per_split;
    sa.bf16_splits = plan.bf16_splits;
    sa.bf16_pages_per_split = (s.sink + s.recent + kPage - 1) / kPage;
    sa.total_splits = plan.total_splits;
    {
        const double sl2 = s.sm_scale * 1.4426950408889634073599;
        sa.scale_log2 = (float)sl2;
        sa.scale_log2_lo = (float)(sl2 - (double)sa.scale_log2);
    }
    sa.debug = s.debug; sa.dbg = dbg;

    ProfScope ps_split(prof, OSCAR_KERNEL_SPLIT, st);
#define OSCAR_SPLIT_CASE(D_, G_) \
    if (s.d == D_ && s.group == G_) e = dispatch_gq<D_, G_>(g, sa, a.batch, st); else
    OSCAR_SPLIT_CASE(64, 32)
    OSCAR_SPLIT_CASE(64, 64)
    OSCAR_SPLIT_CASE(128, 32)
    OSCAR_SPLIT_CASE(128, 64)
    OSCAR_SPLIT_CASE(128, 128)
    e = cudaErrorInvalidValue;
#undef OSCAR_SPLIT_CASE
    ps_split.stop();
    if (e != cudaSuccess) return e;

    ProfScope ps_merge(prof, OSCAR_KERNEL_MERGE, st);

    if (s.d == 128)
        merge_kernel<128><<<a.batch * s.h_q, 128, 0, st>>>(partials, prm.r_vt, a.out, s.h_q, g,
                                                           plan.int2_splits, plan.total_splits);
    else
        merge_kernel<64><<<a.batch * s.h_q, 64, 0, st>>>(partials, prm.r_vt, a.out, s.h_q, g,
                                                         plan.int2_splits, plan.total_splits);
    return cudaGetLastError();
}

}  // namespace oscar
