// Device code of the paged decode, shared by its translation units: decode_kernels.cu (query
// preparation, merge, plan and launch) and the split_*.cu units, each of which instantiates the split
// kernel for a group of shapes.
//
// Method: QbitAI article on OSCAR, serving-pipeline part. At decode, the INT2
// part unpacks codes, dequantizes with scale/zero point and accumulates in
// floating point. A BF16 part covers sink and recent. An online-softmax merge
// combines the two. arXiv 2605.17757 abstracts: the kernels keep the paged
// KV-cache layout and prefix caching (block tables may share pages).
//
// Two or three launches per layer:
//   1. q_prep: q_rot = q @ R_k for every query head, accumulated as two fp32
//      (about 48 bits), one CTA per 32 rotated channels (of one query head, or of
//      all g heads of a KV head when the per-head grid is more than about a wave).
//      It is cut into three 11-bit fp16 tensor-core operands on a fixed-point
//      grid whose exponent comes from a bound (|q| times the largest column norm
//      of R_k), so the CTAs of one head agree on it without exchanging a maximum.
//      Each CTA also writes the exact digit sums of its channels.
//   2. split: one CTA per (split, KV head, sequence).
//      - INT2 splits stream page blocks into shared memory, each lane copying
//        its 16-byte chunks with cp.async, three slots of two pages per warp.
//        They compute q_rot . codes and p . codes with mma.sync m16n8k16 on
//        the packed codes, and keep an online softmax; full pages take a body
//        without per-token masks.
//      - BF16 splits handle sink + recent on CUDA cores: the last split of each
//        (sequence, KV head), or the last two when one wave serves few units.
//      - Each split writes a partial (m, l, acc[d]) per query head of the
//        group, with m in log2 units.
//   3. merge: combines the splits of each query head, un-rotates the INT2
//      accumulator by R_v^T and normalises. Its R_v^T terms load before it
//      waits for the split kernel. One CTA takes one query head, or all g heads
//      of a (sequence, KV head) when one CTA per head would take more than a
//      wave; that one skips the partials of zero weight (the empty splits of
//      shorter sequences). When that merge is short (g x splits <=
//      128, i.e. large batches in several waves) the CTA of the split kernel
//      that finishes a (sequence, KV head) last does it instead, found by an
//      atomic ticket (zeroed by q_prep; nothing waits on another CTA), and
//      there are two launches per layer.

// Exactness of the INT2 logits. With codes c in {0..3}, scale s and zero z per
// group:
//   q . (c*s + z) = s * (q . c) + z * sum(q).
// q . c is computed exactly: every q part is an 11-bit integer on a power-of-two
// grid, so each tensor-core partial sum is an exactly representable fp32. With one
// group per token the logit is formed relative to an integer running reference m:
// z * Q_hi is exact (Q_hi cut to 13 bits), z * Q_hi - m is an exact two-sum, and the
// exact product s * X_hi enters one fused multiply-add that rounds at the scale of
// l - m. With several groups s and z enter through error-free products and the logit
// is carried as hi + lo into the softmax exponent. Either way INT2 logits keep about
// 1e-7 absolute accuracy even where they are ~30 in log2 units.
//
// Unpacking. A packed code pair at bit position p of a 32-bit word becomes an
// fp16 (sub)normal c * 2^(2p-24) with a single mask (positions 5..7 after one
// shift by 10). Each position's power of two is folded into the query operand
// (QK) or into a per-m-step rescale of the output (PV).

#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <atomic>
#include <cfloat>
#include <cmath>
#include <type_traits>

#include "layout.cuh"
#include "oscar_internal.h"

namespace oscar {

struct SplitArgs {
    const __half* qb;             // [B][H_q][3][D] tensor-core query parts
    const float* kap;             // [B][H_q]
    const float* qdig;            // [B][H_q][D/32][3] digit sums per 32-channel slice
    const float* pv_scale;        // [H_kv] 2^sigma for the p * s_v operand
    const __nv_bfloat16* q;       // [B][H_q][D]
    const uint8_t* int2_pool; int64_t int2_pages;
    const int32_t* int2_tables; int int2_stride;
    const int32_t* hist_len; int max_hist;
    const __nv_bfloat16* bf16_pool; int64_t bf16_pages;
    const int32_t* bf16_tables; int bf16_stride;
    const int32_t* bf16_len; int max_bf16;
    float* partials;              // [B][H_q][S][D+2]
    int h_kv, int2_splits, pages_per_split, bf16_splits, bf16_pages_per_split;
    // shared prefix (cascade): pages every sequence's history starts with, read by prefix CTAs that
    // each serve kWarps sequences; their partials take slots [0, prefix_splits), the per-sequence
    // splits follow
    const int32_t* prefix_table; int prefix_pages, prefix_pages_per_split, prefix_splits, n_prefix_ctas, batch;
    int total_splits;             // partial slots per query head: prefix + INT2 + BF16 splits
    float scale_log2, scale_log2_lo;   // sm_scale * log2(e) as hi + lo
    int debug; DebugWord* dbg;
    int fuse_merge;               // the CTA finishing a (sequence, KV head) last merges it
    int* counters;                // [B][H_kv] merge tickets, zeroed by q_prep
    const float* r_vt;            // [H_kv][D][D]
    float* out;                   // [B][H_q][D]
};

namespace {

constexpr int kWarps = 4;
constexpr int kStages = 4;                         // ring stages per warp of the shared-prefix CTAs
constexpr int kSlots = 3;                          // two-page pipeline slots per warp of the INT2 splits
constexpr long long kWaitCycles = 2000000000LL;   // give up on a page copy after ~1 s
constexpr float kNoMax = -1e30f;                   // running max before any token
constexpr int kMaxPagesPerSplit = 128;             // longest INT2 split when the grid has many waves
// last-CTA merge only for short merges (one CTA walks GQ * splits partial rows): large batches;
// bs1 decodes with ~80 splits keep the wider merge kernel
constexpr int kFuseWeights = 128;
constexpr int kSliceCh = 32;                       // rotated channels per q_prep CTA
constexpr size_t kMergeUnitWeightBytes = 160 * 1024;  // largest weight table of the per-unit merge

__device__ __forceinline__ float fast_exp2(float x) { return exp2f(x); }

// Error-free transformations on fp32 (explicit _rn intrinsics: no contraction).
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
    s = __fadd_rn(a, b);
    const float bp = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bp)), __fsub_rn(b, bp));
}

__device__ __forceinline__ void two_prod(float a, float b, float& p, float& e) {
    p = __fmul_rn(a, b);
    e = __fmaf_rn(a, b, -p);
}

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Position p' and fp16 bit pattern of the code pair at position `pos` (0..7) of word w:
// c_lo * 2^(2p'-24) in the low half, c_hi * 2^(2p'-24) in the high half.
__host__ __device__ constexpr int pos_scale(int pos) { return pos <= 4 ? pos : pos - 5; }

// 2^(-2 p'(pos)): undoes the code position's power of two in the P.V output.
__host__ __device__ constexpr float pos_weight(int pos) {
    return pos_scale(pos) == 0 ? 1.0f
         : pos_scale(pos) == 1 ? 0x1p-2f
         : pos_scale(pos) == 2 ? 0x1p-4f
         : pos_scale(pos) == 3 ? 0x1p-6f
                               : 0x1p-8f;
}

template <int POS>
__device__ __forceinline__ uint32_t code_pair(uint32_t w, uint32_t w10) {
    if constexpr (POS <= 4) return w & (0x00030003u << (2 * POS));
    else return w10 & (0x00030003u << (2 * (POS - 5)));
}

// Code pair at position POS as a normal fp16 pair c * 2^(2p'): the masked bits form the mantissa of
// 1024 + c * 2^(2p'), then 1024 is subtracted exactly. Normal operands keep the tensor-core products
// of P.V at full precision (fp16 subnormal operands lose low bits against larger products).
// (w & mask) | bias as one three-input logic instruction (lookup table 0xEA = (a & b) | c).
__device__ __forceinline__ uint32_t and_or(uint32_t w, uint32_t mask, uint32_t bias) {
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(w), "r"(mask), "r"(bias));
    return r;
}

template <int POS>
__device__ __forceinline__ uint32_t code_pair_normal(uint32_t w, uint32_t w10) {
    const uint32_t h = POS <= 4 ? and_or(w, 0x00030003u << (2 * POS), 0x64006400u)
                                : and_or(w10, 0x00030003u << (2 * (POS - 5)), 0x64006400u);
    const __half2 r = __hsub2(*reinterpret_cast<const __half2*>(&h), __half2(__ushort_as_half(0x6400), __ushort_as_half(0x6400)));
    return *reinterpret_cast<const uint32_t*>(&r);
}

__device__ __forceinline__ uint32_t pack_half2(__half lo, __half hi) {
    return (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
}

// Programmatic dependent launch: wait for the preceding grid in the stream (a no-op without the
// launch attribute), and let the next grid start its prologue.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void mbar_init(uint32_t bar, int count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(bar), "r"(bytes) : "memory");
    asm volatile("cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 :: "r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}

// 16-byte asynchronous copy global -> shared (bypassing L1), issued only where `pred` holds, and its
// commit groups: the issuing thread waits for its own copies; a warp barrier then publishes them to the
// other lanes.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool pred) {
    asm volatile("{ .reg .pred p; setp.ne.b32 p, %2, 0; @p cp.async.cg.shared.global [%0], [%1], 16; }"
                 :: "r"(dst), "l"(src), "r"((int)pred) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory"); }

__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t phase) {
    uint32_t ok;
    asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
                 : "=r"(ok) : "r"(bar), "r"(phase) : "memory");
    return ok != 0;
}

// Bounded wait on an mbarrier phase; false if it did not complete within kWaitCycles.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t phase) {
    if (mbar_test(bar, phase)) return true;
    const long long t0 = clock64();
    while (!mbar_test(bar, phase))
        if (clock64() - t0 > kWaitCycles) return false;
    return true;
}

// ---------------------------------------------------------------------------------------------
// Query preparation
// ---------------------------------------------------------------------------------------------

// The rest of q_prep for one (query head, channel) once the four quarter partials of q . R_k[:, c] are
// known: double-float sum, times sm_scale log2(e), the exponent grid from the norm bound, the three
// digits, and (through the warp, whose 32 lanes are the slice's channels) the slice's digit sums.
template <int D>
__device__ __forceinline__ void q_prep_finish(const float (&hi_u)[4], const float (&lo_u)[4], float nq2, float cmax,
                                              float sl2_hi, float sl2_lo, size_t bh, int slice, int cl, int c,
                                              __half* __restrict__ qb, float* __restrict__ kap,
                                              float* __restrict__ qdig) {
    constexpr int NS = D / kSliceCh;
    float h = 0.0f, l = 0.0f;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        float s2, e2;
        two_sum(h, hi_u[u], s2, e2);
        h = s2;
        l = __fadd_rn(l, __fadd_rn(lo_u[u], e2));
    }
    {
        float s2, e2;
        two_sum(h, l, s2, e2);
        h = s2;
        l = e2;
    }
    // times sm_scale * log2(e) (hi + lo): the INT2 logits come out in log2 units
    {
        float p, e, s2, e2;
        two_prod(h, sl2_hi, p, e);
        e = __fmaf_rn(h, sl2_lo, __fmaf_rn(l, sl2_hi, e));
        two_sum(p, e, s2, e2);
        h = s2;
        l = e2;
    }
    // exponent from the bound: (sl2 |q| cmax)^2 with a relative margin for the rounding of |q|^2
    const float sc = sl2_hi * cmax;
    const float bound2 = nq2 * sc * sc * 1.0001f;
    int e2x = 0;
    frexpf(bound2, &e2x);                              // bound2 < 2^e2x
    const int ex = (e2x + 1) >> 1;                     // bound < 2^ex (arithmetic shift: ceil(e2x / 2))
    const bool any = nq2 > 0.0f;
    // r_hi, r_mid, r_lo: successive 11-bit digits of q_rot / 2^(ex-11)
    const float xh = ldexpf(h, 11 - ex), xl = ldexpf(l, 11 - ex);
    const float r_hi = any ? rintf(xh) : 0.0f;
    const float rem1 = __fadd_rn(__fsub_rn(xh, r_hi), xl);                // |rem1| <= 0.5 + tiny
    const float r_mid = any ? rintf(__fmul_rn(rem1, 2048.0f)) : 0.0f;
    const float rem2 = __fsub_rn(__fmul_rn(rem1, 2048.0f), r_mid);
    const float r_lo = any ? rintf(__fmul_rn(rem2, 2048.0f)) : 0.0f;
    const int pos = 2 * ((c / 16) % 4) + (c % 4) / 2;                     // K-layout position of channel c
    const int sh = 4 - 2 * pos_scale(pos);
    __half* dst = qb + (size_t)bh * 3 * D;
    dst[c] = __float2half_rn(ldexpf(r_hi, sh));
    dst[D + c] = __float2half_rn(ldexpf(r_mid, sh));
    dst[2 * D + c] = __float2half_rn(ldexpf(r_lo, sh));
    if (slice == 0 && cl == 0) kap[bh] = any ? ldexpf(1.0f, ex + 9) : 0.0f;
    // exact integer digit sums of the slice (|sum| <= 32 * 2048)
    float d0 = r_hi, d1 = r_mid, d2 = r_lo;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        d0 += __shfl_xor_sync(0xffffffffu, d0, o);
        d1 += __shfl_xor_sync(0xffffffffu, d1, o);
        d2 += __shfl_xor_sync(0xffffffffu, d2, o);
    }
    if (cl == 0) {
        float* qd = qdig + ((size_t)bh * NS + slice) * 3;
        qd[0] = d0;
        qd[1] = d1;
        qd[2] = d2;
    }
}

// One CTA of 128 threads per (query head, slice of 32 rotated channels): thread (channel, quarter)
// accumulates D/4 terms of the dot product.
//   q_rot[c] = sum_i q_i R[i][c] as hi + lo fp32 (error-free products and sums), times
//     sm_scale * log2(e), so the INT2 logits come out in log2 units;
//   E with 2^E > sm_scale log2(e) |q|_2 max_c |R[:, c]|_2 >= max_c |q_rot[c]| (the same in
//     every CTA of the head: every CTA sums |q|^2 in the same order);
//   r_hi, r_mid, r_lo integers (|r| <= 2048) with
//     q_rot = (r_hi + r_mid 2^-11 + r_lo 2^-22) 2^(E-11)  (to ~2^(E-33));
//   qb[part][c] = r_part * 2^(4 - 2p'(c)) as fp16 (exact), p'(c) the fp16 position of channel c
//     in the K layout, so that code(c) * 2^(2p'-24) * qb = code * r_part * 2^-20;
//   kap = 2^(E + 9): S_part = accumulator * kap * 2^(-11 part);
//   qdig[slice][part] = sum over the slice's channels of r_part (exact integers).
template <int D>
__global__ void __launch_bounds__(128)
q_prep_kernel(const __nv_bfloat16* __restrict__ q, const float* __restrict__ r_k, const float* __restrict__ colmax,
              __half* __restrict__ qb, float* __restrict__ kap, float* __restrict__ qdig, int h_q, int g,
              float sl2_hi, float sl2_lo, int* __restrict__ counters, int counters_per_unit) {
    constexpr int Q4 = D / 4;
    __shared__ float qs[D];
    __shared__ float hi_s[4][kSliceCh], lo_s[4][kSliceCh];
    __shared__ float nq2_s;
    const int bh = blockIdx.x, slice = blockIdx.y;
    const int kv = (bh % h_q) / g;
    const int cl = threadIdx.x % kSliceCh, quarter = threadIdx.x / kSliceCh;
    const int c = slice * kSliceCh + cl;
    // R_k terms of this thread: constant calibration data, so they load before the wait for the
    // previous kernel (all in flight at once)
    const float* r = r_k + (size_t)kv * D * D + (size_t)quarter * Q4 * D + c;
    float rv[Q4];
#pragma unroll
    for (int i = 0; i < Q4; ++i) rv[i] = __ldg(r + (size_t)i * D);
    const float cmax = __ldg(colmax + kv);
    pdl_wait();
    pdl_trigger();
    // the split kernel's merge tickets of this (sequence, KV head) start at zero
    if (slice == 0 && (bh % h_q) % g == 0)
        for (int i = threadIdx.x; i < counters_per_unit; i += blockDim.x)
            counters[((size_t)(bh / h_q) * (h_q / g) + kv) * counters_per_unit + i] = 0;
    for (int i = threadIdx.x; i < D; i += blockDim.x) qs[i] = __bfloat162float(q[(size_t)bh * D + i]);
    __syncthreads();
    if (threadIdx.x < 32) {
        // |q|^2 in a fixed order, identical in every CTA of the head
        float s2 = 0.0f;
#pragma unroll
        for (int k = 0; k < D / 32; ++k) s2 = __fmaf_rn(qs[threadIdx.x + 32 * k], qs[threadIdx.x + 32 * k], s2);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s2 = __fadd_rn(s2, __shfl_xor_sync(0xffffffffu, s2, o));
        if (threadIdx.x == 0) nq2_s = s2;
    }
    float hi = 0.0f, lo = 0.0f;
#pragma unroll
    for (int i = 0; i < Q4; ++i) {
        float p, e, s2, e2;
        two_prod(qs[quarter * Q4 + i], rv[i], p, e);
        two_sum(hi, p, s2, e2);
        hi = s2;
        lo = __fadd_rn(lo, __fadd_rn(e, e2));
    }
    hi_s[quarter][cl] = hi;
    lo_s[quarter][cl] = lo;
    __syncthreads();
    if (quarter != 0) return;
    float hi_u[4], lo_u[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) { hi_u[u] = hi_s[u][cl]; lo_u[u] = lo_s[u][cl]; }
    q_prep_finish<D>(hi_u, lo_u, nq2_s, cmax, sl2_hi, sl2_lo, bh, slice, cl, c, qb, kap, qdig);
}

// q_prep for the GQ query heads of one (sequence, KV head) and one slice of 32 rotated channels, for plans
// with many query heads: the R_k terms load once for the GQ heads, and the GQ double-float chains of a
// thread are independent. Every head's |q|^2, dot products and digits are formed in the same order as in
// q_prep_kernel, so both give the same bits.
template <int D, int GQ>
__global__ void __launch_bounds__(128)
q_prep_unit_kernel(const __nv_bfloat16* __restrict__ q, const float* __restrict__ r_k,
                   const float* __restrict__ colmax, __half* __restrict__ qb, float* __restrict__ kap,
                   float* __restrict__ qdig, int h_kv, float sl2_hi, float sl2_lo, int* __restrict__ counters,
                   int counters_per_unit) {
    constexpr int Q4 = D / 4;
    __shared__ float qs[GQ][D];
    __shared__ float hi_s[GQ][4][kSliceCh], lo_s[GQ][4][kSliceCh];
    __shared__ float nq2_s[GQ];
    const int unit = blockIdx.x, slice = blockIdx.y;
    const int kv = unit % h_kv;
    const int cl = threadIdx.x % kSliceCh, quarter = threadIdx.x / kSliceCh;
    const int c = slice * kSliceCh + cl;
    const float* r = r_k + (size_t)kv * D * D + (size_t)quarter * Q4 * D + c;
    float rv[Q4];
#pragma unroll
    for (int i = 0; i < Q4; ++i) rv[i] = __ldg(r + (size_t)i * D);
    const float cmax = __ldg(colmax + kv);
    pdl_wait();
    pdl_trigger();
    if (slice == 0)
        for (int i = threadIdx.x; i < counters_per_unit; i += blockDim.x) counters[(size_t)unit * counters_per_unit + i] = 0;
    const size_t bh0 = (size_t)unit * GQ;                 // b * h_q + kv * GQ
    for (int i = threadIdx.x; i < GQ * D; i += blockDim.x) qs[i / D][i % D] = __bfloat162float(q[bh0 * D + i]);
    __syncthreads();
    // |q|^2 of head h by warp h % 4, in the per-head kernel's order
    for (int h = quarter; h < GQ; h += 4) {
        float s2 = 0.0f;
#pragma unroll
        for (int k = 0; k < D / 32; ++k) s2 = __fmaf_rn(qs[h][cl + 32 * k], qs[h][cl + 32 * k], s2);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s2 = __fadd_rn(s2, __shfl_xor_sync(0xffffffffu, s2, o));
        if (cl == 0) nq2_s[h] = s2;
    }
    float hi[GQ], lo[GQ];
#pragma unroll
    for (int h = 0; h < GQ; ++h) { hi[h] = 0.0f; lo[h] = 0.0f; }
#pragma unroll
    for (int i = 0; i < Q4; ++i) {
#pragma unroll
        for (int h = 0; h < GQ; ++h) {
            float p, e, s2, e2;
            two_prod(qs[h][quarter * Q4 + i], rv[i], p, e);
            two_sum(hi[h], p, s2, e2);
            hi[h] = s2;
            lo[h] = __fadd_rn(lo[h], __fadd_rn(e, e2));
        }
    }
#pragma unroll
    for (int h = 0; h < GQ; ++h) { hi_s[h][quarter][cl] = hi[h]; lo_s[h][quarter][cl] = lo[h]; }
    __syncthreads();
    // warp w finishes heads w, w + 4, ...: its 32 lanes are the slice's channels
    for (int h = quarter; h < GQ; h += 4) {
        float hu[4], lu[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) { hu[u] = hi_s[h][u][cl]; lu[u] = lo_s[h][u][cl]; }
        q_prep_finish<D>(hu, lu, nq2_s[h], cmax, sl2_hi, sl2_lo, bh0 + h, slice, cl, c, qb, kap, qdig);
    }
}

// ---------------------------------------------------------------------------------------------
// Split kernel
// ---------------------------------------------------------------------------------------------


template <int D, int G, int GQ>
struct SplitSmem {
    static constexpr int kBlock = Geo<D, G>::kBlock;
    static constexpr size_t kDynamic = (size_t)kWarps * (kStages > 2 * kSlots ? kStages : 2 * kSlots) * kBlock;
};

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// d = 128 / d = 64 code pair selection for the V operand of m-step mm: rows gid (R0, R2) and
// rows gid+8 (R1, R3); d = 128 takes both from position mm of the low / high half-words, d = 64
// from positions mm and 4+mm of one half-word.
template <int D, int MM>
__device__ __forceinline__ void v_operand(uint32_t X01, uint32_t X01s, uint32_t Y01, uint32_t Y01s, uint32_t X23,
                                          uint32_t X23s, uint32_t Y23, uint32_t Y23s, uint32_t& A0, uint32_t& A1,
                                          uint32_t& A2, uint32_t& A3) {
    if constexpr (D == 128) {
        A0 = code_pair_normal<MM>(X01, X01s); A1 = code_pair_normal<MM>(Y01, Y01s);
        A2 = code_pair_normal<MM>(X23, X23s); A3 = code_pair_normal<MM>(Y23, Y23s);
    } else {
        A0 = code_pair_normal<MM>(X01, X01s); A1 = code_pair_normal<4 + MM>(X01, X01s);
        A2 = code_pair_normal<MM>(X23, X23s); A3 = code_pair_normal<4 + MM>(X23, X23s);
    }
}

template <int D, int KK>
__device__ __forceinline__ void k_operand(const uint32_t (&kw0)[2], const uint32_t (&kw1)[2], uint32_t& A0,
                                          uint32_t& A1, uint32_t& A2, uint32_t& A3) {
    constexpr int W = KK / 4, P = 2 * (KK % 4);
    const uint32_t w0 = kw0[W], w1 = kw1[W];
    A0 = code_pair<P>(w0, w0 >> 10); A1 = code_pair<P>(w1, w1 >> 10);
    A2 = code_pair<P + 1>(w0, w0 >> 10); A3 = code_pair<P + 1>(w1, w1 >> 10);
}

template <int N, typename F>
__device__ __forceinline__ void static_for(F&& f) {
    if constexpr (N > 0) {
        static_for<N - 1>(f);
        f(std::integral_constant<int, N - 1>{});
    }
}

// Query operands of one (sequence, KV head) for this lane, constant over a split's pages: the three
// digit parts as m16n8k16 B fragments, the digit scales and the per-group sums of q_rot (hi + lo).
template <int D, int G, int GQ>
struct QueryOps {
    static constexpr int NK = D / 16, NG = D / G, NHB = (GQ + 3) / 4;
    uint32_t qB1[NK][NHB][2], qB2[NK][2];
    float kap_h[NHB], kap_m[NHB], kap_l[NHB], qs_hi[NHB][NG], qs_lo[NHB][NG];
};

template <int D, int G, int GQ>
__device__ __forceinline__ void load_query_ops(const SplitArgs& a, size_t head0, int gid, int tig,
                                               QueryOps<D, G, GQ>& qo) {
    constexpr int NK = D / 16, NG = D / G, NHB = (GQ + 3) / 4;
    auto& qB1 = qo.qB1;
    auto& qB2 = qo.qB2;
    auto& kap_h = qo.kap_h;
    auto& kap_m = qo.kap_m;
    auto& kap_l = qo.kap_l;
    auto& qs_hi = qo.qs_hi;
    auto& qs_lo = qo.qs_lo;
#pragma unroll
    for (int hb = 0; hb < NHB; ++hb) {
        const int h = 4 * hb + (gid >> 1);
        const int part = gid & 1;
#pragma unroll
        for (int kk = 0; kk < NK; ++kk) {
            uint2 v = make_uint2(0u, 0u);
            if (h < GQ) v = *reinterpret_cast<const uint2*>(a.qb + ((head0 + h) * 3 + part) * D + 16 * kk + 4 * tig);
            qB1[kk][hb][0] = v.x;
            qB1[kk][hb][1] = v.y;
        }
        const int hm = 4 * hb + tig;
        kap_h[hb] = hm < GQ ? a.kap[head0 + hm] : 0.0f;
        kap_m[hb] = kap_h[hb] * 0x1p-11f;
        kap_l[hb] = kap_h[hb] * 0x1p-22f;
#pragma unroll
        for (int gg = 0; gg < NG; ++gg) {
            // sum over the group of q_rot = 2^(E-11) (S_hi + 2^-11 S_mid + 2^-22 S_lo) (kap 2^-20 =
            // 2^(E-11)) as hi + lo fp32, without fp64: the digit sums are exact fp32 integers (<= 2^18),
            // S_hi + 2^-11 S_mid is split error-free, and the 2^-22 S_lo term only enters the low part
            float sh = 0.0f, sm = 0.0f, sl = 0.0f;
            if (hm < GQ) {
#pragma unroll
                for (int s = gg * (G / kSliceCh); s < (gg + 1) * (G / kSliceCh); ++s) {
                    const float* qd = a.qdig + ((head0 + hm) * (D / kSliceCh) + s) * 3;
                    sh += qd[0];
                    sm += qd[1];
                    sl += qd[2];
                }
            }
            float h1, e1;
            two_sum(sh, sm * 0x1p-11f, h1, e1);
            const float k20 = kap_h[hb] * 0x1p-20f;
            const float qh = h1 * k20;
            // hi cut to 13 significant bits, so that z * hi is exact for an fp16 zero point z
            qs_hi[hb][gg] = __uint_as_float(__float_as_uint(qh) & 0xFFFFF800u);
            qs_lo[hb][gg] = __fadd_rn(__fsub_rn(qh, qs_hi[hb][gg]), __fmaf_rn(sl, 0x1p-22f, e1) * k20);
        }
    }
    {
        // lo parts: column n = gid carries head gid/2 (first block) or, for GQ = 8 and odd gid, head 4 + gid/2
        const int h = (GQ == 8 && (gid & 1)) ? 4 + (gid >> 1) : ((gid & 1) ? GQ : (gid >> 1));
#pragma unroll
        for (int kk = 0; kk < NK; ++kk) {
            uint2 v = make_uint2(0u, 0u);
            if (h < GQ) v = *reinterpret_cast<const uint2*>(a.qb + ((head0 + h) * 3 + 2) * D + 16 * kk + 4 * tig);
            qB2[kk][0] = v.x;
            qB2[kk][1] = v.y;
        }
    }
}

// Online-softmax state of one warp: P.V accumulators (rotated basis, scaled by 2^sigma and the code
// positions), running max and sum, and the zero-point sums.
template <int D, int G, int GQ>
struct WarpAcc {
    static constexpr int NK = D / 16, NG = D / G, NHB = (GQ + 3) / 4;
    float O[NHB][NK][4];
    float m_run[NHB], l_run[NHB], zacc[NHB][NG];
    bool valid[NHB];                 // relative-logit bodies: m_run holds the integer reference (warp-uniform)
    __device__ __forceinline__ void init() {
#pragma unroll
        for (int hb = 0; hb < NHB; ++hb) {
#pragma unroll
            for (int mm = 0; mm < NK; ++mm)
#pragma unroll
                for (int e = 0; e < 4; ++e) O[hb][mm][e] = 0.0f;
            m_run[hb] = kNoMax;          // finite: ex2(-inf - kNoMax) = 0 without a guard
            valid[hb] = false;
            l_run[hb] = 0.0f;
#pragma unroll
            for (int gg = 0; gg < NG; ++gg) zacc[hb][gg] = 0.0f;
        }
    }
};

// NP INT2 pages (16 tokens each; with FULL all valid, otherwise the first `nvalid` of the single page) of
// one KV head, staged in shared memory at sb[0..NP), folded into the warp's softmax state. With NP = 2
// the two pages' Q.K products, logits, weights and P.V products are independent chains that the
// scheduler interleaves; they share one test of the lazy reference.
template <int D, int G, int GQ, int NP, bool FULL>
__device__ __forceinline__ void int2_pages(const uint8_t* const (&sb)[NP], int nvalid, int gid, int tig, float pvs,
                                           const QueryOps<D, G, GQ>& qo, WarpAcc<D, G, GQ>& acc) {
    static_assert(NP == 1 || FULL, "several pages at once are full pages");
    using GE = Geo<D, G>;
    constexpr int NK = D / 16, NG = D / G, KPG = G / 16, NHB = (GQ + 3) / 4;
    const auto& qB1 = qo.qB1;
    const auto& qB2 = qo.qB2;
    const auto& kap_h = qo.kap_h;
    const auto& kap_m = qo.kap_m;
    const auto& kap_l = qo.kap_l;
    const auto& qs_hi = qo.qs_hi;
    const auto& qs_lo = qo.qs_lo;
    auto& O = acc.O;
    auto& m_run = acc.m_run;
    auto& l_run = acc.l_run;
    auto& zacc = acc.zacc;
    const bool v0 = FULL || gid < nvalid, v1 = FULL || gid + 8 < nvalid;

    // ---- QK^T on tensor cores: A = K codes [16 tokens x 16 channels], B = query parts
    uint32_t kw0[NP][2], kw1[NP][2];
#pragma unroll
    for (int pi = 0; pi < NP; ++pi) {
        if constexpr (D == 128) {
            const uint2 u0 = *reinterpret_cast<const uint2*>(sb[pi] + gid * GE::kCodeRow + 8 * tig);
            const uint2 u1 = *reinterpret_cast<const uint2*>(sb[pi] + (gid + 8) * GE::kCodeRow + 8 * tig);
            kw0[pi][0] = u0.x; kw0[pi][1] = u0.y; kw1[pi][0] = u1.x; kw1[pi][1] = u1.y;
        } else {
            kw0[pi][0] = *reinterpret_cast<const uint32_t*>(sb[pi] + gid * GE::kCodeRow + 4 * tig);
            kw1[pi][0] = *reinterpret_cast<const uint32_t*>(sb[pi] + (gid + 8) * GE::kCodeRow + 4 * tig);
            kw0[pi][1] = kw1[pi][1] = 0u;
        }
    }
    float S1[NP][NG][NHB][4], S2[NP][NG][4];
#pragma unroll
    for (int pi = 0; pi < NP; ++pi)
#pragma unroll
        for (int gg = 0; gg < NG; ++gg) {
#pragma unroll
            for (int e = 0; e < 4; ++e) S2[pi][gg][e] = 0.0f;
#pragma unroll
            for (int hb = 0; hb < NHB; ++hb)
#pragma unroll
                for (int e = 0; e < 4; ++e) S1[pi][gg][hb][e] = 0.0f;
        }
    static_for<NK>([&](auto kkc) {
        constexpr int kk = decltype(kkc)::value;
        constexpr int gg = kk / KPG;
#pragma unroll
        for (int pi = 0; pi < NP; ++pi) {
            uint32_t A0, A1, A2, A3;
            k_operand<D, kk>(kw0[pi], kw1[pi], A0, A1, A2, A3);
#pragma unroll
            for (int hb = 0; hb < NHB; ++hb)
                mma16816(S1[pi][gg][hb], A0, A1, A2, A3, qB1[kk][hb][0], qB1[kk][hb][1]);
            mma16816(S2[pi][gg], A0, A1, A2, A3, qB2[kk][0], qB2[kk][1]);
        }
    });

    // ---- logits for tokens gid and gid+8 of head 4hb + tig (log2 units: the query carries the scale),
    // weights p, and P' = p * s_v * 2^sigma per token slot as an (hi, lo) fp16 pair
    uint32_t Pv[NP][NHB][NG][2];
#pragma unroll
    for (int hb = 0; hb < NHB; ++hb) {
        const bool hv = GQ % 4 == 0 || 4 * hb + tig < GQ;
        const bool ok0 = v0 && hv, ok1 = v1 && hv;
        float p[NP][2];
        if constexpr (NG == 1) {
            // relative to the integer reference m: l - m = s X_hi + (z Q_hi - m) + z Q_lo + s X_lo, with
            // z Q_hi exact (Q_hi has 13 significant bits, z 11), z Q_hi - m an exact two-sum, and s X_hi
            // exact inside one fused multiply-add whose rounding is at the scale of l - m
            float xh[NP][2], xl[NP][2], sk[NP][2], zk[NP][2], t[NP][2];
#pragma unroll
            for (int pi = 0; pi < NP; ++pi) {
                const __half2* ksz = reinterpret_cast<const __half2*>(sb[pi] + GE::kCodeBytes);
#pragma unroll
                for (int slot = 0; slot < 2; ++slot) {
                    const float lo_raw = (GQ == 8) ? S2[pi][0][2 * slot + hb] : S2[pi][0][2 * slot];
                    xh[pi][slot] = __fmul_rn(S1[pi][0][hb][2 * slot], kap_h[hb]);
                    xl[pi][slot] = __fmaf_rn(S1[pi][0][hb][2 * slot + 1], kap_m[hb], __fmul_rn(lo_raw, kap_l[hb]));
                    const float2 sz = __half22float2(ksz[gid + 8 * slot]);
                    sk[pi][slot] = sz.x;
                    zk[pi][slot] = sz.y;
                }
            }
            auto rel = [&](int pi, int slot, float m) {
                float vh, vl;
                two_sum(__fmul_rn(zk[pi][slot], qs_hi[hb][0]), -m, vh, vl);
                float r = __fmaf_rn(sk[pi][slot], xh[pi][slot], vh);
                r = __fadd_rn(r, vl);
                r = __fmaf_rn(zk[pi][slot], qs_lo[hb][0], r);
                return __fmaf_rn(sk[pi][slot], xl[pi][slot], r);
            };
            auto all_logits = [&](float m) {
                float mx = -INFINITY;
#pragma unroll
                for (int pi = 0; pi < NP; ++pi) {
                    t[pi][0] = ok0 ? rel(pi, 0, m) : -INFINITY;
                    t[pi][1] = ok1 ? rel(pi, 1, m) : -INFINITY;
                    mx = fmaxf(mx, fmaxf(t[pi][0], t[pi][1]));
                }
                return mx;
            };
            const float mx = all_logits(acc.valid[hb] ? m_run[hb] : 0.0f);
            // lazy reference: set on the warp's first page, then raised (to an integer) only when a logit
            // passes it by more than 2^kSoftmaxHeadroomLog2, so p <= 2^8 and the O rescale is rare; only
            // then is the maximum of each head reduced across its lanes and the pages re-evaluated
            if (__any_sync(0xffffffffu, !acc.valid[hb] || mx > (float)kSoftmaxHeadroomLog2)) {
                float mp = mx;
                mp = fmaxf(mp, __shfl_xor_sync(0xffffffffu, mp, 4));
                mp = fmaxf(mp, __shfl_xor_sync(0xffffffffu, mp, 8));
                mp = fmaxf(mp, __shfl_xor_sync(0xffffffffu, mp, 16));
                if (!acc.valid[hb]) {
                    if (hv) m_run[hb] = ceilf(mp);                  // every page holds a valid token
                } else if (mp > (float)kSoftmaxHeadroomLog2) {
                    const float mn = ceilf(m_run[hb] + mp);
                    const float k = mn - m_run[hb];                 // an integer >= 9
                    const float alpha = k > 126.0f ? 0.0f : __int_as_float((127 - (int)k) << 23);   // 2^-k exactly
                    m_run[hb] = mn;
                    l_run[hb] *= alpha;
#pragma unroll
                    for (int mm = 0; mm < NK; ++mm)
#pragma unroll
                        for (int e = 0; e < 4; ++e) O[hb][mm][e] *= alpha;
                    zacc[hb][0] *= alpha;
                }
                acc.valid[hb] = true;
                (void)all_logits(m_run[hb]);
            }
#pragma unroll
            for (int pi = 0; pi < NP; ++pi) {
                p[pi][0] = ex2(t[pi][0]);
                p[pi][1] = ex2(t[pi][1]);
            }
        } else {
            // several groups: the logit as hi + lo against a lazy running maximum
            float lh[NP][2], ll[NP][2];
            float mx = -INFINITY;
#pragma unroll
            for (int pi = 0; pi < NP; ++pi) {
                const __half2* ksz = reinterpret_cast<const __half2*>(sb[pi] + GE::kCodeBytes);
#pragma unroll
                for (int slot = 0; slot < 2; ++slot) {
                    const int tok = gid + 8 * slot;
                    float dh = 0.0f, dl = 0.0f;
#pragma unroll
                    for (int gg = 0; gg < NG; ++gg) {
                        const float lo_raw = (GQ == 8) ? S2[pi][gg][2 * slot + hb] : S2[pi][gg][2 * slot];
                        const float s_hi = __fmul_rn(S1[pi][gg][hb][2 * slot], kap_h[hb]);
                        const float s_r = __fmaf_rn(S1[pi][gg][hb][2 * slot + 1], kap_m[hb],
                                                    __fmul_rn(lo_raw, kap_l[hb]));
                        const float2 sz = __half22float2(ksz[tok * NG + gg]);
                        float p1, e1, p2, e2, t1, e3;
                        two_prod(sz.x, s_hi, p1, e1);
                        two_prod(sz.y, qs_hi[hb][gg], p2, e2);
                        two_sum(p1, p2, t1, e3);
                        const float low = __fadd_rn(__fadd_rn(e1, e2),
                                                    __fadd_rn(e3, __fmaf_rn(sz.x, s_r, __fmul_rn(sz.y, qs_lo[hb][gg]))));
                        float t2, e4;
                        two_sum(dh, t1, t2, e4);
                        dh = t2;
                        dl = __fadd_rn(dl, __fadd_rn(low, e4));
                    }
                    lh[pi][slot] = dh;
                    ll[pi][slot] = dl;
                }
                if (!ok0) { lh[pi][0] = -INFINITY; ll[pi][0] = 0.0f; }
                if (!ok1) { lh[pi][1] = -INFINITY; ll[pi][1] = 0.0f; }
                mx = fmaxf(mx, fmaxf(lh[pi][0], lh[pi][1]));
            }
            // online softmax (lanes sharing tig hold the same head); the reference is raised only when a
            // logit passes it by more than 2^kSoftmaxHeadroomLog2, so p <= 2^8 and the O rescale is rare
            if (__any_sync(0xffffffffu, mx > m_run[hb] + (float)kSoftmaxHeadroomLog2)) {
                float mp = mx;
                mp = fmaxf(mp, __shfl_xor_sync(0xffffffffu, mp, 4));
                mp = fmaxf(mp, __shfl_xor_sync(0xffffffffu, mp, 8));
                mp = fmaxf(mp, __shfl_xor_sync(0xffffffffu, mp, 16));
                const float mn = fmaxf(m_run[hb], mp);
                const float alpha = ex2(m_run[hb] - mn);
                m_run[hb] = mn;
                l_run[hb] *= alpha;
#pragma unroll
                for (int mm = 0; mm < NK; ++mm)
#pragma unroll
                    for (int e = 0; e < 4; ++e) O[hb][mm][e] *= alpha;
#pragma unroll
                for (int gg = 0; gg < NG; ++gg) zacc[hb][gg] *= alpha;
            }
#pragma unroll
            for (int pi = 0; pi < NP; ++pi) {
                p[pi][0] = ex2(__fadd_rn(__fsub_rn(lh[pi][0], m_run[hb]), ll[pi][0]));
                p[pi][1] = ex2(__fadd_rn(__fsub_rn(lh[pi][1], m_run[hb]), ll[pi][1]));
            }
        }
#pragma unroll
        for (int pi = 0; pi < NP; ++pi) {
            l_run[hb] = __fadd_rn(l_run[hb], __fadd_rn(p[pi][0], p[pi][1]));
            const __half2* vsz = reinterpret_cast<const __half2*>(sb[pi] + GE::kSeg + GE::kCodeBytes);
#pragma unroll
            for (int gg = 0; gg < NG; ++gg) {
                const float2 s0 = __half22float2(vsz[gid * NG + gg]);
                const float2 s1 = __half22float2(vsz[(gid + 8) * NG + gg]);
                // p <= 2^8 and s_v <= (2/3) max T_v, and 2^sigma leaves that headroom, so
                // x <= 32752 (1 + tiny): fp16 without a clamp
                const float x0 = ok0 ? __fmul_rn(__fmul_rn(p[pi][0], s0.x), pvs) : 0.0f;
                const float x1 = ok1 ? __fmul_rn(__fmul_rn(p[pi][1], s1.x), pvs) : 0.0f;
                const __half h0 = __float2half_rn(x0), h1 = __float2half_rn(x1);
                Pv[pi][hb][gg][0] = pack_half2(h0, __float2half_rn(__fmul_rn(__fsub_rn(x0, __half2float(h0)), 2048.0f)));
                Pv[pi][hb][gg][1] = pack_half2(h1, __float2half_rn(__fmul_rn(__fsub_rn(x1, __half2float(h1)), 2048.0f)));
                if (ok0) zacc[hb][gg] = __fmaf_rn(p[pi][0], s0.y, zacc[hb][gg]);
                if (ok1) zacc[hb][gg] = __fmaf_rn(p[pi][1], s1.y, zacc[hb][gg]);
            }
        }
    }

    // ---- PV on tensor cores: A = V codes^T [16 channels x 16 tokens], B = p * s_v (hi, lo)
    // the (hi, lo) part this lane's B column needs: hi for even gid, lo for odd gid
    const uint32_t sel = (gid & 1) ? 0x7632u : 0x5410u;
    const int srcA = 8 * tig + (gid >> 1), srcB = srcA + 4;
#pragma unroll
    for (int pi = 0; pi < NP; ++pi) {
        uint32_t X01, Y01, X23, Y23;
        const uint8_t* vc = sb[pi] + GE::kSeg;
        if constexpr (D == 128) {
            const uint32_t wa = *reinterpret_cast<const uint32_t*>(vc + (2 * tig) * GE::kCodeRow + 4 * gid);
            const uint32_t wb = *reinterpret_cast<const uint32_t*>(vc + (2 * tig + 1) * GE::kCodeRow + 4 * gid);
            const uint32_t wc = *reinterpret_cast<const uint32_t*>(vc + (2 * tig + 8) * GE::kCodeRow + 4 * gid);
            const uint32_t wd = *reinterpret_cast<const uint32_t*>(vc + (2 * tig + 9) * GE::kCodeRow + 4 * gid);
            X01 = __byte_perm(wa, wb, 0x5410);
            Y01 = __byte_perm(wa, wb, 0x7632);
            X23 = __byte_perm(wc, wd, 0x5410);
            Y23 = __byte_perm(wc, wd, 0x7632);
        } else {
            const uint32_t wa = *reinterpret_cast<const uint16_t*>(vc + (2 * tig) * GE::kCodeRow + 2 * gid);
            const uint32_t wb = *reinterpret_cast<const uint16_t*>(vc + (2 * tig + 1) * GE::kCodeRow + 2 * gid);
            const uint32_t wc = *reinterpret_cast<const uint16_t*>(vc + (2 * tig + 8) * GE::kCodeRow + 2 * gid);
            const uint32_t wd = *reinterpret_cast<const uint16_t*>(vc + (2 * tig + 9) * GE::kCodeRow + 2 * gid);
            X01 = __byte_perm(wa, wb, 0x5410);
            X23 = __byte_perm(wc, wd, 0x5410);
            Y01 = X01;
            Y23 = X23;
        }
        const uint32_t X01s = X01 >> 10, Y01s = Y01 >> 10, X23s = X23 >> 10, Y23s = Y23 >> 10;
        uint32_t Bf[NHB][NG][2];
#pragma unroll
        for (int hb = 0; hb < NHB; ++hb)
#pragma unroll
            for (int gg = 0; gg < NG; ++gg) {
                const uint32_t a0 = __shfl_sync(0xffffffffu, Pv[pi][hb][gg][0], srcA);
                const uint32_t a1 = __shfl_sync(0xffffffffu, Pv[pi][hb][gg][1], srcA);
                const uint32_t b0 = __shfl_sync(0xffffffffu, Pv[pi][hb][gg][0], srcB);
                const uint32_t b1 = __shfl_sync(0xffffffffu, Pv[pi][hb][gg][1], srcB);
                Bf[hb][gg][0] = __byte_perm(a0, b0, sel);
                Bf[hb][gg][1] = __byte_perm(a1, b1, sel);
            }
        static_for<NK>([&](auto mc) {
            constexpr int mm = decltype(mc)::value;
            constexpr int gg = mm / KPG;
            uint32_t A0, A1, A2, A3;
            v_operand<D, mm>(X01, X01s, Y01, Y01s, X23, X23s, Y23, Y23s, A0, A1, A2, A3);
#pragma unroll
            for (int hb = 0; hb < NHB; ++hb) mma16816(O[hb][mm], A0, A1, A2, A3, Bf[hb][gg][0], Bf[hb][gg][1]);
        });
    }
}

// One INT2 page (16 tokens, the first `nvalid` valid) of one KV head, staged in shared memory at sb.
template <int D, int G, int GQ, bool FULL>
__device__ __forceinline__ void int2_page(const uint8_t* sb, int nvalid, int gid, int tig, float pvs,
                                          const QueryOps<D, G, GQ>& qo, WarpAcc<D, G, GQ>& acc) {
    const uint8_t* const one[1] = {sb};
    int2_pages<D, G, GQ, 1, FULL>(one, nvalid, gid, tig, pvs, qo, acc);
}

// K operand of the low-bit plane: b0 * 2^(2p'-24) per code, the same positions and scale as k_operand.
template <int POS>
__device__ __forceinline__ uint32_t low_bit_pair(uint32_t w, uint32_t w10) {
    if constexpr (POS <= 4) return w & (0x00010001u << (2 * POS));
    else return w10 & (0x00010001u << (2 * (POS - 5)));
}

template <int D, int KK>
__device__ __forceinline__ void k_operand_b0(const uint32_t (&kw0)[2], const uint32_t (&kw1)[2], uint32_t& A0,
                                             uint32_t& A1, uint32_t& A2, uint32_t& A3) {
    constexpr int W = KK / 4, P = 2 * (KK % 4);
    const uint32_t w0 = kw0[W], w1 = kw1[W];
    A0 = low_bit_pair<P>(w0, w0 >> 10); A1 = low_bit_pair<P>(w1, w1 >> 10);
    A2 = low_bit_pair<P + 1>(w0, w0 >> 10); A3 = low_bit_pair<P + 1>(w1, w1 >> 10);
}

// V operand of the Lloyd-Max codebook at position POS: (17.5 c + 1.5 b0) 2^(2p') as an exact normal
// fp16 pair, from c 2^(2p') (as code_pair_normal) and the fused 1.5 (1024 + b0 2^(2p')) - 1536.
template <int POS>
__device__ __forceinline__ uint32_t level_pair_normal(uint32_t w, uint32_t w10) {
    const uint32_t c = code_pair_normal<POS>(w, w10);
    const uint32_t hb = POS <= 4 ? and_or(w, 0x00010001u << (2 * POS), 0x64006400u)
                                 : and_or(w10, 0x00010001u << (2 * (POS - 5)), 0x64006400u);
    const __half2 b = __hfma2(*reinterpret_cast<const __half2*>(&hb), __float2half2_rn(1.5f), __float2half2_rn(-1536.0f));
    const __half2 r = __hfma2(*reinterpret_cast<const __half2*>(&c), __float2half2_rn(17.5f), b);
    return *reinterpret_cast<const uint32_t*>(&r);
}

template <int D, int MM>
__device__ __forceinline__ void v_operand_lm(uint32_t X01, uint32_t X01s, uint32_t Y01, uint32_t Y01s, uint32_t X23,
                                             uint32_t X23s, uint32_t Y23, uint32_t Y23s, uint32_t& A0, uint32_t& A1,
                                             uint32_t& A2, uint32_t& A3) {
    if constexpr (D == 128) {
        A0 = level_pair_normal<MM>(X01, X01s); A1 = level_pair_normal<MM>(Y01, Y01s);
        A2 = level_pair_normal<MM>(X23, X23s); A3 = level_pair_normal<MM>(Y23, Y23s);
    } else {
        A0 = level_pair_normal<MM>(X01, X01s); A1 = level_pair_normal<4 + MM>(X01, X01s);
        A2 = level_pair_normal<MM>(X23, X23s); A3 = level_pair_normal<4 + MM>(X23, X23s);
    }
}

// int2_page for the Lloyd-Max codebook: code c holds level l(c) = -27 + 17.5 c + 1.5 b0 (b0 the code's
// low bit) in units of the stored scale, k = zero + scale * l(c). Q.K runs on two exact planes, the
// codes (as in int2_page) and their low bits, each with its own accumulators:
//   q . k = scale * (17.5 q.c + 1.5 q.b0) + (zero - 27 scale) * sum(q).
// P.V takes A = (17.5 c + 1.5 b0) 2^(2p'), exact normal fp16 values (at most 54 * 2^8), and the
// zero-point sums use zero - 27 scale.
template <int D, int G, int GQ, bool FULL>
__device__ __forceinline__ void int2_page_lm(const uint8_t* sb, int nvalid, int gid, int tig, float pvs,
                                          const QueryOps<D, G, GQ>& qo, WarpAcc<D, G, GQ>& acc) {
    using GE = Geo<D, G>;
    constexpr int NK = D / 16, NG = D / G, KPG = G / 16, NHB = (GQ + 3) / 4;
    const auto& qB1 = qo.qB1;
    const auto& qB2 = qo.qB2;
    const auto& kap_h = qo.kap_h;
    const auto& kap_m = qo.kap_m;
    const auto& kap_l = qo.kap_l;
    const auto& qs_hi = qo.qs_hi;
    const auto& qs_lo = qo.qs_lo;
    auto& O = acc.O;
    auto& m_run = acc.m_run;
    auto& l_run = acc.l_run;
    auto& zacc = acc.zacc;
    const bool v0 = FULL || gid < nvalid, v1 = FULL || gid + 8 < nvalid;

    // ---- QK^T on tensor cores: A = K codes [16 tokens x 16 channels], B = query parts
    uint32_t kw0[2], kw1[2];
    if constexpr (D == 128) {
        const uint2 u0 = *reinterpret_cast<const uint2*>(sb + gid * GE::kCodeRow + 8 * tig);
        const uint2 u1 = *reinterpret_cast<const uint2*>(sb + (gid + 8) * GE::kCodeRow + 8 * tig);
        kw0[0] = u0.x; kw0[1] = u0.y; kw1[0] = u1.x; kw1[1] = u1.y;
    } else {
        kw0[0] = *reinterpret_cast<const uint32_t*>(sb + gid * GE::kCodeRow + 4 * tig);
        kw1[0] = *reinterpret_cast<const uint32_t*>(sb + (gid + 8) * GE::kCodeRow + 4 * tig);
        kw0[1] = kw1[1] = 0u;
    }
    float S1[NG][NHB][4], S2[NG][4], T1[NG][NHB][4], T2[NG][4];
#pragma unroll
    for (int gg = 0; gg < NG; ++gg) {
#pragma unroll
        for (int e = 0; e < 4; ++e) { S2[gg][e] = 0.0f; T2[gg][e] = 0.0f; }
#pragma unroll
        for (int hb = 0; hb < NHB; ++hb)
#pragma unroll
            for (int e = 0; e < 4; ++e) { S1[gg][hb][e] = 0.0f; T1[gg][hb][e] = 0.0f; }
    }
    static_for<NK>([&](auto kkc) {
        constexpr int kk = decltype(kkc)::value;
        uint32_t A0, A1, A2, A3, B0, B1, B2, B3;
        k_operand<D, kk>(kw0, kw1, A0, A1, A2, A3);
        k_operand_b0<D, kk>(kw0, kw1, B0, B1, B2, B3);
        constexpr int gg = kk / KPG;
#pragma unroll
        for (int hb = 0; hb < NHB; ++hb) {
            mma16816(S1[gg][hb], A0, A1, A2, A3, qB1[kk][hb][0], qB1[kk][hb][1]);
            mma16816(T1[gg][hb], B0, B1, B2, B3, qB1[kk][hb][0], qB1[kk][hb][1]);
        }
        mma16816(S2[gg], A0, A1, A2, A3, qB2[kk][0], qB2[kk][1]);
        mma16816(T2[gg], B0, B1, B2, B3, qB2[kk][0], qB2[kk][1]);
    });

    // ---- logits (hi + lo, log2 units) for tokens gid and gid+8 of head 4hb + tig
    const __half2* ksz = reinterpret_cast<const __half2*>(sb + GE::kCodeBytes);
    const __half2* vsz = reinterpret_cast<const __half2*>(sb + GE::kSeg + GE::kCodeBytes);
    uint32_t Pv[NHB][NG][2];     // p * s_v * 2^sigma per token slot, as (hi, lo) fp16 pair
#pragma unroll
    for (int hb = 0; hb < NHB; ++hb) {
        float lh[2], ll[2];
#pragma unroll
        for (int slot = 0; slot < 2; ++slot) {
            const int tok = gid + 8 * slot;
            float dh = 0.0f, dl = 0.0f;
#pragma unroll
            for (int gg = 0; gg < NG; ++gg) {
                const float lo_c = (GQ == 8) ? S2[gg][2 * slot + hb] : S2[gg][2 * slot];
                const float lo_b = (GQ == 8) ? T2[gg][2 * slot + hb] : T2[gg][2 * slot];
                // q.c and q.b0: exact hi parts (integers on the digit grid) and rounded low parts
                const float c_hi = __fmul_rn(S1[gg][hb][2 * slot], kap_h[hb]);
                const float c_r = __fmaf_rn(S1[gg][hb][2 * slot + 1], kap_m[hb], __fmul_rn(lo_c, kap_l[hb]));
                const float b_hi = __fmul_rn(T1[gg][hb][2 * slot], kap_h[hb]);
                const float b_r = __fmaf_rn(T1[gg][hb][2 * slot + 1], kap_m[hb], __fmul_rn(lo_b, kap_l[hb]));
                // y = 17.5 q.c + 1.5 q.b0 as y_hi + y_lo (1.5 b_hi is exact: b0 sums have one bit per code)
                float a1, ea, y_hi, ey;
                two_prod(17.5f, c_hi, a1, ea);
                two_sum(a1, __fmul_rn(1.5f, b_hi), y_hi, ey);
                const float y_lo = __fadd_rn(__fadd_rn(ea, ey), __fmaf_rn(17.5f, c_r, __fmul_rn(1.5f, b_r)));
                const float2 sz = __half22float2(ksz[tok * NG + gg]);
                // zero - 27 scale as zp_hi + zp_lo (27 scale is exact)
                float zp_hi, zp_lo;
                two_sum(sz.y, __fmul_rn(-27.0f, sz.x), zp_hi, zp_lo);
                float p1, e1, p2, e2, t1, e3;
                two_prod(sz.x, y_hi, p1, e1);
                two_prod(zp_hi, qs_hi[hb][gg], p2, e2);
                two_sum(p1, p2, t1, e3);
                const float low = __fadd_rn(__fadd_rn(__fadd_rn(e1, e2), e3),
                                            __fmaf_rn(sz.x, y_lo, __fmaf_rn(zp_hi, qs_lo[hb][gg],
                                                                            __fmul_rn(zp_lo, qs_hi[hb][gg]))));
                if (NG == 1) {
                    dh = t1;
                    dl = low;
                } else {
                    float t2, e4;
                    two_sum(dh, t1, t2, e4);
                    dh = t2;
                    dl = __fadd_rn(dl, __fadd_rn(low, e4));
                }
            }
            lh[slot] = dh;          // already in log2 units (the query carries the scale)
            ll[slot] = dl;
        }
        const bool hv = GQ % 4 == 0 || 4 * hb + tig < GQ;
        const bool ok0 = v0 && hv, ok1 = v1 && hv;
        if (!ok0) { lh[0] = -INFINITY; ll[0] = 0.0f; }
        if (!ok1) { lh[1] = -INFINITY; ll[1] = 0.0f; }
        // online softmax over the page (lanes sharing tig hold the same head). The reference is lazy:
        // raised only when a logit passes it by more than 2^kSoftmaxHeadroomLog2, so p <= 2^8 and the
        // O rescale is rare; only then is the page maximum of each head reduced across its lanes
        if (__any_sync(0xffffffffu, fmaxf(lh[0], lh[1]) > m_run[hb] + (float)kSoftmaxHeadroomLog2)) {
            float mp = fmaxf(lh[0], lh[1]);
            mp = fmaxf(mp, __shfl_xor_sync(0xffffffffu, mp, 4));
            mp = fmaxf(mp, __shfl_xor_sync(0xffffffffu, mp, 8));
            mp = fmaxf(mp, __shfl_xor_sync(0xffffffffu, mp, 16));
            const float mn = fmaxf(m_run[hb], mp);
            const float alpha = ex2(m_run[hb] - mn);
            m_run[hb] = mn;
            l_run[hb] *= alpha;
#pragma unroll
            for (int mm = 0; mm < NK; ++mm)
#pragma unroll
                for (int e = 0; e < 4; ++e) O[hb][mm][e] *= alpha;
#pragma unroll
            for (int gg = 0; gg < NG; ++gg) zacc[hb][gg] *= alpha;
        }
        const float p0 = ex2(__fadd_rn(__fsub_rn(lh[0], m_run[hb]), ll[0]));
        const float p1 = ex2(__fadd_rn(__fsub_rn(lh[1], m_run[hb]), ll[1]));
        l_run[hb] = __fadd_rn(l_run[hb], __fadd_rn(p0, p1));
#pragma unroll
        for (int gg = 0; gg < NG; ++gg) {
            const float2 s0 = __half22float2(vsz[gid * NG + gg]);
            const float2 s1 = __half22float2(vsz[(gid + 8) * NG + gg]);
            // p <= 2^8 and s_v <= (2/3) max T_v, and 2^sigma leaves that headroom, so
            // x <= 32752 (1 + tiny): fp16 without a clamp
            const float x0 = ok0 ? __fmul_rn(__fmul_rn(p0, s0.x), pvs) : 0.0f;
            const float x1 = ok1 ? __fmul_rn(__fmul_rn(p1, s1.x), pvs) : 0.0f;
            const __half h0 = __float2half_rn(x0), h1 = __float2half_rn(x1);
            Pv[hb][gg][0] = pack_half2(h0, __float2half_rn(__fmul_rn(__fsub_rn(x0, __half2float(h0)), 2048.0f)));
            Pv[hb][gg][1] = pack_half2(h1, __float2half_rn(__fmul_rn(__fsub_rn(x1, __half2float(h1)), 2048.0f)));
            if (ok0) zacc[hb][gg] = __fmaf_rn(p0, __fmaf_rn(-27.0f, s0.x, s0.y), zacc[hb][gg]);
            if (ok1) zacc[hb][gg] = __fmaf_rn(p1, __fmaf_rn(-27.0f, s1.x, s1.y), zacc[hb][gg]);
        }
    }

    // ---- PV on tensor cores: A = V codes^T [16 channels x 16 tokens], B = p * s_v (hi, lo)
    uint32_t X01, Y01, X23, Y23;
    const uint8_t* vc = sb + GE::kSeg;
    if constexpr (D == 128) {
        const uint32_t wa = *reinterpret_cast<const uint32_t*>(vc + (2 * tig) * GE::kCodeRow + 4 * gid);
        const uint32_t wb = *reinterpret_cast<const uint32_t*>(vc + (2 * tig + 1) * GE::kCodeRow + 4 * gid);
        const uint32_t wc = *reinterpret_cast<const uint32_t*>(vc + (2 * tig + 8) * GE::kCodeRow + 4 * gid);
        const uint32_t wd = *reinterpret_cast<const uint32_t*>(vc + (2 * tig + 9) * GE::kCodeRow + 4 * gid);
        X01 = __byte_perm(wa, wb, 0x5410);
        Y01 = __byte_perm(wa, wb, 0x7632);
        X23 = __byte_perm(wc, wd, 0x5410);
        Y23 = __byte_perm(wc, wd, 0x7632);
    } else {
        const uint32_t wa = *reinterpret_cast<const uint16_t*>(vc + (2 * tig) * GE::kCodeRow + 2 * gid);
        const uint32_t wb = *reinterpret_cast<const uint16_t*>(vc + (2 * tig + 1) * GE::kCodeRow + 2 * gid);
        const uint32_t wc = *reinterpret_cast<const uint16_t*>(vc + (2 * tig + 8) * GE::kCodeRow + 2 * gid);
        const uint32_t wd = *reinterpret_cast<const uint16_t*>(vc + (2 * tig + 9) * GE::kCodeRow + 2 * gid);
        X01 = __byte_perm(wa, wb, 0x5410);
        X23 = __byte_perm(wc, wd, 0x5410);
        Y01 = X01;
        Y23 = X23;
    }
    const uint32_t X01s = X01 >> 10, Y01s = Y01 >> 10, X23s = X23 >> 10, Y23s = Y23 >> 10;
    // the (hi, lo) part this lane's B column needs: hi for even gid, lo for odd gid
    const uint32_t sel = (gid & 1) ? 0x7632u : 0x5410u;
    const int srcA = 8 * tig + (gid >> 1), srcB = srcA + 4;
    uint32_t Bf[NHB][NG][2];
#pragma unroll
    for (int hb = 0; hb < NHB; ++hb)
#pragma unroll
        for (int gg = 0; gg < NG; ++gg) {
            const uint32_t a0 = __shfl_sync(0xffffffffu, Pv[hb][gg][0], srcA);
            const uint32_t a1 = __shfl_sync(0xffffffffu, Pv[hb][gg][1], srcA);
            const uint32_t b0 = __shfl_sync(0xffffffffu, Pv[hb][gg][0], srcB);
            const uint32_t b1 = __shfl_sync(0xffffffffu, Pv[hb][gg][1], srcB);
            Bf[hb][gg][0] = __byte_perm(a0, b0, sel);
            Bf[hb][gg][1] = __byte_perm(a1, b1, sel);
        }
    static_for<NK>([&](auto mc) {
        constexpr int mm = decltype(mc)::value;
        constexpr int gg = mm / KPG;
        uint32_t A0, A1, A2, A3;
        v_operand_lm<D, mm>(X01, X01s, Y01, Y01s, X23, X23s, Y23, Y23s, A0, A1, A2, A3);
#pragma unroll
        for (int hb = 0; hb < NHB; ++hb) mma16816(O[hb][mm], A0, A1, A2, A3, Bf[hb][gg][0], Bf[hb][gg][1]);
    });
}

// The page body of the context's codebook.
// The page body of the context's codebook; FULL: all 16 tokens of the page are valid.
template <int D, int G, int GQ, int CB, bool FULL>
__device__ __forceinline__ void page_body(const uint8_t* sb, int nvalid, int gid, int tig, float pvs,
                                          const QueryOps<D, G, GQ>& qo, WarpAcc<D, G, GQ>& acc) {
    if constexpr (CB == OSCAR_CODEBOOK_LLOYD_MAX) int2_page_lm<D, G, GQ, FULL>(sb, nvalid, gid, tig, pvs, qo, acc);
    else int2_page<D, G, GQ, FULL>(sb, nvalid, gid, tig, pvs, qo, acc);
}

// Streams this warp's pages (first + kWarps j, j < n_mine) of one (sequence, KV head, split) through
// shared memory: kSlots slots of two pages, every lane copying its 16-byte chunks of a page with
// cp.async, one commit group per slot, so waiting for all but the kSlots - 1 newest groups completes
// the oldest slot. prologue() runs once the first copies are in flight; pair(stage0, stage1) takes two
// full pages with valid ids (all but the warp's last pair, normally, after one uniform test), and
// body(stage, nvalid) any other page with a valid id.
template <int D, int G, typename Pro, typename Pair, typename Body>
__device__ __forceinline__ void page_loop(const SplitArgs& a, int kv, int len, int first, int n_mine,
                                          const int32_t* table, uint8_t* stage_base, Pro&& prologue, Pair&& pair,
                                          Body&& body) {
    using GE = Geo<D, G>;
    constexpr int kChunks = GE::kBlock / 16;                 // 16-byte chunks per page block
    constexpr int kPerLane = (kChunks + 31) / 32;
    constexpr uint32_t kSlotBytes = 2 * GE::kBlock;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    uint8_t* my_stage = stage_base + (size_t)warp * kSlots * kSlotBytes;
    const uint32_t stage_s = (uint32_t)__cvta_generic_to_shared(my_stage) + 16 * lane;
    const uint8_t* const pool_kv = a.int2_pool + (size_t)kv * GE::kBlock + 16 * lane;
    const uint32_t page_stride = (uint32_t)a.h_kv * GE::kBlock;
    const bool tail_lane = kChunks % 32 == 0 || lane < kChunks % 32;   // copies the page's last chunk row
    const int n_pairs = (n_mine + 1) / 2;
    // pages j < j_full hold 16 tokens; only the sequence's last page can be shorter
    const int j_full = (n_mine > 0 && first + kWarps * (n_mine - 1) == (len - 1) / kPage && len % kPage != 0)
                           ? n_mine - 1 : n_mine;
    // page ids, 32 at a time across the lanes: chunk c (pages 32c .. 32c+31 of the warp) lives in
    // ids[c & 1], loaded two chunks ahead; when its first pair is issued the chunk is checked once
    // (out-of-range ids become invalid pages, recorded in debug mode) and vm[c & 1] holds its ballot
    int32_t ids0 = lane < n_mine ? table[first + kWarps * lane] : -1;
    int32_t ids1 = lane + 32 < n_mine ? table[first + kWarps * (lane + 32)] : -1;
    uint32_t vm0 = 0u, vm1 = 0u;
    uint32_t valid_bits = 0u;                               // bits 2s, 2s+1: the pages of slot s are real
    auto check_chunk = [&](int c, int32_t& ids, uint32_t& vm) {
        const bool ok = ids >= 0 && (int64_t)ids < a.int2_pages;
        if (a.debug && !ok && 32 * c + lane < n_mine) record_error(&a.dbg->kind, &a.dbg->index, 2, ids);
        vm = __ballot_sync(0xffffffffu, ok);
        ids = ok ? ids : 0;
    };
    auto copy_page = [&](uint32_t dst, int32_t phys) {
        const uint8_t* src = pool_kv + (size_t)((uint32_t)phys * page_stride);
#pragma unroll
        for (int k = 0; k < kPerLane; ++k) cp_async16(dst + 512 * k, src + 512 * k, k + 1 < kPerLane || tail_lane);
    };
    // pages 2i and 2i+1 of the warp into slot s (both in one chunk of ids: 2i is even)
    auto issue = [&](int i, int s) {
        const int j0 = 2 * i;
        const bool odd_chunk = (j0 >> 5) & 1;
        if ((j0 & 31) == 0) {
            if (odd_chunk) check_chunk(j0 >> 5, ids1, vm1); else check_chunk(j0 >> 5, ids0, vm0);
        }
        const int32_t cur = odd_chunk ? ids1 : ids0;
        const uint32_t vb = ((odd_chunk ? vm1 : vm0) >> (j0 & 31)) & 3u;
        const int32_t p0 = __shfl_sync(0xffffffffu, cur, j0 & 31);
        const int32_t p1 = __shfl_sync(0xffffffffu, cur, (j0 & 31) + 1);
        valid_bits = (valid_bits & ~(3u << (2 * s))) | (vb << (2 * s));
        const uint32_t dst = stage_s + s * kSlotBytes;
        if (vb & 1u) copy_page(dst, p0);
        if (vb & 2u) copy_page(dst + GE::kBlock, p1);
        cp_async_commit();
    };
    for (int i = 0; i < kSlots; ++i) {
        if (i < n_pairs) issue(i, i);
        else cp_async_commit();              // empty group: the wait count stays uniform
    }
    prologue();
    int slot = 0;
    for (int i = 0; i < n_pairs; ++i) {
        cp_async_wait<kSlots - 1>();         // this lane's copies of pair i have landed
        __syncwarp();                        // ... and every other lane's
        const uint8_t* sb = my_stage + slot * kSlotBytes;
        const uint32_t vb = (valid_bits >> (2 * slot)) & 3u;
        if (vb == 3u && 2 * i + 1 < j_full) {
            pair(sb, sb + GE::kBlock);
        } else {
#pragma unroll 1
            for (int e = 0; e < 2; ++e)
                if (vb & (1u << e)) {
                    // tokens of this page in the sequence (1..16)
                    const int nv = min(kPage, len - (first + kWarps * (2 * i + e)) * kPage);
                    body(sb + e * GE::kBlock, nv);
                }
        }
        __syncwarp();                        // every lane is done reading the slot before it is refilled
        if (i + kSlots < n_pairs) {
            const int ii = i + kSlots;
            issue(ii, slot);
            if (((2 * ii + 1) & 31) == 31) {      // chunk (2ii+1)/32 fully issued: load chunk + 2 into its slot
                const int nj = 2 * ii + 1 + 33 + lane;
                const int32_t v = nj < n_mine ? table[first + kWarps * nj] : -1;
                if (((2 * ii + 1) >> 5) & 1) ids1 = v; else ids0 = v;
            }
        } else {
            cp_async_commit();
        }
        if (++slot == kSlots) slot = 0;
    }
    cp_async_wait<0>();
}

// INT2 history split on tensor cores. Writes this warp's state into acc_s / ml_s.
template <int D, int G, int GQ, int CB>
__device__ void int2_split(const SplitArgs& a, int split, int kv, int b, uint8_t* stage_base, float* acc_s,
                           float (*ml_s)[GQ][2]) {
    constexpr int NK = D / 16;          // k-steps (QK) = m-steps (PV)
    constexpr int NG = D / G;
    constexpr int KPG = G / 16;         // k-steps per group
    constexpr int NHB = (GQ + 3) / 4;   // blocks of 4 query heads
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int gid = lane >> 2, tig = lane & 3;
    const int h_q = a.h_kv * GQ;
    const size_t head0 = (size_t)b * h_q + kv * GQ;

    int len = a.hist_len[b];
    const int cap = min(a.max_hist, a.int2_stride * kPage);
    if (len < 0 || len > cap) {
        if (a.debug && threadIdx.x == 0) record_error(&a.dbg->kind, &a.dbg->index, 3, len);
        len = len < 0 ? 0 : cap;
    }
    const int n_pages = (len + kPage - 1) / kPage;
    const int pg0 = split * a.pages_per_split;
    const int pg1 = min(n_pages, pg0 + a.pages_per_split);
    const int first = pg0 + warp;
    const int n_mine = first < pg1 ? (pg1 - first + kWarps - 1) / kWarps : 0;
    const int32_t* table = a.int2_tables + (size_t)b * a.int2_stride;

    {
        WarpAcc<D, G, GQ> acc;
        acc.init();
        auto& O = acc.O;
        auto& m_run = acc.m_run;
        auto& l_run = acc.l_run;
        auto& zacc = acc.zacc;
        QueryOps<D, G, GQ> qo;
        float pvs = 1.0f, inv_pvs = 1.0f;
        page_loop<D, G>(
            a, kv, len, first, n_mine, table, stage_base,
            [&] {
                pdl_wait();
                pdl_trigger();
                load_query_ops<D, G, GQ>(a, head0, gid, tig, qo);
                pvs = a.pv_scale[kv];
                inv_pvs = 1.0f / pvs;
            },
            [&](const uint8_t* sb0, const uint8_t* sb1) {
                if constexpr (CB == OSCAR_CODEBOOK_LLOYD_MAX || GQ == 8) {
                    // one page at a time: two pages' state does not fit beside these bodies' registers
#pragma unroll 1
                    for (int e = 0; e < 2; ++e)
                        page_body<D, G, GQ, CB, true>(e ? sb1 : sb0, kPage, gid, tig, pvs, qo, acc);
                } else {
                    const uint8_t* const two[2] = {sb0, sb1};
                    int2_pages<D, G, GQ, 2, true>(two, kPage, gid, tig, pvs, qo, acc);
                }
            },
            [&](const uint8_t* sb, int nv) { page_body<D, G, GQ, CB, false>(sb, nv, gid, tig, pvs, qo, acc); });

        // ---- this warp's state -> shared memory (scaled to the CTA max)
#pragma unroll
        for (int hb = 0; hb < NHB; ++hb) {
            float l = l_run[hb];
            l += __shfl_xor_sync(0xffffffffu, l, 4);
            l += __shfl_xor_sync(0xffffffffu, l, 8);
            l += __shfl_xor_sync(0xffffffffu, l, 16);
            l_run[hb] = l;
#pragma unroll
            for (int gg = 0; gg < NG; ++gg) {
                float z = zacc[hb][gg];
                z += __shfl_xor_sync(0xffffffffu, z, 4);
                z += __shfl_xor_sync(0xffffffffu, z, 8);
                z += __shfl_xor_sync(0xffffffffu, z, 16);
                zacc[hb][gg] = z;
            }
            const int h = 4 * hb + tig;
            if (h < GQ && gid == 0) { ml_s[warp][h][0] = m_run[hb]; ml_s[warp][h][1] = l_run[hb]; }
        }
        __syncthreads();
#pragma unroll
        for (int hb = 0; hb < NHB; ++hb) {
            const int h = 4 * hb + tig;
            if (h >= GQ) continue;
            float mm_ = -INFINITY;
#pragma unroll
            for (int w2 = 0; w2 < kWarps; ++w2) mm_ = fmaxf(mm_, ml_s[w2][h][0]);
            const float f = m_run[hb] <= kNoMax ? 0.0f : fast_exp2(m_run[hb] - mm_);
            if (f == 0.0f) continue;
#pragma unroll
            for (int mm = 0; mm < NK; ++mm) {
                const int gg = mm / KPG;
                // rows gid and gid+8 of m-step mm carry 2^(2p') of their code position and 2^sigma
                const int pos0 = mm;
                const int pos1 = (D == 128) ? mm : 4 + mm;
                const float sc0 = pos_weight(pos0) * inv_pvs;
                const float sc1 = pos_weight(pos1) * inv_pvs;
                const float o0 = __fmaf_rn(O[hb][mm][1], 0x1p-11f, O[hb][mm][0]) * sc0 + zacc[hb][gg];
                const float o1 = __fmaf_rn(O[hb][mm][3], 0x1p-11f, O[hb][mm][2]) * sc1 + zacc[hb][gg];
                atomicAdd(&acc_s[h * D + 16 * mm + gid], o0 * f);
                atomicAdd(&acc_s[h * D + 16 * mm + gid + 8], o1 * f);
            }
        }
    }
}

// Shared-prefix split: prefix pages [pg0, pg1) of one KV head for a group of kWarps sequences
// (warp w serves sequence kWarps * sg + w). Each page is copied once into the CTA's ring of
// kWarps * kStages stages and read by every warp, so the prefix crosses HBM once per group rather than
// once per sequence. Thread 0 issues the copies; a stage is refilled once all warps have released it
// (an mbarrier with one arrival per warp). Every wait is bounded. Each warp writes the partial of its
// own sequence's query heads to slot ps.
template <int D, int G, int GQ, int CB>
__device__ void prefix_split(const SplitArgs& a, int ps, int kv, int sg, uint8_t* stage_base, uint64_t* bars) {
    using GE = Geo<D, G>;
    constexpr int NK = D / 16, NG = D / G, KPG = G / 16, NHB = (GQ + 3) / 4;
    constexpr int S = kWarps * kStages;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int gid = lane >> 2, tig = lane & 3;
    const int h_q = a.h_kv * GQ;
    const int b = sg * kWarps + warp;
    const bool active = b < a.batch;
    const int pg0 = ps * a.prefix_pages_per_split;
    const int n = max(0, min(a.prefix_pages, pg0 + a.prefix_pages_per_split) - pg0);
    const uint32_t stage_s = (uint32_t)__cvta_generic_to_shared(stage_base);
    const uint32_t full_s = (uint32_t)__cvta_generic_to_shared(bars);     // S barriers: page landed
    const uint32_t empty_s = full_s + 8 * S;                                // S barriers: all warps done
    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(full_s + 8 * i, 1);
            mbar_init(empty_s + 8 * i, kWarps);
        }
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const uint8_t* const pool_kv = a.int2_pool + (size_t)kv * GE::kBlock;
    const size_t page_stride = (size_t)a.h_kv * GE::kBlock;
    const int32_t* table = a.prefix_table + pg0;
    int issued = 0;                                  // thread 0: pages copied (or marked) so far
    auto issue = [&](int i) {
        const int st = i % S;
        const int32_t phys = table[i];
        if (phys >= 0 && phys < a.int2_pages) {
            bulk_load(stage_s + st * GE::kBlock, pool_kv + (size_t)phys * page_stride, GE::kBlock, full_s + 8 * st);
        } else {
            if (a.debug) record_error(&a.dbg->kind, &a.dbg->index, 2, phys);
            mbar_arrive(full_s + 8 * st);
        }
        issued = i + 1;
    };
    if (threadIdx.x == 0)
        for (int i = 0; i < S && i < n; ++i) issue(i);

    // the query operands come from q_prep: wait for it (the first copies are already in flight)
    pdl_wait();
    pdl_trigger();
    QueryOps<D, G, GQ> qo;
    WarpAcc<D, G, GQ> acc;
    acc.init();
    const size_t head0 = (size_t)(active ? b : 0) * h_q + kv * GQ;
    if (active) load_query_ops<D, G, GQ>(a, head0, gid, tig, qo);
    const float pvs = a.pv_scale[kv];

    bool failed = false;
    int i = 0;
    for (; i < n; ++i) {
        const int st = i % S;
        const uint32_t phase = (i / S) & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(full_s + 8 * st, phase))) {
            failed = true;
            break;
        }
        const int32_t phys = table[i];
        if (active && phys >= 0 && phys < a.int2_pages)
            page_body<D, G, GQ, CB, true>(stage_base + (size_t)st * GE::kBlock, kPage, gid, tig, pvs, qo, acc);
        __syncwarp();
        if (lane == 0) mbar_arrive(empty_s + 8 * st);
        if (threadIdx.x == 0 && i + S < n) {
            // the stage is reused once every warp has released page i
            if (mbar_wait(empty_s + 8 * st, phase)) issue(i + S);
            else record_error(&a.dbg->kind, &a.dbg->index, 4, pg0 + i);
        }
    }
    if (failed && lane == 0) record_error(&a.dbg->kind, &a.dbg->index, 4, pg0 + i);
    if (threadIdx.x == 0) {
        // copies still in flight land before the CTA (and its shared memory) goes away (bounded)
        for (int j = i; j < issued; ++j) (void)mbar_wait(full_s + 8 * (j % S), (j / S) & 1);
    }
    if (!active) return;
    auto& O = acc.O;
    auto& m_run = acc.m_run;
    auto& l_run = acc.l_run;
    auto& zacc = acc.zacc;
    if (failed) {
#pragma unroll
        for (int hb = 0; hb < NHB; ++hb) { m_run[hb] = -INFINITY; l_run[hb] = 0.0f; }
    }
    // ---- this warp's partial: m = its running max, l and acc relative to it
    const float inv_pvs = 1.0f / pvs;
#pragma unroll
    for (int hb = 0; hb < NHB; ++hb) {
        float l = l_run[hb];
        l += __shfl_xor_sync(0xffffffffu, l, 4);
        l += __shfl_xor_sync(0xffffffffu, l, 8);
        l += __shfl_xor_sync(0xffffffffu, l, 16);
        float z[NG];
#pragma unroll
        for (int gg = 0; gg < NG; ++gg) {
            z[gg] = zacc[hb][gg];
            z[gg] += __shfl_xor_sync(0xffffffffu, z[gg], 4);
            z[gg] += __shfl_xor_sync(0xffffffffu, z[gg], 8);
            z[gg] += __shfl_xor_sync(0xffffffffu, z[gg], 16);
        }
        const int h = 4 * hb + tig;
        if (h >= GQ) continue;
        float* dst = a.partials + (((size_t)b * h_q + kv * GQ + h) * a.total_splits + ps) * (D + 2);
        if (gid == 0) {
            dst[0] = m_run[hb];
            dst[1] = l;
        }
#pragma unroll
        for (int mm = 0; mm < NK; ++mm) {
            const int gg = mm / KPG;
            const float sc0 = pos_weight(mm) * inv_pvs;
            const float sc1 = pos_weight((D == 128) ? mm : 4 + mm) * inv_pvs;
            dst[2 + 16 * mm + gid] = __fmaf_rn(O[hb][mm][1], 0x1p-11f, O[hb][mm][0]) * sc0 + z[gg];
            dst[2 + 16 * mm + gid + 8] = __fmaf_rn(O[hb][mm][3], 0x1p-11f, O[hb][mm][2]) * sc1 + z[gg];
        }
    }
}

// Online-softmax update for one page of 16 tokens held one token per lane
// (lanes t and t+16 carry the same logit). Logits arrive as hi + lo.
template <int GQ>
__device__ __forceinline__ void softmax_page(float (&lg)[GQ], float (&lgl)[GQ], float (&m)[GQ], float (&l)[GQ],
                                             float (&alpha)[GQ], float (&p)[GQ]) {
#pragma unroll
    for (int h = 0; h < GQ; ++h) {
        float mp = lg[h];
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) mp = fmaxf(mp, __shfl_xor_sync(0xffffffffu, mp, o));
        const float mn = fmaxf(m[h], mp);
        if (mn == -INFINITY) {
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

// BF16 sink/recent split on CUDA cores (<= 320 tokens per sequence).
template <int D, int GQ>
__device__ void bf16_split(const SplitArgs& a, int split, int kv, int b, float* qs, float (*p_s)[16][GQ],
                           float* acc_s, float (*ml_s)[GQ][2]) {
    constexpr int CPL = D / 32;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int t = lane & 15, hf = lane >> 4;
    const int h_q = a.h_kv * GQ;
    for (int i = threadIdx.x; i < GQ * D; i += blockDim.x)
        qs[i] = __bfloat162float(a.q[((size_t)b * h_q + kv * GQ) * D + i]);
    __syncthreads();
    float m[GQ], l[GQ];
#pragma unroll
    for (int h = 0; h < GQ; ++h) { m[h] = -INFINITY; l[h] = 0.0f; }
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
        const int tmax = min(kPage, len - pg * kPage);
        // the page's V rows (CPL channels of every token per lane) are requested now, so they arrive
        // while the logits and the softmax are computed
        uint32_t vraw[kPage][CPL / 2];
#pragma unroll
        for (int tt = 0; tt < kPage; ++tt) {
            if (tt < tmax) {
                if constexpr (CPL == 4) {
                    const uint2 u = *reinterpret_cast<const uint2*>(vp + tt * D + 4 * lane);
                    vraw[tt][0] = u.x;
                    vraw[tt][1] = u.y;
                } else {
                    vraw[tt][0] = *reinterpret_cast<const uint32_t*>(vp + tt * D + 2 * lane);
                }
            } else {
#pragma unroll
                for (int j = 0; j < CPL / 2; ++j) vraw[tt][j] = 0u;
            }
        }
        float lg[GQ];
#pragma unroll
        for (int h = 0; h < GQ; ++h) lg[h] = 0.0f;
        const __nv_bfloat16* krow = kp + t * D + hf * (D / 2);
        uint4 ku[D / 16];
#pragma unroll
        for (int c8 = 0; c8 < D / 16; ++c8) ku[c8] = *reinterpret_cast<const uint4*>(krow + 8 * c8);
#pragma unroll
        for (int c8 = 0; c8 < D / 16; ++c8) {
            const __nv_bfloat162* k2 = reinterpret_cast<const __nv_bfloat162*>(&ku[c8]);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 kf = __bfloat1622float2(k2[e]);
                const int c = hf * (D / 2) + 8 * c8 + 2 * e;
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
#pragma unroll
        for (int tt = 0; tt < kPage; ++tt) {
            if (tt >= tmax) break;
            float v[CPL];
#pragma unroll
            for (int j = 0; j < CPL / 2; ++j) {
                const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&vraw[tt][j]));
                v[2 * j] = f.x;
                v[2 * j + 1] = f.y;
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

// Online-softmax merge of one (sequence, KV head)'s splits, run by the CTA that finishes last
// (GQ * total_splits <= kFuseWeights): per query head, weights 2^(m_s - M) over the split partials,
// the INT2 splits' sum un-rotated by R_v^T, plus the BF16 split, over L. w_s (the page-stage shared
// memory) holds GQ * total_splits floats. Records written by other CTAs are read through L2
// (ld.global.cg), never from a possibly stale L1 line; loads are batched so that each round has
// many in flight.
template <int D, int GQ>
__device__ __noinline__ void merge_group(const SplitArgs& a, int kv, int b, float* acc_s, float* w_s) {
    __shared__ float l_s[GQ];
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
    const int h_q = a.h_kv * GQ, T = a.total_splits;
    const float* part0 = a.partials + (size_t)(b * h_q + kv * GQ) * T * (D + 2);
    for (int h = warp; h < GQ; h += kWarps) {
        const float* part = part0 + (size_t)h * T * (D + 2);
        float m[kFuseWeights / 32], l[kFuseWeights / 32];
        float M = -INFINITY;
#pragma unroll
        for (int k = 0; k < kFuseWeights / 32; ++k) {
            const int sp = lane + 32 * k;
            m[k] = sp < T ? __ldcg(part + (size_t)sp * (D + 2)) : -INFINITY;
            l[k] = sp < T ? __ldcg(part + (size_t)sp * (D + 2) + 1) : 0.0f;
            M = fmaxf(M, m[k]);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        float L = 0.0f;
#pragma unroll
        for (int k = 0; k < kFuseWeights / 32; ++k) {
            const int sp = lane + 32 * k;
            const float w = (M == -INFINITY || m[k] == -INFINITY) ? 0.0f : fast_exp2(m[k] - M);
            if (sp < T) w_s[h * T + sp] = w;
            L = fmaf(l[k], w, L);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
        if (lane == 0) l_s[h] = L;
    }
    __syncthreads();
    const int c = tid;
    float ab[GQ];
#pragma unroll
    for (int h = 0; h < GQ; ++h) {
        float ai = 0.0f;
        ab[h] = 0.0f;
        if (c < D) {
            const float* part = part0 + (size_t)h * T * (D + 2) + 2 + c;
            for (int s0 = 0; s0 < T; s0 += 16) {
                float v[16];
#pragma unroll
                for (int k = 0; k < 16; ++k) v[k] = s0 + k < T ? __ldcg(part + (size_t)(s0 + k) * (D + 2)) : 0.0f;
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const int sp = s0 + k;
                    if (sp >= T) break;
                    const float x = v[k] * w_s[h * T + sp];
                    if (sp < a.prefix_splits + a.int2_splits) ai += x; else ab[h] += x;
                }
            }
            acc_s[h * D + c] = ai;
        }
    }
    __syncthreads();
    if (c < D) {
        float o[GQ];
#pragma unroll
        for (int h = 0; h < GQ; ++h) o[h] = 0.0f;
        const float* rt = a.r_vt + (size_t)kv * D * D + c;
        for (int i0 = 0; i0 < D; i0 += 16) {
            float r[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) r[i] = __ldg(rt + (size_t)(i0 + i) * D);
#pragma unroll
            for (int i = 0; i < 16; ++i)
#pragma unroll
                for (int h = 0; h < GQ; ++h) o[h] = fmaf(acc_s[h * D + i0 + i], r[i], o[h]);
        }
#pragma unroll
        for (int h = 0; h < GQ; ++h) {
            const float L = l_s[h];
            a.out[((size_t)b * h_q + kv * GQ + h) * D + c] = L > 0.0f ? (o[h] + ab[h]) / L : 0.0f;
        }
    }
}

// Resident CTAs per SM the split kernel is compiled for: 3 (168 registers) for the uniform codebook. The
// two-page body wants about 157 registers; at 4 CTAs (128) it is squeezed, and at bs1 the longer splits
// of a 3-CTA wave also spread each warp's fixed costs over more pages (33.5 against 35.4 us per layer;
// batch 64 within 1 %). The Lloyd-Max body holds a second set of Q.K accumulators.
__host__ __device__ constexpr int split_min_blocks(int gq, int cb) {
    return cb == OSCAR_CODEBOOK_LLOYD_MAX ? (gq == 8 ? 2 : 3) : 3;
}

template <int D, int G, int GQ, int CB>
__global__ void __launch_bounds__(kWarps * 32, split_min_blocks(GQ, CB))
split_kernel(SplitArgs a) {
    extern __shared__ __align__(128) uint8_t dyn_smem[];
    __shared__ __align__(8) uint64_t bars[2 * kWarps * kStages];
    __shared__ __align__(16) float acc_s[GQ * D];
    __shared__ float ml_s[kWarps][GQ][2];
    __shared__ float p_s[kWarps][16][GQ];

    // flat grid: the shared-prefix CTAs (prefix split fastest, then KV head, then sequence group),
    // then one CTA per (split, KV head, sequence), split fastest
    const int cta = blockIdx.x;
    if (cta < a.n_prefix_ctas) {
        const int ps = cta % a.prefix_splits, rest = cta / a.prefix_splits;
        prefix_split<D, G, GQ, CB>(a, ps, rest % a.h_kv, rest / a.h_kv, dyn_smem, bars);
        return;
    }
    const int reg = cta - a.n_prefix_ctas;
    const int t_reg = a.int2_splits + a.bf16_splits;
    const int split = reg % t_reg, kv = (reg / t_reg) % a.h_kv, b = reg / t_reg / a.h_kv;
    const int h_q = a.h_kv * GQ;
    for (int i = threadIdx.x; i < GQ * D; i += blockDim.x) acc_s[i] = 0.0f;
    __syncthreads();

    if (split < a.int2_splits) {
        int2_split<D, G, GQ, CB>(a, split, kv, b, dyn_smem, acc_s, ml_s);
    } else {
        pdl_wait();
        pdl_trigger();
        bf16_split<D, GQ>(a, split, kv, b, reinterpret_cast<float*>(dyn_smem), p_s, acc_s, ml_s);
    }
    __syncthreads();

    // ---- the partial of each query head of the group
    for (int h = 0; h < GQ; ++h) {
        float mm = -INFINITY;
        for (int w2 = 0; w2 < kWarps; ++w2) mm = fmaxf(mm, ml_s[w2][h][0]);
        float ll = 0.0f;
        for (int w2 = 0; w2 < kWarps; ++w2) {
            const float mw = ml_s[w2][h][0];
            if (mw != -INFINITY) ll += ml_s[w2][h][1] * fast_exp2(mw - mm);
        }
        float* dst = a.partials + (((size_t)b * h_q + kv * GQ + h) * a.total_splits + a.prefix_splits + split) * (D + 2);
        for (int c = threadIdx.x; c < D; c += blockDim.x) dst[2 + c] = acc_s[h * D + c];
        if (threadIdx.x == 0) { dst[0] = mm; dst[1] = ll; }
    }
    if (a.fuse_merge) {
        // the last CTA of this (sequence, KV head) to finish merges all of its splits
        __shared__ int ticket_s;
        __syncthreads();
        if (threadIdx.x == 0) {
            __threadfence();
            ticket_s = atomicAdd(a.counters + (size_t)b * a.h_kv + kv, 1);
        }
        __syncthreads();
        if (ticket_s == t_reg - 1) {
            __threadfence();
            merge_group<D, GQ>(a, kv, b, acc_s, reinterpret_cast<float*>(dyn_smem));
        }
    }
}

// Merge of all splits of one query head (plans with long merges: one wave of few units, or many
// splits). Block of 4*D threads: thread (c, quarter) takes the splits s = quarter + 4k for channel c,
// kPer of them per round with every load of the round in flight at once, and a quarter of the
// un-rotation terms, which load before the wait for the split kernel.
template <int D>
__global__ void __launch_bounds__(4 * D)
merge_kernel(const float* __restrict__ partials, const float* __restrict__ r_vt, float* __restrict__ out, int h_q,
             int g, int int2_splits, int total_splits) {
    constexpr int kPer = 24;                 // 96 splits per round: one round at bs1 (79 splits)
    __shared__ float red_m[4], red_l[4];
    __shared__ float acc_rot[D];
    __shared__ float part_i[4][D], part_b[4][D];
    const int bh = blockIdx.x;
    const int kv = (bh % h_q) / g;
    const int tid = threadIdx.x, c = tid % D, quarter = tid / D;
    const float* rt = r_vt + (size_t)kv * D * D + (size_t)quarter * (D / 4) * D + c;
    float rv[D / 4];
#pragma unroll
    for (int i = 0; i < D / 4; ++i) rv[i] = __ldg(rt + (size_t)i * D);
    pdl_wait();
    pdl_trigger();
    const float* part = partials + (size_t)bh * total_splits * (D + 2);
    const int lane = tid % 32;
    float M = -INFINITY, L = 0.0f, ai = 0.0f, ab = 0.0f;
    for (int s0 = 0; s0 < total_splits; s0 += 4 * kPer) {
        // the quarter's splits s0 + 4k + quarter: lane k of each warp loads split k's (m, l) (the same
        // for every channel), every thread its channel's accumulator of each split
        float m_k = -INFINITY, l_k = 0.0f;
        {
            const int sp = s0 + 4 * lane + quarter;
            if (lane < kPer && sp < total_splits) {
                const float* r = part + (size_t)sp * (D + 2);
                m_k = __ldcg(r);
                l_k = __ldcg(r + 1);
            }
        }
        float as[kPer];
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int sp = s0 + 4 * k + quarter;
            as[k] = sp < total_splits ? __ldcg(part + (size_t)sp * (D + 2) + 2 + c) : 0.0f;
        }
        float mloc = m_k;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, o));
        if (c == 0) red_m[quarter] = mloc;
        __syncthreads();
        const float mn = fmaxf(M, fmaxf(fmaxf(red_m[0], red_m[1]), fmaxf(red_m[2], red_m[3])));
        const float sc = M == -INFINITY ? 0.0f : fast_exp2(M - mn);
        ai *= sc;
        ab *= sc;
        L *= sc;
        const float w_k = m_k == -INFINITY ? 0.0f : fast_exp2(m_k - mn);
        float lw = l_k * w_k;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) lw += __shfl_xor_sync(0xffffffffu, lw, o);
        L += lw;
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int sp = s0 + 4 * k + quarter;
            const float w = __shfl_sync(0xffffffffu, w_k, k);
            if (sp < int2_splits) ai = fmaf(as[k], w, ai); else ab = fmaf(as[k], w, ab);
        }
        M = mn;
        __syncthreads();
    }
    part_i[quarter][c] = ai;
    part_b[quarter][c] = ab;
    if (c == 0) red_l[quarter] = L;
    __syncthreads();
    if (quarter == 0) acc_rot[c] = (part_i[0][c] + part_i[1][c]) + (part_i[2][c] + part_i[3][c]);
    __syncthreads();
    float o = 0.0f;
#pragma unroll
    for (int i = 0; i < D / 4; ++i) o = fmaf(acc_rot[quarter * (D / 4) + i], rv[i], o);
    part_i[quarter][c] = o;
    __syncthreads();
    if (quarter == 0) {
        const float Lt = (red_l[0] + red_l[1]) + (red_l[2] + red_l[3]);
        const float oi = (part_i[0][c] + part_i[1][c]) + (part_i[2][c] + part_i[3][c]);
        const float ob = (part_b[0][c] + part_b[1][c]) + (part_b[2][c] + part_b[3][c]);
        out[(size_t)bh * D + c] = Lt > 0.0f ? (oi + ob) / Lt : 0.0f;
    }
}

// Merge of all splits of the GQ query heads of one (sequence, KV head), for plans whose per-head merge
// grid would take more than one wave (many query heads): R_v^T is read once per (sequence, KV head)
// instead of once per query head, and the grid is GQ times smaller. Block of 4*D threads: warp h finds
// head h's split weights; thread (c, quarter) then sums its quarter of the splits for every head (loads
// of kRound splits in flight per round, spread over the heads) and a quarter of the un-rotation terms.
template <int D, int GQ>
__global__ void __launch_bounds__(4 * D)
merge_unit_kernel(const float* __restrict__ partials, const float* __restrict__ r_vt, float* __restrict__ out,
                  int h_kv, int int2_splits, int total_splits) {
    constexpr int kRound = 24;                          // accumulator loads per thread per round
    constexpr int kPerHead = (kRound + GQ - 1) / GQ;    // splits of each head per round and quarter
    static_assert(GQ <= 4 * D / 32, "one warp per query head");
    extern __shared__ float w_s[];                      // [GQ][total_splits] split weights
    __shared__ float l_s[GQ];
    __shared__ float red_i[4][GQ][D], red_b[4][GQ][D];
    __shared__ float acc_rot[GQ][D], acc_b[GQ][D];
    const int unit = blockIdx.x, b = unit / h_kv, kv = unit % h_kv;
    const int tid = threadIdx.x, c = tid % D, quarter = tid / D, warp = tid / 32, lane = tid % 32;
    const int T = total_splits;
    const float* rt = r_vt + (size_t)kv * D * D + (size_t)quarter * (D / 4) * D + c;
    float rv[D / 4];
#pragma unroll
    for (int i = 0; i < D / 4; ++i) rv[i] = __ldg(rt + (size_t)i * D);
    pdl_wait();
    pdl_trigger();
    const float* part0 = partials + ((size_t)b * h_kv * GQ + (size_t)kv * GQ) * T * (D + 2);
    if (warp < GQ) {
        const float* part = part0 + (size_t)warp * T * (D + 2);
        float M = -INFINITY;
        for (int s0 = 0; s0 < T; s0 += 32)
            if (s0 + lane < T) M = fmaxf(M, __ldcg(part + (size_t)(s0 + lane) * (D + 2)));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        float L = 0.0f;
        for (int s0 = 0; s0 < T; s0 += 32) {
            const int sp = s0 + lane;
            if (sp < T) {
                const float m = __ldcg(part + (size_t)sp * (D + 2));
                const float w = (M == -INFINITY || m == -INFINITY) ? 0.0f : fast_exp2(m - M);
                w_s[warp * T + sp] = w;
                L = fmaf(__ldcg(part + (size_t)sp * (D + 2) + 1), w, L);
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
        if (lane == 0) l_s[warp] = L;
    }
    __syncthreads();
    float ai[GQ], ab[GQ];
#pragma unroll
    for (int h = 0; h < GQ; ++h) { ai[h] = 0.0f; ab[h] = 0.0f; }
    for (int k0 = 0; 4 * k0 + quarter < T; k0 += kPerHead) {
        // splits with weight 0 (empty splits of the shorter sequences, or far below the maximum) are not read
        float v[GQ][kPerHead], wv[GQ][kPerHead];
#pragma unroll
        for (int h = 0; h < GQ; ++h)
#pragma unroll
            for (int k = 0; k < kPerHead; ++k) {
                const int sp = 4 * (k0 + k) + quarter;
                wv[h][k] = sp < T ? w_s[h * T + sp] : 0.0f;
                v[h][k] = wv[h][k] != 0.0f ? __ldcg(part0 + ((size_t)h * T + sp) * (D + 2) + 2 + c) : 0.0f;
            }
#pragma unroll
        for (int h = 0; h < GQ; ++h)
#pragma unroll
            for (int k = 0; k < kPerHead; ++k) {
                const int sp = 4 * (k0 + k) + quarter;
                const float x = v[h][k] * wv[h][k];
                if (sp < int2_splits) ai[h] += x; else ab[h] += x;
            }
    }
#pragma unroll
    for (int h = 0; h < GQ; ++h) { red_i[quarter][h][c] = ai[h]; red_b[quarter][h][c] = ab[h]; }
    __syncthreads();
    for (int h = quarter; h < GQ; h += 4) {
        acc_rot[h][c] = (red_i[0][h][c] + red_i[1][h][c]) + (red_i[2][h][c] + red_i[3][h][c]);
        acc_b[h][c] = (red_b[0][h][c] + red_b[1][h][c]) + (red_b[2][h][c] + red_b[3][h][c]);
    }
    __syncthreads();
    // un-rotation: quarter q of the terms of every head, then the quarters are summed per head
#pragma unroll
    for (int h = 0; h < GQ; ++h) {
        float o = 0.0f;
#pragma unroll
        for (int i = 0; i < D / 4; ++i) o = fmaf(acc_rot[h][quarter * (D / 4) + i], rv[i], o);
        red_i[quarter][h][c] = o;
    }
    __syncthreads();
    for (int h = quarter; h < GQ; h += 4) {
        const float Lt = l_s[h];
        const float oi = (red_i[0][h][c] + red_i[1][h][c]) + (red_i[2][h][c] + red_i[3][h][c]);
        out[((size_t)unit * GQ + h) * D + c] = Lt > 0.0f ? (oi + acc_b[h][c]) / Lt : 0.0f;
    }
}

// Launch with programmatic stream serialization: the kernel may start while the previous grid in the
// stream finishes; every kernel here waits (griddepcontrol.wait) before touching its predecessors' data.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

template <int D, int G, int GQ, int CB>
cudaError_t launch_split(const SplitArgs& a, int batch, cudaStream_t st) {
    auto kern = split_kernel<D, G, GQ, CB>;
    const size_t smem = SplitSmem<D, G, GQ>::kDynamic;
    const cudaError_t attr = smem_opt_in<split_kernel<D, G, GQ, CB>>(smem);
    if (attr != cudaSuccess) return attr;
    const long long ctas = a.n_prefix_ctas + (long long)(a.int2_splits + a.bf16_splits) * a.h_kv * batch;
    if (ctas > 0x7fffffffLL) return cudaErrorInvalidValue;
    return launch_pdl(kern, dim3((unsigned)ctas), dim3(kWarps * 32), smem, st, a);
}

template <int D, int G, int CB>
cudaError_t dispatch_gq(int gq, const SplitArgs& a, int batch, cudaStream_t st) {
    switch (gq) {
        case 1: return launch_split<D, G, 1, CB>(a, batch, st);
        case 2: return launch_split<D, G, 2, CB>(a, batch, st);
        case 4: return launch_split<D, G, 4, CB>(a, batch, st);
        case 8: return launch_split<D, G, 8, CB>(a, batch, st);
    }
    return cudaErrorInvalidValue;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Resident split CTAs per SM for the shape on the current device (queried once per device).
template <int D, int G, int GQ, int CB>
int split_occupancy() {
    static std::atomic<int> occ[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) dev = 64;
    if (dev < 64) {
        const int cached = occ[dev].load(std::memory_order_acquire);
        if (cached > 0) return cached;
    }
    int n = 0;
    auto kern = split_kernel<D, G, GQ, CB>;
    if (smem_opt_in<split_kernel<D, G, GQ, CB>>(SplitSmem<D, G, GQ>::kDynamic) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kWarps * 32, SplitSmem<D, G, GQ>::kDynamic) !=
            cudaSuccess || n < 1) {
        cudaGetLastError();
        n = 1;
    }
    if (dev < 64) occ[dev].store(n, std::memory_order_release);
    return n;
}

template <int D, int G, int CB>
int occupancy_gq(int gq) {
    switch (gq) {
        case 1: return split_occupancy<D, G, 1, CB>();
        case 2: return split_occupancy<D, G, 2, CB>();
        case 4: return split_occupancy<D, G, 4, CB>();
        default: return split_occupancy<D, G, 8, CB>();
    }
}

template <int CB>
int split_ctas_per_sm_cb(const Shape& s) {
    const int gq = s.h_q / s.h_kv;
    if (s.d == 64) return s.group == 32 ? occupancy_gq<64, 32, CB>(gq) : occupancy_gq<64, 64, CB>(gq);
    if (s.group == 32) return occupancy_gq<128, 32, CB>(gq);
    if (s.group == 64) return occupancy_gq<128, 64, CB>(gq);
    return occupancy_gq<128, 128, CB>(gq);
}

}  // namespace

// Split-kernel launchers and occupancy queries, one translation unit per group of shapes (compiled in
// parallel): D = 128 uniform G = 128; D = 128 uniform G = 32 and 64; D = 128 Lloyd-Max; D = 64.
cudaError_t split_launch_u128_g128(int gq, const SplitArgs& a, int batch, cudaStream_t st);
int split_occupancy_u128_g128(int gq);
cudaError_t split_launch_u128_small_g(int group, int gq, const SplitArgs& a, int batch, cudaStream_t st);
int split_occupancy_u128_small_g(int group, int gq);
cudaError_t split_launch_lm128(int group, int gq, const SplitArgs& a, int batch, cudaStream_t st);
int split_occupancy_lm128(int group, int gq);
cudaError_t split_launch_d64(int group, int codebook, int gq, const SplitArgs& a, int batch, cudaStream_t st);
int split_occupancy_d64(int group, int codebook, int gq);

}  // namespace oscar
