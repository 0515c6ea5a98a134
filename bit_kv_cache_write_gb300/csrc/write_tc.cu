// Bulk write on the tcgen05 tensor cores: rotate -> clip -> group scale/zero ->
// 2-bit quantize -> pack, for many tokens at once.
//
// Method: QbitAI article on OSCAR, serving-pipeline part (rotate, clip,
// quantize, pack four codes per byte, scale and zero point per group) and
// section "OSCAR aligns the rotation with attention" (the fixed per-layer
// rotation R and clip thresholds).
//
// The rotation of a tile of 128 tokens is a GEMM, X[128 x d] . R[d x d]. X is
// bf16, loaded by TMA with a 128-byte swizzle. R is held in shared memory as
// three bf16 pieces, R ~= R1 + R2 + R3 (24 significant bits): bf16 x bf16
// products are exact in fp32, so the rotation keeps fp32-level accuracy. One
// thread issues tcgen05.mma into an fp32 accumulator in tensor memory, small
// pieces first. Four accumulators rotate over three epilogue warp-groups, so the
// MMAs of the next tiles overlap the epilogues of the current ones. Each epilogue thread owns one
// token row (one TMEM lane). It clips the row, takes the group min/max, decides the codes in fp32
// exactly as the CUDA-core kernel does, stores the packed codes, and then the scale/zero (after the
// rare exact path below, which can change only those).
//
// Error bound of the tensor-core rotation. Within one MMA step the products are
// aligned to the largest term and truncated about 24 bits below it, and the sum
// is truncated to fp32. So a step errs by at most 9 * 2^-23 * M (16 products each
// off by under 2^-24 M, plus the final truncation), with M bounded
// by sum_i |x_i R_ic| <= ||x||_2 (R orthogonal). Only the d/16 steps of the
// leading piece carry a full-size M. When that bound could move the stored zero
// or scale by more than one fp16 step (tested on the fp16 roundings of the bound's ends), the
// candidate min/max channels are
// recomputed with a double-float dot product over a row of R^T (up to 4 candidates per round, each
// spread over the warp), as on the CUDA-core path. Those exact values set the stored zero and scale.
//
// Every CTA takes a share of one head's token tiles for K and then the same tiles for V, so the
// rare exact path (mostly V rows) spreads evenly over the GPU; R_v replaces R_k in shared memory
// once the K tiles' MMAs are done.
//
// Roles: warp 0 loads (TMA), warp 1 allocates tensor memory and issues the MMAs,
// warps 2..13 run the epilogue as three warp-groups that take tiles in turn, tile i in accumulator
// i % 4 (warp w reads TMEM lanes 32*(w%4) .. +31). 14 warps at 128 registers fit one SM without
// spills; 18 warps would cap every thread at 96, because one of the four schedulers of an SM
// would carry five warps from its 16K registers. Every
// mbarrier wait is bounded. A role that gives up sets a shared flag and records
// kind 4 in the error word. The others then stop, and the copies and MMAs still
// in flight are drained (bounded) before tensor memory is freed.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cfloat>
#include <cstring>

#include "layout.cuh"
#include "oscar_internal.h"

namespace oscar {
namespace {

constexpr int kTile = 128;                     // tokens per tile (UMMA M)
constexpr int kPieces = kRotationPieces;       // bf16 pieces of R
constexpr int kStages = 3;                     // X tile buffers
constexpr int kGroups = 3;                     // epilogue warp-groups
constexpr int kAccs = 4;                       // fp32 accumulators in TMEM (kAccs / kGroups per group)
constexpr int kEpiWarps = 4 * kGroups;
constexpr int kThreads = 32 * (2 + kEpiWarps);
constexpr long long kWaitCycles = 2000000000LL;

template <int D>
struct TcLayout {
    static constexpr int kPieceBytes = D * D * 2;          // one piece, SW128 K-major image
    static constexpr int kTileBytes = kTile * D * 2;       // one X tile
    static constexpr int kHalves = D / 64;                 // 128-byte swizzle atoms along K
    static constexpr int kOffB = 0;
    static constexpr int kOffA = kOffB + kPieces * kPieceBytes;
    static constexpr int kOffT = kOffA + kStages * kTileBytes;
    // T_k, T_v of the head
    static constexpr int kOffBar = kOffT + 2 * D * 4;
    static constexpr int kBars = 2 * kStages + 2 * kAccs + 1;     // full, empty, acc_full[], acc_empty[], b_full
    static constexpr int kOffMisc = kOffBar + kBars * 8;
    static constexpr int kBytes = kOffMisc + 16;
    static constexpr size_t kDynamic = (size_t)kBytes + 1024;
    static constexpr int kTmemCols = kAccs * D <= 128 ? 128 : (kAccs * D <= 256 ? 256 : 512);
};

// ---- small PTX helpers ------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint32_t bar, int count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(bar), "r"(bytes) : "memory");
}
// try_wait with a suspend-time hint: the warp sleeps (up to ~0.1 ms) instead of spinning on the
// issue slots that the other warps of the SM need.
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t phase) {
    uint32_t ok;
    asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3; selp.u32 %0, 1, 0, p; }"
                 : "=r"(ok) : "r"(bar), "r"(phase), "r"(100000u) : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t phase) {
    if (mbar_test(bar, phase)) return true;
    const long long t0 = clock64();
    while (!mbar_test(bar, phase))
        if (clock64() - t0 > kWaitCycles) return false;
    return true;
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 :: "r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, 8-row groups 1024 B apart.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;                  // leading-dimension offset (unused for swizzled K-major)
    d |= (uint64_t)(1024 >> 4) << 32;        // stride-dimension offset
    d |= (uint64_t)1 << 46;                  // descriptor version
    d |= (uint64_t)2 << 61;                  // 128-byte swizzle
    return d;
}

// Instruction descriptor, kind::f16: bf16 A and B, fp32 accumulator, both K-major.
__host__ __device__ constexpr uint32_t idesc_bf16(int m, int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void umma_ss(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile("{ .reg .pred p; setp.ne.b32 p, %4, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }"
                 :: "r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
}
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" :: "r"(bar) : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float* v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
        :: "r"(taddr),
           "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
           "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
           "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
           "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15])),
           "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])), "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])),
           "r"(__float_as_uint(v[20])), "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
           "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])), "r"(__float_as_uint(v[27])),
           "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])), "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
        : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// ---- epilogue ---------------------------------------------------------------------------------

// Packed fp32 pairs (sm_100 and later): each half of sub/mul/add/fma.f32x2 rounds to nearest
// exactly as the scalar instruction does.
__device__ __forceinline__ uint64_t f32x2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ uint64_t sub_f32x2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}

// Three-input fp32 min / max (one instruction each on sm_100 and later; finite inputs here).
__device__ __forceinline__ float fmin3(float a, float b, float c) {
    float r;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
    s = __fadd_rn(a, b);
    const float bp = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bp)), __fsub_rn(b, bp));
}

__host__ __device__ constexpr int bit_offset(int kind, int c, int d) {
    return kind == 0 ? k_bit_offset(c, d) : v_bit_offset(c, d);
}

// The packed bit offset of channel 32 ch + j is off(j) + off(32 ch) for both layouts and head
// sizes, with no carry out of a 32-bit word and a word shift of at most one. So one 32-channel
// chunk body, with compile-time offsets, serves every chunk.
__host__ __device__ constexpr bool chunk_additive(int kind, int d) {
    for (int ch = 0; ch < d / 32; ++ch) {
        const int delta = bit_offset(kind, 32 * ch, d);
        if (delta / 32 > 1) return false;
        for (int j = 0; j < 32; ++j) {
            const int b = bit_offset(kind, j, d);
            if (bit_offset(kind, 32 * ch + j, d) != b + delta || b % 32 + delta % 32 >= 32) return false;
        }
    }
    return true;
}
static_assert(chunk_additive(0, 64) && chunk_additive(0, 128) && chunk_additive(1, 64) && chunk_additive(1, 128),
              "packed layout not chunk-additive");

// Pass 2 packs in fp32. Packed pairs are adjacent channels (j, j+1), j even. Channel c of a chunk
// goes to a 16-bit slot (word, half) = (off / 32, off / 16 % 2) at field shift off % 16. Both
// channels of a pair share the field shift, and the pairs with the same two slots form one chain.
// A chain is packed by Horner steps on exact small integers, so each slot ends as 2^23 + its
// 16-bit value (the float bits hold it in the low half).
__host__ __device__ constexpr int slot_of(int kind, int c, int d) {
    return 2 * (bit_offset(kind, c, d) >> 5) + ((bit_offset(kind, c, d) >> 4) & 1);
}
__host__ __device__ constexpr int field_of(int kind, int c, int d) { return bit_offset(kind, c, d) & 15; }
// the first pair of pair j's chain
__host__ __device__ constexpr int chain_head(int kind, int j, int d) {
    for (int i = 0; i < j; i += 2)
        if (slot_of(kind, i, d) == slot_of(kind, j, d) && slot_of(kind, i + 1, d) == slot_of(kind, j + 1, d)) return i;
    return j;
}
// the pair of chain h whose field shift is s, or -1
__host__ __device__ constexpr int chain_pair(int kind, int h, int s, int d) {
    for (int j = h; j < 32; j += 2)
        if (chain_head(kind, j, d) == h && field_of(kind, j, d) == s) return j;
    return -1;
}
// every pair's channels share a field shift, every chain holds field 0, and the two channels of
// a pair sit in different slots
__host__ __device__ constexpr bool float_packable(int kind, int d) {
    for (int j = 0; j < 32; j += 2) {
        if (field_of(kind, j, d) != field_of(kind, j + 1, d)) return false;
        if (slot_of(kind, j, d) == slot_of(kind, j + 1, d)) return false;
        if (chain_head(kind, j, d) == j && chain_pair(kind, j, 0, d) < 0) return false;
    }
    return true;
}
static_assert(float_packable(0, 64) && float_packable(0, 128) && float_packable(1, 64) && float_packable(1, 128),
              "packed layout not packable in fp32 pairs");

// One Horner step per field of chain H, from field S down to 0 (PREV = the field before, or -1).
template <int KIND, int D, int H, int S, int PREV>
__device__ __forceinline__ uint64_t chain_step(const float (&v)[32], uint64_t mn2, uint64_t inv2, uint64_t acc) {
    if constexpr (S < 0) {
        return acc;
    } else {
        constexpr int J = chain_pair(KIND, H, S, D);
        if constexpr (J < 0) {
            return chain_step<KIND, D, H, S - 2, PREV>(v, mn2, inv2, acc);
        } else {
            // rint(u) + 1.5 * 2^23, then minus 1.5 * 2^23 (or minus 2^22 on field 0, leaving 2^23 + code)
            const uint64_t r2 = add_f32x2(mul_f32x2(sub_f32x2(f32x2(v[J], v[J + 1]), mn2), inv2),
                                          f32x2(12582912.0f, 12582912.0f));
            const uint64_t c2 = S == 0 ? sub_f32x2(r2, f32x2(4194304.0f, 4194304.0f))
                                       : sub_f32x2(r2, f32x2(12582912.0f, 12582912.0f));
            uint64_t a = c2;
            if constexpr (PREV >= 0) {
                constexpr float k = (float)(1 << (PREV - S));
                a = fma_f32x2(acc, f32x2(k, k), c2);                   // exact: every partial sum < 2^24
            }
            return chain_step<KIND, D, H, S - 2, S>(v, mn2, inv2, a);
        }
    }
}

// Packs one 32-channel chunk: slot k ends as the float 2^23 + (its 16-bit value).
template <int KIND, int D, int H = 0>
__device__ __forceinline__ void pack_chains(const float (&v)[32], uint64_t mn2, uint64_t inv2, uint32_t* slot) {
    if constexpr (H < 32) {
        if constexpr (chain_head(KIND, H, D) == H) {
            const uint64_t acc = chain_step<KIND, D, H, 14, -1>(v, mn2, inv2, 0ull);
            slot[slot_of(KIND, H, D)] = (uint32_t)acc;
            slot[slot_of(KIND, H + 1, D)] = (uint32_t)(acc >> 32);
        }
        pack_chains<KIND, D, H + 2>(v, mn2, inv2, slot);
    }
}

template <int D, int G>
__device__ __forceinline__ uint8_t* row_segment(int64_t slot, int head, int h_kv, int kind, uint8_t* __restrict__ int2_pool) {
    using GE = Geo<D, G>;
    const int64_t pg = slot / kPage;
    return int2_pool + ((size_t)pg * h_kv + head) * GE::kBlock + (size_t)kind * GE::kSeg;
}

template <int D, int G>
__device__ __forceinline__ void store_codes(const uint32_t* words, int64_t slot, int head, int h_kv, int kind,
                                            uint8_t* __restrict__ int2_pool) {
    using GE = Geo<D, G>;
    uint32_t* dst = reinterpret_cast<uint32_t*>(row_segment<D, G>(slot, head, h_kv, kind, int2_pool) +
                                                (int)(slot % kPage) * GE::kCodeRow);
#pragma unroll
    for (int w = 0; w < D / 16; w += 4)
        *reinterpret_cast<uint4*>(dst + w) = make_uint4(words[w], words[w + 1], words[w + 2], words[w + 3]);
}

template <int D, int G>
__device__ __forceinline__ void store_sz(const float* mn, const float* mx, int64_t slot, int head, int h_kv, int kind,
                                         uint8_t* __restrict__ int2_pool) {
    using GE = Geo<D, G>;
    constexpr int NG = D / G;
    __half2* szd = reinterpret_cast<__half2*>(row_segment<D, G>(slot, head, h_kv, kind, int2_pool) + GE::kCodeBytes) +
                   (int)(slot % kPage) * NG;
#pragma unroll
    for (int g = 0; g < NG; ++g)
        szd[g] = __halves2half2(__float2half_rn(__fdiv_rn(__fsub_rn(mx[g], mn[g]), 3.0f)), __float2half_rn(mn[g]));
}

template <int D, int G>
__device__ __forceinline__ void group_inv(const float* mn, const float* mx, float* inv) {
#pragma unroll
    for (int g = 0; g < D / G; ++g) {
        const float rng = __fsub_rn(mx[g], mn[g]);
        inv[g] = !(rng >= FLT_MIN) ? 0.0f : __fdiv_rn(3.0f, rng);       // degenerate group: codes 0
    }
}

// fp16 (round to nearest even) of x as an integer that is monotone in x: consecutive fp16 values
// differ by one.
__device__ __forceinline__ int f16_ordered(float x) {
    const int b = (int)__half_as_ushort(__float2half_rn(x));
    return (b & 0x8000) ? 0x8000 - b : b + 0x8000;
}

// Whether a value known to lie within +-e of v could round to an fp16 more than one step away
// from fp16(v).
__device__ __forceinline__ bool f16_unsure(float v, float e) {
    const int o = f16_ordered(v);
    return o - f16_ordered(v - e) > 1 || f16_ordered(v + e) - o > 1;
}

// The stored zero fp16(mn) and scale fp16((mx - mn) / 3) of a group whose exact min/max lie
// within +-err of (mn, mx): bit 0 = the zero may be off by more than one fp16 step, bit 1 = the
// scale may.
__device__ __forceinline__ int sz_unsure(float mn, float mx, float err) {
    const float e = err * 1.01f;                 // covers the fp32 rounding of the tests themselves
    return (f16_unsure(mn, e) ? 1 : 0) | (f16_unsure(__fdiv_rn(__fsub_rn(mx, mn), 3.0f), e * (2.0f / 3.0f)) ? 2 : 0);
}

template <int NG>
struct GroupStats {
    float mn[NG], mx[NG];
};

template <int NCH>
struct ChunkStats {
    float mn[NCH], mx[NCH];
};

template <int NG, int NCH>
struct FixState {
    uint32_t cand[NCH];                             // candidate channels, bit j of word ch = channel 32ch+j
    float mn[NG], mx[NG];                           // stats over non-candidates (+ exact candidates)
    bool need_min[NG], need_max[NG];
};

// Rare path for a warp-tile, part 1 (needs the accumulator): some row has a group whose stored
// zero or scale could be off by more than one fp16 step. Marks every channel that may hold such
// a group's min (max) as a candidate and takes the group stats over the other channels. Only
// 32-channel chunks whose min (max) comes near the cut are reread.
template <int D, int G>
__device__ __forceinline__ FixState<D / G, D / 32> fixup_detect(uint32_t tacc, const float* __restrict__ t_s,
                                                              bool need, float err, GroupStats<D / G> st,
                                                              ChunkStats<D / 32> cs) {
    constexpr int NG = D / G;
    constexpr int NCH = D / 32;
    FixState<NG, NCH> fs;
    float lo_cut[NG], hi_cut[NG];
#pragma unroll
    for (int g = 0; g < NG; ++g) {
        const int u = need ? sz_unsure(st.mn[g], st.mx[g], err) : 0;
        fs.need_min[g] = u != 0;                    // the scale needs both ends
        fs.need_max[g] = (u & 2) != 0;
        lo_cut[g] = fs.need_min[g] ? st.mn[g] + 2.0f * err : -FLT_MAX;
        hi_cut[g] = fs.need_max[g] ? st.mx[g] - 2.0f * err : FLT_MAX;
        fs.mn[g] = fs.need_min[g] ? FLT_MAX : st.mn[g];
        fs.mx[g] = fs.need_max[g] ? -FLT_MAX : st.mx[g];
    }
    for (int ch = 0; ch < NCH; ++ch) {
        const int g = (32 * ch) / G;
        float lc = -FLT_MAX, hc = FLT_MAX, cmn0 = 0.0f, cmx0 = 0.0f;
        bool nmin = false, nmax = false;
#pragma unroll
        for (int k = 0; k < NCH; ++k)
            if (k == ch) { cmn0 = cs.mn[k]; cmx0 = cs.mx[k]; }
#pragma unroll
        for (int gg = 0; gg < NG; ++gg)
            if (gg == g) { lc = lo_cut[gg]; hc = hi_cut[gg]; nmin = fs.need_min[gg]; nmax = fs.need_max[gg]; }
        const bool touched = cmn0 <= lc || cmx0 >= hc;
        uint32_t cm = 0u;
        float cmn = cmn0, cmx = cmx0;
        if (__any_sync(0xffffffffu, touched)) {
            float v[32];
            tmem_ld32(tacc + 32 * ch, v);
            tmem_wait_ld();
            if (touched) {
                cmn = FLT_MAX;
                cmx = -FLT_MAX;
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const float xh = v[j];                 // clipped in pass 1
                    const bool is_c = xh <= lc || xh >= hc;
                    cm |= (uint32_t)is_c << j;
                    if (!is_c) { cmn = fminf(cmn, xh); cmx = fmaxf(cmx, xh); }
                }
            }
        }
#pragma unroll
        for (int gg = 0; gg < NG; ++gg)
            if (gg == g) {
                if (nmin) fs.mn[gg] = fminf(fs.mn[gg], cmn);
                if (nmax) fs.mx[gg] = fmaxf(fs.mx[gg], cmx);
            }
#pragma unroll
        for (int k = 0; k < NCH; ++k)
            if (k == ch) fs.cand[k] = cm;
    }
    return fs;
}

// Part 2 (after the accumulator is released): the candidates' exact values, each a double-float
// dot over a row of R^T spread across the warp (lane l takes terms PER*l ..), up to 4 candidates
// at a time with their loads issued together; returns the repaired stats of this row's groups.
// (The codes of these channels are 0 near the min and 3 near the max either way.)
template <int D, int G>
__device__ __forceinline__ GroupStats<D / G> fixup_exact(FixState<D / G, D / 32> fs, const float* __restrict__ t_s,
                                                       int tok, int head, int h_kv,
                                                       const __nv_bfloat16* __restrict__ x_base,
                                                       const float* __restrict__ rt_head, int lane) {
    constexpr int NG = D / G;
    constexpr int NCH = D / 32;
    constexpr int PER = D / 32;                     // terms per lane
    constexpr int B = 4;                            // candidates per round
    for (;;) {
        int s_src[B], s_c[B];
        float rv[B][PER], xv[B][PER];
        bool left = true;                           // warp-uniform: some lane still has candidates
#pragma unroll
        for (int k = 0; k < B; ++k) {
            s_src[k] = -1;
            s_c[k] = 0;
            if (!left) continue;
            bool mine = false;
#pragma unroll
            for (int ch = 0; ch < NCH; ++ch) mine |= fs.cand[ch] != 0u;
            const uint32_t has = __ballot_sync(0xffffffffu, mine);
            if (!has) {
                left = false;
                continue;
            }
            s_src[k] = __ffs(has) - 1;
            int myc = 0;
            if (lane == s_src[k]) {
                bool done = false;
#pragma unroll
                for (int ch = 0; ch < NCH; ++ch)
                    if (!done && fs.cand[ch]) {
                        myc = 32 * ch + __ffs(fs.cand[ch]) - 1;
                        fs.cand[ch] &= fs.cand[ch] - 1;
                        done = true;
                    }
            }
            s_c[k] = __shfl_sync(0xffffffffu, myc, s_src[k]);
            const int st_tok = __shfl_sync(0xffffffffu, tok, s_src[k]);
            const float* rr = rt_head + (size_t)s_c[k] * D + PER * lane;
            const __nv_bfloat16* xr = x_base + ((size_t)st_tok * h_kv + head) * D + PER * lane;
            if constexpr (PER == 4) {
                const float4 r4 = *reinterpret_cast<const float4*>(rr);
                const uint2 xb = *reinterpret_cast<const uint2*>(xr);
                rv[k][0] = r4.x; rv[k][1] = r4.y; rv[k][2] = r4.z; rv[k][3] = r4.w;
                xv[k][0] = __uint_as_float(xb.x << 16); xv[k][1] = __uint_as_float(xb.x & 0xFFFF0000u);
                xv[k][2] = __uint_as_float(xb.y << 16); xv[k][3] = __uint_as_float(xb.y & 0xFFFF0000u);
            } else {
                const float2 r2 = *reinterpret_cast<const float2*>(rr);
                const uint32_t xb = *reinterpret_cast<const uint32_t*>(xr);
                rv[k][0] = r2.x; rv[k][1] = r2.y;
                xv[k][0] = __uint_as_float(xb << 16); xv[k][1] = __uint_as_float(xb & 0xFFFF0000u);
            }
        }
        if (s_src[0] < 0) break;
#pragma unroll
        for (int k = 0; k < B; ++k) {
            if (s_src[k] < 0) break;                // slots fill in order: the rest are empty
            float hi = 0.0f, lo = 0.0f;
#pragma unroll
            for (int j = 0; j < PER; ++j) {
                const float p = __fmul_rn(xv[k][j], rv[k][j]);
                const float pe = __fmaf_rn(xv[k][j], rv[k][j], -p);
                float t, e;
                two_sum(hi, p, t, e);
                hi = t;
                lo = __fadd_rn(lo, __fadd_rn(pe, e));
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float h2 = __shfl_xor_sync(0xffffffffu, hi, o);
                const float l2 = __shfl_xor_sync(0xffffffffu, lo, o);
                float t, e;
                two_sum(hi, h2, t, e);
                hi = t;
                lo = __fadd_rn(__fadd_rn(lo, l2), e);
            }
            if (s_src[k] >= 0 && lane == s_src[k]) {
                const int c = s_c[k];
                const float exc = fminf(fmaxf(__fadd_rn(hi, lo), -t_s[c]), t_s[c]);
#pragma unroll
                for (int g = 0; g < NG; ++g)
                    if (c / G == g) {
                        if (fs.need_min[g]) fs.mn[g] = fminf(fs.mn[g], exc);
                        if (fs.need_max[g]) fs.mx[g] = fmaxf(fs.mx[g], exc);
                    }
            }
        }
    }
    GroupStats<NG> out;
#pragma unroll
    for (int g = 0; g < NG; ++g) { out.mn[g] = fs.mn[g]; out.mx[g] = fs.mx[g]; }
    return out;
}

// Epilogue of one tile for one warp: lane = token row, its fp32 row in TMEM at tacc. Two passes
// over 32-column chunks (clip + group stats, then codes) keep few values live. Rows past n or with
// a bad slot (ok false) take part in the warp-wide steps but store nothing. Arrives on acc_empty
// once the accumulator has been read for the last time.
// The rare path as one out-of-line call (the fast path keeps its registers): marks the candidates
// while the accumulator is still held, releases it, then recomputes the candidates exactly.
template <int D, int G>
__device__ __noinline__ GroupStats<D / G> fixup(uint32_t tacc, uint32_t acc_empty, const float* __restrict__ t_s,
                                                 bool need, float err, GroupStats<D / G> st, ChunkStats<D / 32> cs,
                                                 int tok, int head, int h_kv, const __nv_bfloat16* __restrict__ x_base,
                                                 const float* __restrict__ rt_head, int lane) {
    const FixState<D / G, D / 32> fs = fixup_detect<D, G>(tacc, t_s, need, err, st, cs);
    tc_fence_before();
    mbar_arrive(acc_empty);
    return fixup_exact<D, G>(fs, t_s, tok, head, h_kv, x_base, rt_head, lane);
}

template <int D, int G, int KIND>
__device__ __forceinline__ void epilogue_tile(uint32_t tacc, uint32_t acc_empty, const float* __restrict__ t_s,
                                              int tok, int64_t slot, bool ok, int head, int h_kv,
                                              const __nv_bfloat16* __restrict__ x_base,
                                              const float* __restrict__ rt_head, uint8_t* __restrict__ int2_pool,
                                              int lane) {
    constexpr int NG = D / G;
    constexpr int NCH = D / 32;

    // ---- pass 1: clip, group min/max, ||x|| (rotation preserves the norm)
    float mn[NG], mx[NG];
#pragma unroll
    for (int g = 0; g < NG; ++g) { mn[g] = FLT_MAX; mx[g] = -FLT_MAX; }
    uint64_t sq2 = 0ull;                            // packed (sum over even, sum over odd channels)
    float chmn[NCH], chmx[NCH];                     // per-chunk clipped min/max (fixup detection)
    // not unrolled over chunks: the compiler would otherwise keep several chunks live
#pragma unroll 1
    for (int ch = 0; ch < NCH; ++ch) {
        float v[32];
        tmem_ld32(tacc + 32 * ch, v);
        tmem_wait_ld();
        // the clipped row goes back into the accumulator, so pass 2 (and the rare path) read it
        // clipped; ||x|| is taken before the clip
        float cmn = FLT_MAX, cmx = -FLT_MAX;
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
            const float4 t = *reinterpret_cast<const float4*>(t_s + 32 * ch + j);
            const uint64_t a2 = f32x2(v[j], v[j + 1]), b2 = f32x2(v[j + 2], v[j + 3]);
            sq2 = fma_f32x2(a2, a2, sq2);                 // even channels in the low half, odd in the high
            sq2 = fma_f32x2(b2, b2, sq2);
            v[j] = fminf(fmaxf(v[j], -t.x), t.x);
            v[j + 1] = fminf(fmaxf(v[j + 1], -t.y), t.y);
            v[j + 2] = fminf(fmaxf(v[j + 2], -t.z), t.z);
            v[j + 3] = fminf(fmaxf(v[j + 3], -t.w), t.w);
            cmn = fmin3(cmn, v[j], v[j + 1]);
            cmn = fmin3(cmn, v[j + 2], v[j + 3]);
            cmx = fmax3(cmx, v[j], v[j + 1]);
            cmx = fmax3(cmx, v[j + 2], v[j + 3]);
        }
        tmem_st32(tacc + 32 * ch, v);
        // a 32-channel chunk lies inside one group (G >= 32)
#pragma unroll
        for (int g = 0; g < NG; ++g)
            if ((32 * ch) / G == g) { mn[g] = fminf(mn[g], cmn); mx[g] = fmaxf(mx[g], cmx); }
#pragma unroll
        for (int k = 0; k < NCH; ++k)
            if (k == ch) { chmn[k] = cmn; chmx[k] = cmx; }
    }
    tmem_wait_st();                                 // pass 2 reads back what pass 1 stored
    const float sq0 = __uint_as_float((uint32_t)sq2), sq1 = __uint_as_float((uint32_t)(sq2 >> 32));
    const float err = 1.01f * (float)(D / 16) * 9.0f * 0x1p-23f * sqrtf((sq0 + sq1) * 1.002f);
    bool need = false;
#pragma unroll
    for (int g = 0; g < NG; ++g) need |= ok && sz_unsure(mn[g], mx[g], err) != 0;
    // stats for the stored scale/zero; the codes use the tensor-core stats (their shift is far
    // inside the rounding tolerance, and min/max channels code 0/3 either way)
    float mn_sz[NG], mx_sz[NG];
#pragma unroll
    for (int g = 0; g < NG; ++g) { mn_sz[g] = mn[g]; mx_sz[g] = mx[g]; }
    const bool any_need = __any_sync(0xffffffffu, need);

    // ---- pass 2: codes in fp32, packed by fp32 Horner steps (one chunk body; offsets = off(j) + off(32 ch))
    float inv[NG];
    group_inv<D, G>(mn, mx, inv);
    uint32_t words[D / 16];
#pragma unroll
    for (int w = 0; w < D / 16; ++w) words[w] = 0u;
#pragma unroll 1
    for (int ch = 0; ch < NCH; ++ch) {
        float v[32];
        tmem_ld32(tacc + 32 * ch, v);
        tmem_wait_ld();
        if (ch == NCH - 1 && !any_need) {          // else held until the candidates are marked
            tc_fence_before();
            mbar_arrive(acc_empty);
        }
        float gmn = mn[0], ginv = inv[0];
#pragma unroll
        for (int g = 1; g < NG; ++g)
            if ((32 * ch) / G == g) { gmn = mn[g]; ginv = inv[g]; }
        // u = (x_hat - mn) * inv, then + 1.5 * 2^23, two channels per packed fp32 instruction (each
        // half rounds exactly as the scalar op would). u is in [0, 3 + tiny], so adding 1.5 * 2^23
        // rounds it half-to-even onto the integer grid; subtracting 1.5 * 2^23 again leaves the code
        // (2^22 instead on a chain's field 0, which leaves 2^23 + code). x_hat was clipped in pass 1.
        const uint64_t mn2 = f32x2(gmn, gmn), inv2 = f32x2(ginv, ginv);
        uint32_t slot[D / 8];
#pragma unroll
        for (int k = 0; k < D / 8; ++k) slot[k] = 0x4B000000u;
        pack_chains<KIND, D>(v, mn2, inv2, slot);
        // the low 16 bits of each slot's float bits hold its codes; PRMT joins the two halves of a word
        const int delta = bit_offset(KIND, 32 * ch, D);
        const int bs = delta & 31;
        if (delta >> 5) {
#pragma unroll
            for (int w = D / 16 - 1; w >= 1; --w) words[w] += __byte_perm(slot[2 * w - 2], slot[2 * w - 1], 0x5410) << bs;
        } else {
#pragma unroll
            for (int w = 0; w < D / 16; ++w) words[w] += __byte_perm(slot[2 * w], slot[2 * w + 1], 0x5410) << bs;
        }
    }
    // the codes are final (they use the tensor-core stats): store them now, so that only a few
    // registers stay live through the rare path below
    if (ok) store_codes<D, G>(words, slot, head, h_kv, KIND, int2_pool);
    if (any_need) {
        GroupStats<NG> st;
#pragma unroll
        for (int g = 0; g < NG; ++g) { st.mn[g] = mn[g]; st.mx[g] = mx[g]; }
        ChunkStats<NCH> cs;
#pragma unroll
        for (int k = 0; k < NCH; ++k) { cs.mn[k] = chmn[k]; cs.mx[k] = chmx[k]; }
        const GroupStats<NG> ex = fixup<D, G>(tacc, acc_empty, t_s, need, err, st, cs, tok, head, h_kv, x_base,
                                              rt_head, lane);
        if (need) {
#pragma unroll
            for (int g = 0; g < NG; ++g) { mn_sz[g] = ex.mn[g]; mx_sz[g] = ex.mx[g]; }
        }
    }
    if (ok) store_sz<D, G>(mn_sz, mx_sz, slot, head, h_kv, KIND, int2_pool);
}

template <int D, int G>
__global__ void __maxnreg__(128)
write_tc_kernel(const __grid_constant__ CUtensorMap map_k, const __grid_constant__ CUtensorMap map_v,
                const uint16_t* __restrict__ r_img, const float* __restrict__ r_kt, const float* __restrict__ r_vt,
                const float* __restrict__ t_all,
                const __nv_bfloat16* __restrict__ k_in, const __nv_bfloat16* __restrict__ v_in,
                const int64_t* __restrict__ dst_slots, int n, int h_kv, uint8_t* __restrict__ int2_pool,
                int64_t int2_pages, int debug, DebugWord* dbg) {
    using L = TcLayout<D>;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned base (pointer arithmetic keeps the shared address space visible)
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    // every CTA takes its share of this head's token tiles for K, then the same tiles for V
    // (local tiles 0 .. my_tiles-1 are K, my_tiles .. 2 my_tiles-1 are V)
    const int head = blockIdx.y;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int n_tiles = (n + kTile - 1) / kTile;
    const int my_tiles = (int)blockIdx.x < n_tiles ? (n_tiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const int my_total = 2 * my_tiles;
    auto tile_of = [&](int i) { return (int)blockIdx.x + (i < my_tiles ? i : i - my_tiles) * (int)gridDim.x; };

    const uint32_t sb = smem_u32(smem);
    const uint32_t b_s = sb + L::kOffB, a_s = sb + L::kOffA;
    float* t_s = reinterpret_cast<float*>(smem + L::kOffT);
    const uint32_t bar0 = sb + L::kOffBar;
    auto full = [&](int s) { return bar0 + 8 * s; };
    auto empty = [&](int s) { return bar0 + 8 * (kStages + s); };
    auto acc_full = [&](int a) { return bar0 + 8 * (2 * kStages + a); };
    auto acc_empty = [&](int a) { return bar0 + 8 * (2 * kStages + kAccs + a); };
    const uint32_t b_full = bar0 + 8 * (2 * kStages + 2 * kAccs);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffMisc);
    volatile int* fail = reinterpret_cast<volatile int*>(smem + L::kOffMisc + 4);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) { mbar_init(full(s), 1); mbar_init(empty(s), 1); }
        for (int a = 0; a < kAccs; ++a) { mbar_init(acc_full(a), 1); mbar_init(acc_empty(a), 128); }
        mbar_init(b_full, 1);
        *fail = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        // the three pieces of R_k of this head: calibration data, loaded before waiting on the
        // preceding grid (R_v replaces them after the last K tile)
        mbar_expect_tx(b_full, kPieces * L::kPieceBytes);
        for (int p = 0; p < kPieces; ++p)
            bulk_load(b_s + p * L::kPieceBytes, r_img + ((size_t)head * kPieces + p) * (size_t)(D * D), L::kPieceBytes,
                      b_full);
    }
    for (int i = threadIdx.x; i < 2 * D; i += kThreads)
        t_s[i] = t_all[((size_t)(i / D) * h_kv + head) * D + i % D];
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     :: "r"(smem_u32(tmem_slot)), "r"(L::kTmemCols) : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // programmatic dependent launch: token rows, slots and the pool may come from the preceding grid
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == 0) {
        // ---- TMA producer
        if (lane == 0) {
            int issued = 0;
            for (int i = 0; i < my_total; ++i) {
                const CUtensorMap* map = i < my_tiles ? &map_k : &map_v;
                if (*fail) break;
                const int s = i % kStages;
                if (!mbar_wait(empty(s), ((i / kStages) & 1) ^ 1)) {
                    *fail = 1;
                    record_error(&dbg->kind, &dbg->index, 4, i);
                    break;
                }
                const int tile = tile_of(i);
                mbar_expect_tx(full(s), L::kTileBytes);
#pragma unroll
                for (int h = 0; h < L::kHalves; ++h)
                    tma_load_2d(a_s + s * L::kTileBytes + h * (kTile * 128), map, head * D + 64 * h, tile * kTile, full(s));
                issued = i + 1;
            }
            // drain: every issued tile's copy must land before the CTA may leave
            for (int j = issued - kStages < 0 ? 0 : issued - kStages; j < issued; ++j)
                (void)mbar_wait(full(j % kStages), (j / kStages) & 1);
        }
    } else if (warp == 1) {
        // ---- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16(kTile, D);
            int issued = 0;
            bool ok = mbar_wait(b_full, 0);
            if (!ok) {
                *fail = 1;
                record_error(&dbg->kind, &dbg->index, 4, -1);
            }
            for (int i = 0; ok && i < my_total; ++i) {
                if (*fail) break;
                if (i == my_tiles) {
                    // switch to R_v: every K-tile MMA must have finished reading the pieces
                    if (!mbar_wait(acc_full((i - 1) % kAccs), ((i - 1) / kAccs) & 1)) {
                        *fail = 1;
                        record_error(&dbg->kind, &dbg->index, 4, i);
                        break;
                    }
                    tc_fence_after();
                    mbar_expect_tx(b_full, kPieces * L::kPieceBytes);
                    for (int p = 0; p < kPieces; ++p)
                        bulk_load(b_s + p * L::kPieceBytes, r_img + (((size_t)h_kv + head) * kPieces + p) * (size_t)(D * D),
                                  L::kPieceBytes, b_full);
                    if (!mbar_wait(b_full, 1)) {
                        *fail = 1;
                        record_error(&dbg->kind, &dbg->index, 4, i);
                        break;
                    }
                }
                const int s = i % kStages, a = i % kAccs;
                if (!mbar_wait(acc_empty(a), ((i / kAccs) & 1) ^ 1) || !mbar_wait(full(s), (i / kStages) & 1)) {
                    *fail = 1;
                    record_error(&dbg->kind, &dbg->index, 4, i);
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem + a * D;
                uint32_t accum = 0;
#pragma unroll
                for (int p = kPieces - 1; p >= 0; --p) {
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        const uint32_t aa = a_s + s * L::kTileBytes + (ks / 4) * (kTile * 128) + (ks % 4) * 32;
                        const uint32_t bb = b_s + p * L::kPieceBytes + (ks / 4) * (D * 128) + (ks % 4) * 32;
                        umma_ss(d_tmem, sw128_desc(aa), sw128_desc(bb), idesc, accum);
                        accum = 1;
                    }
                }
                umma_commit(empty(s));
                umma_commit(acc_full(a));
                issued = i + 1;
            }
            // drain: the last commit covers every MMA issued before it
            if (issued > 0) (void)mbar_wait(acc_full((issued - 1) % kAccs), ((issued - 1) / kAccs) & 1);
        }
    } else {
        // ---- epilogue: warp-group e takes local tiles e, e + kGroups, ... (accumulator i % kAccs);
        // thread = token row = TMEM lane 32*(warp%4) + lane
        const int e = (warp - 2) / 4;
        const int q = warp % 4;
        const int m = 32 * q + lane;
        for (int i = e; i < my_total; i += kGroups) {
            const int a = i % kAccs;
            const int kind = i < my_tiles ? 0 : 1;
            const __nv_bfloat16* x_base = kind == 0 ? k_in : v_in;
            const float* rt_head = (kind == 0 ? r_kt : r_vt) + (size_t)head * D * D;
            const int tok = tile_of(i) * kTile + m;
            bool ok = tok < n;
            const int64_t slot = ok ? dst_slots[tok] : -1;        // issued before the wait
            const bool got = mbar_wait(acc_full(a), (i / kAccs) & 1);
            const int stop = *fail;
            if (__any_sync(0xffffffffu, !got || stop)) {       // warp-uniform exit
                if (lane == 0) {
                    *fail = 1;
                    record_error(&dbg->kind, &dbg->index, 4, i);
                }
                break;
            }
            tc_fence_after();
            if (ok && (slot < 0 || slot / kPage >= int2_pages)) {
                if (debug) record_error(&dbg->kind, &dbg->index, 1, slot);
                ok = false;
            }
            const uint32_t tacc = tmem + a * D + ((uint32_t)(32 * q) << 16);
            if (kind == 0)
                epilogue_tile<D, G, 0>(tacc, acc_empty(a), t_s, tok, slot, ok, head, h_kv, x_base, rt_head, int2_pool, lane);
            else
                epilogue_tile<D, G, 1>(tacc, acc_empty(a), t_s + D, tok, slot, ok, head, h_kv, x_base, rt_head, int2_pool,
                                       lane);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(tmem), "r"(L::kTmemCols) : "memory");
    }
}

// ---- host side ------------------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}

// [n][h_kv * d] bf16 rows, boxes of 64 channels x 128 tokens, 128-byte swizzle.
bool make_row_map(CUtensorMap* map, const void* base, int n, int h_kv, int d) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)h_kv * d, (cuuint64_t)n};
    const cuuint64_t strides[1] = {(cuuint64_t)h_kv * d * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)kTile};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D, int G>
cudaError_t launch_tc(const Shape& s, const LayerParams& p, int num_sms, const void* k, const void* v,
                      const int64_t* slots, int n, void* int2_pool, int64_t int2_pages, DebugWord* dbg,
                      Profiler* prof, cudaStream_t st) {
    using L = TcLayout<D>;
    auto kern = write_tc_kernel<D, G>;
    const cudaError_t attr = smem_opt_in<write_tc_kernel<D, G>>(L::kDynamic);
    if (attr != cudaSuccess) return attr;
    CUtensorMap mk, mv;
    if (!make_row_map(&mk, k, n, s.h_kv, D) || !make_row_map(&mv, v, n, s.h_kv, D)) return cudaErrorInvalidValue;
    const int n_tiles = (n + kTile - 1) / kTile;
    int gx = num_sms / s.h_kv;
    gx = gx < 1 ? 1 : (gx > n_tiles ? n_tiles : gx);
    ProfScope ps(prof, OSCAR_KERNEL_WRITE, st);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(gx, s.h_kv, 1);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = L::kDynamic;
    cfg.stream = st;
    cudaLaunchAttribute la[1];
    la[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    la[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = la;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, mk, mv, p.r_img, p.r_kt, p.r_vt, p.t_k, static_cast<const __nv_bfloat16*>(k),
                              static_cast<const __nv_bfloat16*>(v), slots, n, s.h_kv,
                              static_cast<uint8_t*>(int2_pool), int2_pages, s.debug, dbg);
}

// bf16 (round to nearest even) of a finite float, as raw bits.
uint16_t bf16_bits(float x) {
    uint32_t u;
    std::memcpy(&u, &x, 4);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}
float bf16_value(uint16_t b) {
    const uint32_t u = (uint32_t)b << 16;
    float x;
    std::memcpy(&x, &u, 4);
    return x;
}

}  // namespace

bool write_tc_eligible(const Shape& s, const void* k, const void* v, const void* int2_pool, int n) {
    if (n < kTcMinTokens || (s.d != 64 && s.d != 128)) return false;
    // TMA row maps need 16-byte aligned bases; the epilogue stores 16-byte code rows
    if ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(int2_pool)) & 15)
        return false;
    return encode_fn() != nullptr;
}

cudaError_t launch_write_tc(const Shape& s, const LayerParams& p, int num_sms, const void* k, const void* v,
                            const int64_t* slots, int n, void* int2_pool, int64_t int2_pages, DebugWord* dbg,
                            Profiler* prof, cudaStream_t st) {
#define OSCAR_TC_CASE(D_, G_) \
    if (s.d == D_ && s.group == G_) return launch_tc<D_, G_>(s, p, num_sms, k, v, slots, n, int2_pool, int2_pages, dbg, prof, st);
    OSCAR_TC_CASE(64, 32)
    OSCAR_TC_CASE(64, 64)
    OSCAR_TC_CASE(128, 32)
    OSCAR_TC_CASE(128, 64)
    OSCAR_TC_CASE(128, 128)
#undef OSCAR_TC_CASE
    return cudaErrorInvalidValue;
}

void build_rotation_images(const float* r, int h_kv, int d, uint16_t* out) {
    // out[h][piece][image]: B[n = output channel j][k = input channel i] = piece(R[i][j]), K-major,
    // 128-byte swizzle atoms of 8 rows x 64 channels (16-byte chunk index XOR row % 8)
    for (int h = 0; h < h_kv; ++h) {
        const float* rh = r + (size_t)h * d * d;
        uint16_t* oh = out + (size_t)h * kPieces * d * d;
        for (int i = 0; i < d; ++i)
            for (int j = 0; j < d; ++j) {
                float rest = rh[(size_t)i * d + j];
                const int half = i / 64, kk = i % 64, chunk = kk / 8, e = kk % 8;
                const size_t off =
                    ((size_t)half * d * 128 + (size_t)j * 128 + (size_t)((chunk ^ (j % 8)) * 16) + e * 2) / 2;
                for (int pce = 0; pce < kPieces; ++pce) {
                    const uint16_t b = bf16_bits(rest);
                    oh[(size_t)pce * d * d + off] = b;
                    rest -= bf16_value(b);
                }
            }
    }
}

}  // namespace oscar
