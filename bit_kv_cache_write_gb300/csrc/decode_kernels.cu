// Paged decode attention over the three-segment cache: INT2 history and BF16 sink/recent. This unit
// holds the split plan and the launch sequence (query preparation, split, merge); the kernels are in
// decode_device.cuh, and the split kernel's instantiations in the split_*.cu units.

#include "decode_device.cuh"

namespace oscar {

int split_ctas_per_sm(const Shape& s) {
    const int gq = s.h_q / s.h_kv;
    if (s.d == 64) return split_occupancy_d64(s.group, s.codebook, gq);
    if (s.codebook == OSCAR_CODEBOOK_LLOYD_MAX) return split_occupancy_lm128(s.group, gq);
    if (s.group == 128) return split_occupancy_u128_g128(gq);
    return split_occupancy_u128_small_g(s.group, gq);
}

DecodePlan plan_decode(const Shape& s, int num_sms, int batch, int max_hist, int prefix_pages) {
    DecodePlan p{};
    const int max_pages = (max_hist + kPage - 1) / kPage;
    const long long units_ll = (long long)batch * s.h_kv;     // batch <= 65535 is checked by every caller
    const int units = units_ll > (1 << 30) ? (1 << 30) : (int)units_ll;
    // one wave of units * (INT2 splits + 1 BF16 split) resident CTAs when that keeps splits short
    // (few units: bs1 decode); otherwise at most kMaxPagesPerSplit pages per split, in as many
    // waves as that takes (many units or long sequences)
    const int slots = split_ctas_per_sm(s) * num_sms;
    // BF16 splits: two when the grid is one wave of few units (bs1), so that the BF16 segment's CTAs
    // (CUDA-core attention, about 1.7x an INT2 split's bytes at 100k) finish within the INT2 splits'
    // time while taking few of the wave's CTA slots (measured against three and five); otherwise one
    const int bf16_pages = (s.sink + s.recent + kPage - 1) / kPage;
    p.bf16_splits = (units > 0 && slots / units >= 16 && bf16_pages >= 2) ? 2 : 1;
    p.bf16_pages_per_split = (bf16_pages + p.bf16_splits - 1) / p.bf16_splits;
    int splits = units > 0 ? slots / units - p.bf16_splits : 1;
    if (splits < 1) splits = 1;
    const int by_len = (max_pages + kMaxPagesPerSplit - 1) / kMaxPagesPerSplit;
    if (splits < by_len) splits = by_len;
    if (max_pages > 0 && splits > max_pages) splits = max_pages;
    if (max_pages == 0) splits = 1;
    p.pages_per_split = max_pages > 0 ? (max_pages + splits - 1) / splits : 1;
    p.int2_splits = max_pages > 0 ? (max_pages + p.pages_per_split - 1) / p.pages_per_split : 1;
    p.total_splits = p.int2_splits + p.bf16_splits;
    if (prefix_pages > 0) {
        // shared prefix: each prefix CTA serves kWarps sequences, every warp walks all the CTA's pages, so
        // a prefix split of kMaxPagesPerSplit / kWarps pages costs about one INT2 split of the longest size
        p.prefix_pages_per_split = kMaxPagesPerSplit / kWarps;
        p.prefix_splits = (prefix_pages + p.prefix_pages_per_split - 1) / p.prefix_pages_per_split;
        p.n_prefix_ctas = p.prefix_splits * s.h_kv * ((batch + kWarps - 1) / kWarps);
        p.total_splits += p.prefix_splits;
    }
    p.ws_partials = align256((size_t)batch * s.h_q * p.total_splits * (s.d + 2) * sizeof(float));
    p.ws_qrot = align256((size_t)batch * s.h_q * 3 * s.d * sizeof(__half)) +
                align256((size_t)batch * s.h_q * sizeof(float)) +
                align256((size_t)batch * s.h_q * (s.d / kSliceCh) * 3 * sizeof(float));
    p.ws_counters = align256((size_t)units * sizeof(int));
    p.ws_total = p.ws_partials + p.ws_qrot + p.ws_counters;
    // the last-CTA merge keeps its weights in the page-stage shared memory (at least 12 KB)
    p.fuse_merge = prefix_pages == 0 && (size_t)(s.h_q / s.h_kv) * p.total_splits <= kFuseWeights;
    // the merge kernel runs one CTA per SM (512 threads, about 120 registers): when one CTA per query head
    // would take more than one wave, one CTA per (sequence, KV head) merges all its query heads and reads
    // R_v^T once for them
    p.merge_per_unit = !p.fuse_merge && s.h_q / s.h_kv >= 2 && (long long)batch * s.h_q > num_sms &&
                       (size_t)(s.h_q / s.h_kv) * p.total_splits * sizeof(float) <= kMergeUnitWeightBytes;
    // q_prep: one CTA per (query head, slice) while that grid fits about one wave of its small CTAs;
    // beyond that one CTA per (sequence, KV head, slice) loads the R_k terms once for the g heads
    p.qprep_per_unit = s.h_q / s.h_kv >= 2 && (long long)batch * s.h_q * (s.d / kSliceCh) > 8LL * num_sms;
    return p;
}

cudaError_t launch_decode(const Shape& s, const LayerParams& prm, const DecodePlan& plan,
                          const DecodeArgs& a, DebugWord* dbg, Profiler* prof, cudaStream_t st) {
    const int g = s.h_q / s.h_kv;
    char* base = static_cast<char*>(a.ws);
    float* partials = reinterpret_cast<float*>(base);
    const size_t nh = (size_t)a.batch * s.h_q;
    char* qbase = base + plan.ws_partials;
    __half* qb = reinterpret_cast<__half*>(qbase);
    float* kap = reinterpret_cast<float*>(qbase + align256(nh * 3 * s.d * sizeof(__half)));
    float* qdig = reinterpret_cast<float*>(reinterpret_cast<char*>(kap) + align256(nh * sizeof(float)));
    int* counters = reinterpret_cast<int*>(base + plan.ws_partials + plan.ws_qrot);
    const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(a.q);

    const double sl2d = s.sm_scale * 1.4426950408889634073599;     // sm_scale * log2(e)
    const float sl2_hi = (float)sl2d, sl2_lo = (float)(sl2d - (double)sl2_hi);
    cudaError_t e = cudaSuccess;
    {
        ProfScope ps(prof, OSCAR_KERNEL_QROT, st);
        const dim3 grid(a.batch * s.h_q, s.d / kSliceCh);
        const dim3 ugrid(a.batch * s.h_kv, s.d / kSliceCh);
#define OSCAR_QPREP_UNIT(D_, G_)                                                                            \
        if (plan.qprep_per_unit && s.d == D_ && g == G_)                                                    \
            e = launch_pdl(q_prep_unit_kernel<D_, G_>, ugrid, dim3(128), 0, st, q, prm.r_k, prm.rk_colmax, qb,   \
                           kap, qdig, s.h_kv, sl2_hi, sl2_lo, counters, 1);                                 \
        else
        OSCAR_QPREP_UNIT(128, 2) OSCAR_QPREP_UNIT(128, 4) OSCAR_QPREP_UNIT(128, 8)
        OSCAR_QPREP_UNIT(64, 2) OSCAR_QPREP_UNIT(64, 4) OSCAR_QPREP_UNIT(64, 8)
#undef OSCAR_QPREP_UNIT
        if (s.d == 128)
            e = launch_pdl(q_prep_kernel<128>, grid, dim3(128), 0, st, q, prm.r_k, prm.rk_colmax, qb, kap, qdig,
                           s.h_q, g, sl2_hi, sl2_lo, counters, 1);
        else
            e = launch_pdl(q_prep_kernel<64>, grid, dim3(128), 0, st, q, prm.r_k, prm.rk_colmax, qb, kap, qdig,
                           s.h_q, g, sl2_hi, sl2_lo, counters, 1);
    }
    if (e != cudaSuccess) return e;

    SplitArgs sa{};
    sa.qb = qb; sa.kap = kap; sa.qdig = qdig; sa.q = q; sa.pv_scale = prm.pv_scale;
    sa.int2_pool = a.int2_pool; sa.int2_pages = a.int2_pages;
    sa.int2_tables = a.int2_tables; sa.int2_stride = a.int2_stride;
    sa.hist_len = a.hist_len; sa.max_hist = a.max_hist;
    sa.bf16_pool = reinterpret_cast<const __nv_bfloat16*>(a.bf16_pool); sa.bf16_pages = a.bf16_pages;
    sa.bf16_tables = a.bf16_tables; sa.bf16_stride = a.bf16_stride;
    sa.bf16_len = a.bf16_len; sa.max_bf16 = s.sink + s.recent;
    sa.partials = partials;
    sa.h_kv = s.h_kv; sa.int2_splits = plan.int2_splits; sa.pages_per_split = plan.pages_per_split;
    sa.bf16_splits = plan.bf16_splits;
    sa.bf16_pages_per_split = plan.bf16_pages_per_split;
    sa.total_splits = plan.total_splits;
    sa.prefix_table = a.prefix_table; sa.prefix_pages = a.prefix_pages;
    sa.prefix_pages_per_split = plan.prefix_pages_per_split; sa.prefix_splits = plan.prefix_splits;
    sa.n_prefix_ctas = plan.n_prefix_ctas; sa.batch = a.batch;
    sa.scale_log2 = sl2_hi;
    sa.scale_log2_lo = sl2_lo;
    sa.debug = s.debug; sa.dbg = dbg;
    sa.fuse_merge = plan.fuse_merge ? 1 : 0;
    sa.counters = counters;
    sa.r_vt = prm.r_vt;
    sa.out = a.out;

    ProfScope ps_split(prof, OSCAR_KERNEL_SPLIT, st);
    if (s.d == 64) e = split_launch_d64(s.group, s.codebook, g, sa, a.batch, st);
    else if (s.codebook == OSCAR_CODEBOOK_LLOYD_MAX) e = split_launch_lm128(s.group, g, sa, a.batch, st);
    else if (s.group == 128) e = split_launch_u128_g128(g, sa, a.batch, st);
    else e = split_launch_u128_small_g(s.group, g, sa, a.batch, st);
    ps_split.stop();
    if (e != cudaSuccess) return e;
    if (plan.fuse_merge) return cudaSuccess;           // merged by the last CTA of each unit

    ProfScope ps_merge(prof, OSCAR_KERNEL_MERGE, st);
    if (plan.merge_per_unit) {
        const size_t wbytes = (size_t)g * plan.total_splits * sizeof(float);
        const dim3 grid(a.batch * s.h_kv), block(4 * s.d);
        const int i2 = plan.prefix_splits + plan.int2_splits;
#define OSCAR_MERGE_UNIT(D_, G_)                                                                            \
        if (s.d == D_ && g == G_) {                                                                         \
            const cudaError_t at = smem_opt_in<merge_unit_kernel<D_, G_>>(kMergeUnitWeightBytes);         \
            if (at != cudaSuccess) return at;                                                                \
            return launch_pdl(merge_unit_kernel<D_, G_>, grid, block, wbytes, st, (const float*)partials,  \
                              prm.r_vt, a.out, s.h_kv, i2, plan.total_splits);                              \
        }
        OSCAR_MERGE_UNIT(128, 2) OSCAR_MERGE_UNIT(128, 4) OSCAR_MERGE_UNIT(128, 8)
        OSCAR_MERGE_UNIT(64, 2) OSCAR_MERGE_UNIT(64, 4) OSCAR_MERGE_UNIT(64, 8)
#undef OSCAR_MERGE_UNIT
        return cudaErrorInvalidValue;
    }
    if (s.d == 128)
        return launch_pdl(merge_kernel<128>, dim3(a.batch * s.h_q), dim3(4 * 128), 0, st, (const float*)partials,
                          prm.r_vt, a.out, s.h_q, g, plan.prefix_splits + plan.int2_splits, plan.total_splits);
    return launch_pdl(merge_kernel<64>, dim3(a.batch * s.h_q), dim3(4 * 64), 0, st, (const float*)partials,
                      prm.r_vt, a.out, s.h_q, g, plan.prefix_splits + plan.int2_splits, plan.total_splits);
}

}  // namespace oscar
