/*
 * oscar.h: C ABI of liboscar, the GB300 (sm_103a) implementation of OSCAR's
 * INT2 KV-cache write path and paged INT2 decode attention.
 *
 * Method sources (the OSCAR pages):
 *   [ABS]  "OSCAR: Offline Spectral Covariance-Aware Rotation for 2-bit KV Cache
 *          Quantization", arXiv 2605.17757, v1 and v2 abstracts. Fixed
 *          per-layer rotations and clipping thresholds are derived offline. The
 *          INT2 kernels keep paged KV-cache layouts and prefix caching working.
 *   [QBIT] QbitAI article on OSCAR:
 *          - section "OSCAR aligns the rotation with attention":
 *            R = U * Hadamard * bit-reversal, per layer and per head, estimated
 *            offline and reused unchanged;
 *          - the serving-pipeline part:
 *            the three-segment token pool is BF16 sink (64) | INT2 history |
 *            BF16 recent (256). The oldest recent token is rotated, clipped,
 *            quantized and packed into the history, four 2-bit codes per byte.
 *            At decode, the INT2 part unpacks and dequantizes with a scale and
 *            zero point, the BF16 part covers sink/recent, and an
 *            online-softmax merge combines the two.
 *
 * ---------------------------------------------------------------------------
 * Conventions shared by every call
 * ---------------------------------------------------------------------------
 * - Rotation acts on row vectors: x_rot = x @ R, with R a d x d fp32 matrix
 *   stored row-major.
 * - Write path, per (token, KV head, K or V) vector x (bf16, d channels):
 *     x_rot = x @ R  (fp32 accumulation)
 *     x_hat = min(max(x_rot, -T), T)
 *     Per group of G consecutive rotated channels:
 *       mn = min, mx = max, rng = mx - mn (fp32).
 *       If rng < FLT_MIN, every code is 0. Otherwise
 *         code = clamp(rint((x_hat - mn) * (3 / rng)), 0, 3),
 *       with every step done in fp32 round-to-nearest-even, in this order.
 *     scale = fp16(rng / 3), zero = fp16(mn).
 *   Dequant: x_deq = code * scale + zero, in the rotated basis.
 * - With codebook OSCAR_CODEBOOK_LLOYD_MAX (the stronger codebook the [QBIT]
 *   article's closing part pairs with the rotation) every group is
 *   normalised by its own mean mu and standard deviation sigma (fp64, over
 *   the G clipped rotated values) and takes the nearest of the four levels
 *   delta * (-27, -8, 8, 27): the Gaussian Lloyd-Max levels (+-0.4528,
 *   +-1.510) rounded to multiples of delta = 0.45278 / 8 (0.0566). The code
 *   is 0..3 for those levels (ties to the lower one); scale = fp16(sigma *
 *   delta), zero = fp16(mu); sigma = 0 gives scale 0 and codes 0.
 *   Dequant: x_deq = zero + scale * l(code), l = (-27, -8, 8, 27). Layout,
 *   bit order and page size are unchanged.
 * - Decode, per query head h with KV head h / (H_q / H_kv):
 *     logits over the BF16 segment use the unrotated q;
 *     logits over the INT2 history use q_rot = q @ R_k;
 *     logit = sm_scale * dot(...);
 *     p = one softmax over both segments;
 *     out = p_bf16 @ V_bf16 + (p_int2 @ V_deq) @ R_v^T, written as fp32.
 *   There is no causal mask and no positional encoding inside the op.
 *
 * ---------------------------------------------------------------------------
 * Memory layout (library-defined; the pages only fix "4 codes per byte")
 * ---------------------------------------------------------------------------
 * INT2 pool, bytes:     [num_pages][H_kv][2 (K, V)][segment]
 *   segment = codes [P][d/4] bytes, then sz [P][d/G] x {fp16 scale, fp16 zero}
 *   segment bytes = P*d/4 + 4*P*d/G (d=128, G=128: 576; G=64: 640; d=64, G=32: 384)
 *   Code bits in one token row (2*d bits, little-endian words; bit b is bit
 *   b%8 of byte b/8), with n = d/16:
 *     K: kk=c/16, t=(c%16)/4, i=c%4
 *        o_K(c) = 8n*t + 32*(kk/4) + 16*(i%2) + 2*(2*(kk%4) + i/2)
 *     V: m=c/16, r=c%16
 *        o_V(c) = 4n*(r%8) + 2n*(r/8) + 2*m
 *   (These maps put the codes of one m16n8k16 tensor-core fragment into one
 *   32-bit word.)
 * BF16 pool, bf16:      [num_pages][H_kv][2 (K, V)][P][d], unrotated.
 * Slot ids (int64):     slot = page * P + row.
 * Block tables (int32): [batch][stride] physical page ids. Logical token t of
 *   sequence b is at page table[b*stride + t/P], row t%P. Tables may alias
 *   pages (prefix sharing). A page that other sequences share must never be a
 *   write or demote destination: copy-on-write belongs to the caller.
 * q: bf16 [batch][H_q][d]. out: fp32 [batch][H_q][d]. K/V inputs: bf16 [n][H_kv][d].
 *
 * ---------------------------------------------------------------------------
 * Ownership, streams, errors
 * ---------------------------------------------------------------------------
 * - Pools, tables, lengths, q, out and the workspace are caller-owned device
 *   memory. The library owns only the per-layer calibration buffers (R, T and
 *   derived copies) and a device error word.
 * - `stream` is a cudaStream_t passed as void*; NULL is the legacy default
 *   stream. Every launch call is asynchronous on that stream. Except where
 *   stated, no call synchronizes.
 * - A context belongs to the device that was current at oscar_create. Every
 *   call that takes a context must be made with that device current; on any
 *   other device it returns OSCAR_ERR_INVALID_ARG before launching anything.
 * - Host-side validation runs before any launch. A failing call has launched
 *   nothing and returns a negative oscar_status. A launch failure returns
 *   OSCAR_ERR_CUDA. oscar_last_error() gives a one-line message for the
 *   calling thread's most recent failure. No call aborts or traps.
 * - With config.debug_bounds != 0, kernels check every page id, slot and
 *   length against the sizes passed in. An out-of-range access is skipped and
 *   recorded in the device error word, which oscar_debug_error() reads.
 * - Supported shapes: d in {64, 128}; G in {32, 64, 128} with G <= d;
 *   P = 16; H_q/H_kv in {1, 2, 4, 8}; sink + recent <= 512.
 *   Other shapes return OSCAR_ERR_UNSUPPORTED.
 */
#ifndef OSCAR_H
#define OSCAR_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define OSCAR_API __attribute__((visibility("default")))
#else
#define OSCAR_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    OSCAR_OK = 0,
    OSCAR_ERR_INVALID_ARG = -1,    /* null pointer, negative size, layer out of range */
    OSCAR_ERR_UNSUPPORTED = -2,    /* shape outside the supported set */
    OSCAR_ERR_NOT_CALIBRATED = -3, /* layer used before oscar_calibrate_upload */
    OSCAR_ERR_CUDA = -4,           /* CUDA runtime error (launch, copy, device) */
    OSCAR_ERR_BOUNDS = -5,         /* debug bounds check recorded an out-of-range index */
    OSCAR_ERR_NO_MEMORY = -6,      /* device allocation failed */
    OSCAR_ERR_WORKSPACE = -7       /* workspace null or smaller than required */
} oscar_status;

/* 2-bit codebook of the INT2 history (oscar_config_t.codebook). */
typedef enum {
    OSCAR_CODEBOOK_UNIFORM = 0,    /* 4 uniform levels between the group min and max (the pages' OSCAR) */
    OSCAR_CODEBOOK_LLOYD_MAX = 1   /* 4 Gaussian Lloyd-Max levels, rounded (see below) */
} oscar_codebook;

typedef struct {
    int n_layers;     /* layers with their own calibration (R_k, R_v, T_k, T_v) */
    int n_q_heads;    /* H_q */
    int n_kv_heads;   /* H_kv; H_q / H_kv query heads share one KV head */
    int head_dim;     /* d */
    int group;        /* G: consecutive rotated channels sharing one scale/zero */
    int page_size;    /* P: tokens per page, must be 16 */
    int sink;         /* BF16 sink tokens (64 in the pages' system) */
    int recent;       /* BF16 recent window (256 in the pages' system) */
    float sm_scale;   /* logit scale; 1/sqrt(d) if <= 0 */
    int debug_bounds; /* nonzero: kernels bounds-check indices into the error word */
    int codebook;     /* oscar_codebook; 0 (uniform) when zero-initialised */
} oscar_config_t;

typedef struct oscar_ctx oscar_ctx_t;

/* Create a context on the current CUDA device.
 * Validates cfg, then allocates the per-layer calibration buffers and the
 * error word. Per layer:
 *   (3 * H_kv * d * d + 2 * H_kv * d + 2 * H_kv) * 4 bytes: R_k, R_v, R_v^T, T_k,
 *     T_v, and per KV head one P.V exponent and a bound of R_k's column norms;
 *   H_kv * d * d * 4 bytes: R_k^T (the exact path of the tensor-core write);
 *   2 * 3 * H_kv * d * d * 2 bytes: R_k and R_v as three bf16 pieces each, in
 *     the shared-memory image the tensor-core write loads.
 * (3.7 MB per layer at H_kv = 8, d = 128.) On failure *out is NULL.
 * Blocking: returns after the allocations complete. */
OSCAR_API oscar_status oscar_create(const oscar_config_t* cfg, oscar_ctx_t** out);

/* Free everything the context owns. NULL is allowed. The caller must make sure
 * no work that uses ctx is still in flight. */
OSCAR_API void oscar_destroy(oscar_ctx_t* ctx);

/* Upload the offline calibration of one layer ([QBIT] section "OSCAR aligns
 * the rotation with attention": per-layer, per-head fixed rotation and clip
 * threshold, reused as-is at inference).
 *   R_k, R_v: HOST fp32 [H_kv][d][d], row-major, x_rot = x @ R.
 *   T_k, T_v: HOST fp32 [H_kv][d], clip thresholds (>= 0).
 * Copies to library-owned device buffers, then derives R_v^T and an fp16
 * hi/lo split of R on `stream`.
 * Blocking: returns after the copies and derivations finish, so the host
 * buffers may be freed on return. */
OSCAR_API oscar_status oscar_calibrate_upload(oscar_ctx_t* ctx, int layer,
                                    const float* R_k, const float* R_v,
                                    const float* T_k, const float* T_v, void* stream);

/* Write path ([QBIT] serving pipeline: rotate, clip, quantize, pack; [ABS]:
 * fused write kernel). Quantizes n new tokens into INT2 slots.
 *   k, v:      DEVICE bf16 [n][H_kv][d], unrotated.
 *   slots:     DEVICE int64 [n], INT2 slot of each token (page*P + row).
 *              Slots must be distinct.
 *   int2_pool: DEVICE INT2 pool, int2_pool_pages pages (layout above).
 * Writes codes and scale/zero for every head, K and V.
 * Asynchronous on `stream`. n == 0 is a no-op. */
OSCAR_API oscar_status oscar_write_tokens(oscar_ctx_t* ctx, int layer,
                                const void* k, const void* v,
                                const int64_t* slots, int n,
                                void* int2_pool, int64_t int2_pool_pages, void* stream);

/* Demote ([QBIT] serving pipeline: as decoding advances, the oldest BF16 recent
 * token is rotated, clipped, quantized and packed into the INT2 history).
 * Reads the BF16 K/V rows at src_slots and writes their INT2 form at dst_slots.
 *   bf16_pool: DEVICE BF16 pool, bf16_pool_pages pages.
 *   src_slots: DEVICE int64 [n], slots in the BF16 pool.
 *   dst_slots: DEVICE int64 [n], distinct slots in the INT2 pool.
 * The caller then advances its recent ring and its lengths.
 * Asynchronous on `stream`. n == 0 is a no-op. */
OSCAR_API oscar_status oscar_demote_recent(oscar_ctx_t* ctx, int layer,
                                 const void* bf16_pool, int64_t bf16_pool_pages,
                                 const int64_t* src_slots,
                                 void* int2_pool, int64_t int2_pool_pages,
                                 const int64_t* dst_slots, int n, void* stream);

/* Bytes of device workspace oscar_decode needs for `batch` sequences whose
 * INT2 history holds at most max_hist tokens. Returns 0 on bad arguments
 * (NULL ctx, negative sizes, batch above 65535). */
OSCAR_API size_t oscar_decode_workspace_size(const oscar_ctx_t* ctx, int batch, int max_hist);

/* Paged decode attention for one layer ([QBIT] serving pipeline, decode: INT2
 * unpack + scale/zero dequant + float accumulation, a BF16 part for
 * sink/recent, and an online-softmax merge; [ABS]: paged layouts and prefix
 * caching preserved).
 *   q:            DEVICE bf16 [batch][H_q][d].
 *   int2_pool:    DEVICE INT2 pool of int2_pool_pages pages.
 *   int2_tables:  DEVICE int32 [batch][int2_table_stride].
 *   hist_len:     DEVICE int32 [batch]. Every entry is <= max_hist and
 *                 <= P * int2_table_stride. 0 means no history.
 *   bf16_pool:    DEVICE BF16 pool of bf16_pool_pages pages.
 *   bf16_tables:  DEVICE int32 [batch][bf16_table_stride].
 *   bf16_len:     DEVICE int32 [batch], <= sink + recent and
 *                 <= P * bf16_table_stride. 0 means no BF16 tokens.
 *   out:          DEVICE fp32 [batch][H_q][d]. A sequence with no tokens at all
 *                 gets zeros.
 *   workspace:    DEVICE, >= oscar_decode_workspace_size(ctx, batch, max_hist)
 *                 bytes, 256-byte aligned. It holds split partials and is
 *                 scratch between calls.
 * Asynchronous on `stream`. batch == 0 is a no-op; batch > 65535 returns
 * OSCAR_ERR_UNSUPPORTED. */
OSCAR_API oscar_status oscar_decode(oscar_ctx_t* ctx, int layer, const void* q,
                          const void* int2_pool, int64_t int2_pool_pages,
                          const int32_t* int2_tables, int int2_table_stride,
                          const int32_t* hist_len, int max_hist,
                          const void* bf16_pool, int64_t bf16_pool_pages,
                          const int32_t* bf16_tables, int bf16_table_stride,
                          const int32_t* bf16_len,
                          float* out, void* workspace, size_t workspace_bytes,
                          int batch, void* stream);

/* Paged decode attention when every sequence of the batch starts with the
 * same INT2 pages (a radix prefix-cache hit; [QBIT] serving pipeline: radix
 * prefix cache; [ABS]: prefix caching preserved). Sequence b's INT2 history
 * is the shared prefix, prefix_pages full pages (16 * prefix_pages tokens)
 * listed once in prefix_table, followed by its own hist_len[b] tokens in
 * int2_tables[b] (logical page 0 of that table holds token 16*prefix_pages).
 * The result equals oscar_decode over the concatenated tables. The shared
 * pages are read once per (KV head, group of four sequences) instead of once
 * per sequence.
 *   prefix_table: DEVICE int32 [prefix_pages] page ids in the INT2 pool.
 *   prefix_pages: >= 0; 0 makes the call an oscar_decode.
 * Other arguments as for oscar_decode; hist_len / max_hist count only the
 * tokens after the prefix. The BF16 segment (sink + recent) stays per
 * sequence. workspace: >= oscar_decode_shared_prefix_workspace_size(ctx,
 * batch, prefix_pages, max_hist) bytes, 256-byte aligned. Asynchronous on
 * `stream`. */
OSCAR_API size_t oscar_decode_shared_prefix_workspace_size(const oscar_ctx_t* ctx, int batch, int prefix_pages,
                                                          int max_hist);
OSCAR_API oscar_status oscar_decode_shared_prefix(oscar_ctx_t* ctx, int layer, const void* q,
                                                  const void* int2_pool, int64_t int2_pool_pages,
                                                  const int32_t* prefix_table, int prefix_pages,
                                                  const int32_t* int2_tables, int int2_table_stride,
                                                  const int32_t* hist_len, int max_hist,
                                                  const void* bf16_pool, int64_t bf16_pool_pages,
                                                  const int32_t* bf16_tables, int bf16_table_stride,
                                                  const int32_t* bf16_len,
                                                  float* out, void* workspace, size_t workspace_bytes,
                                                  int batch, void* stream);

/* oscar_decode without a caller workspace. The pages have no counterpart for
 * this call. It exists for callers that cannot allocate device memory:
 *   - a host engine that only hands the op its input and output buffers;
 *   - a serving loop whose allocator owns the whole device budget;
 *   - a decode step recorded under CUDA stream capture, where cudaMalloc is
 *     not permitted.
 * The scratch is one static device array of 8 MiB, which every GPU that loads
 * the library holds until process exit. Arguments and results are those of
 * oscar_decode, minus the workspace. Sizes whose
 * oscar_decode_workspace_size(ctx, batch, max_hist) exceeds 8 MiB are rejected
 * with OSCAR_ERR_WORKSPACE before anything is launched. The call allocates
 * nothing (no cudaMalloc/cudaFree or allocating library routine).
 * The first call on a device looks up the array's device address; make that
 * first call before any stream capture. All calls share the one array, and it
 * keeps the last call's contents. Calls whose work overlaps on the GPU (e.g.
 * on two streams at once) race on it and must be serialised by the caller.
 * Nothing in it has to start at zero. Asynchronous on `stream` like
 * oscar_decode. */
OSCAR_API oscar_status oscar_decode_static_workspace(oscar_ctx_t* ctx, int layer, const void* q,
                                                     const void* int2_pool, int64_t int2_pool_pages,
                                                     const int32_t* int2_tables, int int2_table_stride,
                                                     const int32_t* hist_len, int max_hist,
                                                     const void* bf16_pool, int64_t bf16_pool_pages,
                                                     const int32_t* bf16_tables, int bf16_table_stride,
                                                     const int32_t* bf16_len, float* out, int batch, void* stream);

/* Bytes of one INT2 page (all heads, K and V) and of one BF16 page. */
/* Offline calibration targets on the GPU ([QBIT] section "OSCAR aligns the
 * rotation with attention": per layer and per head, the key target Q^T Q and
 * the score-weighted value target V^T S^T S V, estimated from a few
 * calibration samples). The host then takes their eigenvectors U and forms
 * R = U H P and the clip thresholds. This call needs no context.
 *   q_cal:    DEVICE fp32 [n][H_q][d] calibration queries.
 *   k_cal, v_cal: DEVICE fp32 [m][H_kv][d] calibration keys and values.
 *   target_k, target_v: DEVICE fp64 [H_kv][d][d], written. For KV head h, the
 *             key target stacks the queries of its H_q/H_kv query heads as
 *             rows (n * H_q/H_kv rows). S is the row-wise softmax of
 *             sm_scale * Q K^T over the m keys of head h, with no mask, and
 *             the value target is (S V)^T (S V).
 *   workspace: DEVICE, >= oscar_calibration_workspace_size(n, H_q, H_kv, d)
 *             bytes, 256-byte aligned (the rows of S V, fp64).
 * Supported: d in {64, 128}; H_q a multiple of H_kv; n >= 1; 1 <= m <= 8192.
 * Other sizes return OSCAR_ERR_UNSUPPORTED or OSCAR_ERR_INVALID_ARG before
 * anything is launched. Asynchronous on `stream`. All arithmetic is fp64. */
OSCAR_API size_t oscar_calibration_workspace_size(int n, int n_q_heads, int n_kv_heads, int head_dim);
OSCAR_API oscar_status oscar_calibration_targets(const float* q_cal, const float* k_cal, const float* v_cal,
                                                 int n, int m, int n_q_heads, int n_kv_heads, int head_dim,
                                                 double sm_scale, double* target_k, double* target_v,
                                                 void* workspace, size_t workspace_bytes, void* stream);

OSCAR_API size_t oscar_int2_page_bytes(const oscar_ctx_t* ctx);
OSCAR_API size_t oscar_bf16_page_bytes(const oscar_ctx_t* ctx);

/* Kernel classes for oscar_profile_read. */
typedef enum {
    OSCAR_KERNEL_WRITE = 0,   /* write / demote kernel */
    OSCAR_KERNEL_QROT = 1,    /* query rotation q @ R_k */
    OSCAR_KERNEL_SPLIT = 2,   /* split-K partials over INT2 history and BF16 segment */
    OSCAR_KERNEL_MERGE = 3,   /* online-softmax merge + un-rotation */
    OSCAR_KERNEL_COUNT = 4
} oscar_kernel_id;

/* Measurement hook (no counterpart on the pages): while enabled, every launch
 * is bracketed by a pair of CUDA events recorded on the launching stream.
 * Off by default. enable = 0 stops recording and keeps what was recorded. */
OSCAR_API oscar_status oscar_profile_enable(oscar_ctx_t* ctx, int enable);

/* Total device time (ms) and launch count of one kernel class since the last
 * read. Synchronizes on the recorded events, then clears them. */
OSCAR_API oscar_status oscar_profile_read(oscar_ctx_t* ctx, int kernel, double* total_ms, long long* launches);

/* Static text for a status code. */
OSCAR_API const char* oscar_status_string(oscar_status status);

/* One-line description of the calling thread's most recent failure ("" if none). */
OSCAR_API const char* oscar_last_error(void);

/* Read and clear the device error word (debug_bounds mode).
 * Synchronizes the device. Returns OSCAR_OK if nothing was recorded, otherwise
 * OSCAR_ERR_BOUNDS, with *kind set to the check that failed (1 slot, 2 page
 * id, 3 length, 4 a page copy that did not land within its bounded wait) and
 * *index to the offending value (either pointer may be NULL). Kind 4 is
 * recorded in every mode; kinds 1-3 only with debug_bounds. */
OSCAR_API oscar_status oscar_debug_error(oscar_ctx_t* ctx, int* kind, long long* index);

#ifdef __cplusplus
}
#endif

#endif /* OSCAR_H */
