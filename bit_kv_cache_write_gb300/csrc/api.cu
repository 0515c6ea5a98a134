// Host implementation of the C ABI in include/oscar.h: argument validation,
// library-owned calibration buffers, launch planning and error reporting.

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <algorithm>
#include <new>
#include <vector>

#include "oscar_internal.h"

namespace {

thread_local char g_last_error[256] = "";

oscar_status fail(oscar_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
    return st;
}

oscar_status cuda_fail(cudaError_t e, const char* where) {
    return fail(OSCAR_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

// Host-side fault injection for tests: OSCAR_FAULT=alloc|upload|launch makes
// the matching step fail with its error status before touching the device.
bool fault(const char* what) {
    const char* f = std::getenv("OSCAR_FAULT");
    return f && std::strcmp(f, what) == 0;
}

bool pow2_in(int v, int lo, int hi) { return v >= lo && v <= hi && (v & (v - 1)) == 0; }

size_t layer_floats(const oscar::Shape& s) {
    return 3 * (size_t)s.h_kv * s.d * s.d + 2 * (size_t)s.h_kv * s.d + 2 * (size_t)s.h_kv;
}

// The context's buffers live on the device that was current at oscar_create; launches go to the
// current device, so the two must agree.
oscar_status check_device(const oscar_ctx_t* ctx) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev != ctx->device)
        return fail(OSCAR_ERR_INVALID_ARG, "current device %d is not the context's device %d", dev, ctx->device);
    return OSCAR_OK;
}

oscar_status check_ctx_layer(const oscar_ctx_t* ctx, int layer) {
    if (!ctx) return fail(OSCAR_ERR_INVALID_ARG, "ctx is NULL");
    if (layer < 0 || layer >= ctx->cfg.n_layers)
        return fail(OSCAR_ERR_INVALID_ARG, "layer %d outside [0, %d)", layer, ctx->cfg.n_layers);
    if (!ctx->calibrated[layer])
        return fail(OSCAR_ERR_NOT_CALIBRATED, "layer %d has no uploaded calibration", layer);
    return check_device(ctx);
}

}  // namespace

namespace oscar {

oscar_status record_failure(oscar_status st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
    va_end(ap);
    return st;
}

LayerParams layer_params(const oscar_ctx* ctx, int layer) {
    const Shape& s = ctx->shape;
    const size_t hdd = (size_t)s.h_kv * s.d * s.d, hd = (size_t)s.h_kv * s.d;
    const float* base = ctx->params + layer * layer_floats(s);
    LayerParams p;
    p.r_k = base;
    p.r_v = base + hdd;
    p.r_vt = base + 2 * hdd;
    p.t_k = base + 3 * hdd;
    p.t_v = base + 3 * hdd + hd;
    p.pv_scale = base + 3 * hdd + 2 * hd;
    p.rk_colmax = base + 3 * hdd + 2 * hd + s.h_kv;
    p.r_img = ctx->r_img + layer * ctx->r_img_elems;
    p.r_kt = ctx->r_kt + layer * hdd;
    return p;
}

}  // namespace oscar

extern "C" {

const char* oscar_status_string(oscar_status st) {
    switch (st) {
        case OSCAR_OK: return "ok";
        case OSCAR_ERR_INVALID_ARG: return "invalid argument";
        case OSCAR_ERR_UNSUPPORTED: return "unsupported shape";
        case OSCAR_ERR_NOT_CALIBRATED: return "layer not calibrated";
        case OSCAR_ERR_CUDA: return "CUDA error";
        case OSCAR_ERR_BOUNDS: return "index out of bounds";
        case OSCAR_ERR_NO_MEMORY: return "out of device memory";
        case OSCAR_ERR_WORKSPACE: return "workspace too small";
    }
    return "unknown status";
}

const char* oscar_last_error(void) { return g_last_error; }

oscar_status oscar_create(const oscar_config_t* cfg, oscar_ctx_t** out) {
    if (!out) return fail(OSCAR_ERR_INVALID_ARG, "out is NULL");
    *out = nullptr;
    if (!cfg) return fail(OSCAR_ERR_INVALID_ARG, "cfg is NULL");
    const oscar_config_t& c = *cfg;
    if (c.n_layers <= 0 || c.n_q_heads <= 0 || c.n_kv_heads <= 0 || c.sink < 0 || c.recent < 0)
        return fail(OSCAR_ERR_INVALID_ARG, "sizes must be positive (layers %d, heads %d/%d, sink %d, recent %d)",
                    c.n_layers, c.n_q_heads, c.n_kv_heads, c.sink, c.recent);
    if (c.head_dim != 64 && c.head_dim != 128)
        return fail(OSCAR_ERR_UNSUPPORTED, "head_dim %d not in {64, 128}", c.head_dim);
    if (!pow2_in(c.group, 32, 128) || c.group > c.head_dim)
        return fail(OSCAR_ERR_UNSUPPORTED, "group %d not in {32, 64, 128} or above head_dim", c.group);
    if (c.page_size != oscar::kPage) return fail(OSCAR_ERR_UNSUPPORTED, "page_size %d != 16", c.page_size);
    if (c.n_q_heads % c.n_kv_heads || !pow2_in(c.n_q_heads / c.n_kv_heads, 1, 8))
        return fail(OSCAR_ERR_UNSUPPORTED, "H_q/H_kv = %d/%d not in {1, 2, 4, 8}", c.n_q_heads, c.n_kv_heads);
    if (c.codebook != OSCAR_CODEBOOK_UNIFORM && c.codebook != OSCAR_CODEBOOK_LLOYD_MAX)
        return fail(OSCAR_ERR_UNSUPPORTED, "codebook %d not in {0 (uniform), 1 (Lloyd-Max)}", c.codebook);
    if (c.sink + c.recent > oscar::kMaxBf16)
        return fail(OSCAR_ERR_UNSUPPORTED, "sink + recent = %d above %d", c.sink + c.recent, oscar::kMaxBf16);
    if (fault("alloc")) return fail(OSCAR_ERR_NO_MEMORY, "injected allocation failure (OSCAR_FAULT=alloc)");

    oscar_ctx_t* ctx = new (std::nothrow) oscar_ctx_t();
    if (!ctx) return fail(OSCAR_ERR_NO_MEMORY, "host allocation failed");
    ctx->cfg = c;
    oscar::Shape& s = ctx->shape;
    s.h_q = c.n_q_heads; s.h_kv = c.n_kv_heads; s.d = c.head_dim; s.group = c.group;
    s.page = c.page_size; s.sink = c.sink; s.recent = c.recent;
    s.sm_scale = c.sm_scale > 0.0f ? (double)c.sm_scale : 1.0 / std::sqrt((double)c.head_dim);
    s.debug = c.debug_bounds ? 1 : 0;
    s.codebook = c.codebook;
    ctx->calibrated.assign(c.n_layers, 0);

    cudaError_t e = cudaGetDevice(&ctx->device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&ctx->num_sms, cudaDevAttrMultiProcessorCount, ctx->device);
    if (e != cudaSuccess) { delete ctx; return cuda_fail(e, "device query"); }
    ctx->params_floats = layer_floats(s) * c.n_layers;
    e = cudaMalloc(&ctx->params, ctx->params_floats * sizeof(float));
    if (e != cudaSuccess) {
        delete ctx;
        cudaGetLastError();
        return fail(OSCAR_ERR_NO_MEMORY, "cudaMalloc of %zu calibration bytes: %s",
                    ctx->params_floats * sizeof(float), cudaGetErrorString(e));
    }
    ctx->r_img_elems = 2 * (size_t)s.h_kv * oscar::kRotationPieces * s.d * s.d;
    e = cudaMalloc(&ctx->r_img, ctx->r_img_elems * c.n_layers * sizeof(uint16_t));
    if (e == cudaSuccess) {
        e = cudaMalloc(&ctx->r_kt, (size_t)s.h_kv * s.d * s.d * c.n_layers * sizeof(float));
        if (e != cudaSuccess) cudaFree(ctx->r_img);
    }
    if (e != cudaSuccess) {
        cudaFree(ctx->params);
        delete ctx;
        cudaGetLastError();
        return fail(OSCAR_ERR_NO_MEMORY, "cudaMalloc of %zu rotation-image bytes: %s",
                    ctx->r_img_elems * c.n_layers * sizeof(uint16_t), cudaGetErrorString(e));
    }
    e = cudaMalloc(&ctx->dbg, sizeof(oscar::DebugWord));
    if (e == cudaSuccess) e = cudaMemset(ctx->dbg, 0, sizeof(oscar::DebugWord));
    if (e != cudaSuccess) {
        cudaFree(ctx->params);
        cudaFree(ctx->r_img);
        cudaFree(ctx->r_kt);
        delete ctx;
        cudaGetLastError();
        return fail(OSCAR_ERR_NO_MEMORY, "cudaMalloc of the error word: %s", cudaGetErrorString(e));
    }
    *out = ctx;
    return OSCAR_OK;
}

void oscar_destroy(oscar_ctx_t* ctx) {
    if (!ctx) return;
    for (auto& v : ctx->prof.pending)
        for (auto& pr : v) { cudaEventDestroy(pr.first); cudaEventDestroy(pr.second); }
    cudaFree(ctx->params);
    cudaFree(ctx->r_img);
    cudaFree(ctx->r_kt);
    cudaFree(ctx->dbg);
    delete ctx;
}

oscar_status oscar_calibrate_upload(oscar_ctx_t* ctx, int layer, const float* R_k, const float* R_v,
                                    const float* T_k, const float* T_v, void* stream) {
    if (!ctx) return fail(OSCAR_ERR_INVALID_ARG, "ctx is NULL");
    if (layer < 0 || layer >= ctx->cfg.n_layers)
        return fail(OSCAR_ERR_INVALID_ARG, "layer %d outside [0, %d)", layer, ctx->cfg.n_layers);
    if (!R_k || !R_v || !T_k || !T_v) return fail(OSCAR_ERR_INVALID_ARG, "calibration pointer is NULL");
    if (oscar_status dst = check_device(ctx); dst != OSCAR_OK) return dst;
    const oscar::Shape& s = ctx->shape;
    const size_t hdd = (size_t)s.h_kv * s.d * s.d, hd = (size_t)s.h_kv * s.d;
    for (size_t i = 0; i < hdd; ++i)
        if (!std::isfinite(R_k[i]) || !std::isfinite(R_v[i]))
            return fail(OSCAR_ERR_INVALID_ARG, "rotation entry %zu is not finite", i);
    for (size_t i = 0; i < hd; ++i)
        if (!(T_k[i] >= 0.0f) || !(T_v[i] >= 0.0f) || !std::isfinite(T_k[i]) || !std::isfinite(T_v[i]))
            return fail(OSCAR_ERR_INVALID_ARG, "threshold entry %zu is negative or not finite", i);
    if (fault("upload")) return fail(OSCAR_ERR_CUDA, "injected upload failure (OSCAR_FAULT=upload)");

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    oscar::LayerParams p = oscar::layer_params(ctx, layer);
    float* base = const_cast<float*>(p.r_k);
    cudaError_t e = cudaMemcpyAsync(base, R_k, hdd * sizeof(float), cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(base + hdd, R_v, hdd * sizeof(float), cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(const_cast<float*>(p.t_k), T_k, hd * sizeof(float), cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(const_cast<float*>(p.t_v), T_v, hd * sizeof(float), cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = oscar::launch_transpose(p.r_v, const_cast<float*>(p.r_vt), s.h_kv, s.d, st);
    if (e == cudaSuccess) e = oscar::launch_transpose(p.r_k, const_cast<float*>(p.r_kt), s.h_kv, s.d, st);
    // Per KV head power of two 2^sigma for the decode's p * s_v operand. Every stored V scale is
    // fp16((mx - mn) / 3) <= (2/3) max T_v (values are clipped to [-T, T]), so p * s_v * 2^sigma
    // stays at or below 32752 (fp16) while small weights keep clear of fp16 subnormals.
    std::vector<float> pvs(s.h_kv);
    for (int h = 0; h < s.h_kv; ++h) {
        float tmax = 0.0f;
        for (int c = 0; c < s.d; ++c) tmax = std::max(tmax, T_v[(size_t)h * s.d + c]);
        const double smax = std::max(1e-30, (2.0 / 3.0) * (double)tmax * 1.001);
        // weights reach 2^kSoftmaxHeadroomLog2 between the decode's lazy max updates
        int sigma = (int)std::floor(std::log2(32752.0 / smax)) - oscar::kSoftmaxHeadroomLog2;
        sigma = std::min(40, std::max(-40, sigma));
        pvs[h] = std::ldexp(1.0f, sigma);
    }
    // Per KV head, an upper bound of the largest column norm of R_k: |(q R_k)_c| <= |q| * max_c |R_k[:, c]|
    // bounds every rotated query channel, which fixes the query digits' common exponent without a
    // cross-channel maximum.
    for (int h = 0; h < s.h_kv; ++h) {
        double cmax = 0.0;
        for (int c = 0; c < s.d; ++c) {
            double n2 = 0.0;
            for (int i = 0; i < s.d; ++i) {
                const double r = R_k[((size_t)h * s.d + i) * s.d + c];
                n2 += r * r;
            }
            cmax = std::max(cmax, std::sqrt(n2));
        }
        pvs.push_back((float)(cmax * (1.0 + 1e-6)) + 1e-30f);
    }
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(const_cast<float*>(p.pv_scale), pvs.data(), 2 * s.h_kv * sizeof(float),
                            cudaMemcpyHostToDevice, st);
    // bf16 pieces of R_k and R_v as tensor-core operand images for the bulk write
    std::vector<uint16_t> img(ctx->r_img_elems);
    oscar::build_rotation_images(R_k, s.h_kv, s.d, img.data());
    oscar::build_rotation_images(R_v, s.h_kv, s.d, img.data() + ctx->r_img_elems / 2);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(const_cast<uint16_t*>(p.r_img), img.data(), ctx->r_img_elems * sizeof(uint16_t),
                            cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "calibration upload");
    ctx->calibrated[layer] = 1;
    return OSCAR_OK;
}

oscar_status oscar_write_tokens(oscar_ctx_t* ctx, int layer, const void* k, const void* v,
                                const int64_t* slots, int n, void* int2_pool, int64_t int2_pool_pages,
                                void* stream) {
    oscar_status st = check_ctx_layer(ctx, layer);
    if (st != OSCAR_OK) return st;
    if (n < 0) return fail(OSCAR_ERR_INVALID_ARG, "n = %d is negative", n);
    if (n == 0) return OSCAR_OK;
    if (!k || !v || !slots || !int2_pool) return fail(OSCAR_ERR_INVALID_ARG, "device pointer is NULL");
    if (int2_pool_pages <= 0) return fail(OSCAR_ERR_INVALID_ARG, "int2_pool_pages must be positive");
    if (fault("launch")) return fail(OSCAR_ERR_CUDA, "injected launch failure (OSCAR_FAULT=launch)");
    cudaError_t e = oscar::launch_write(ctx->shape, oscar::layer_params(ctx, layer), ctx->num_sms, k, v, slots, n,
                                        nullptr, 0, nullptr, int2_pool, int2_pool_pages, ctx->dbg, &ctx->prof,
                                        static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? OSCAR_OK : cuda_fail(e, "write kernel launch");
}

oscar_status oscar_demote_recent(oscar_ctx_t* ctx, int layer, const void* bf16_pool, int64_t bf16_pool_pages,
                                 const int64_t* src_slots, void* int2_pool, int64_t int2_pool_pages,
                                 const int64_t* dst_slots, int n, void* stream) {
    oscar_status st = check_ctx_layer(ctx, layer);
    if (st != OSCAR_OK) return st;
    if (n < 0) return fail(OSCAR_ERR_INVALID_ARG, "n = %d is negative", n);
    if (n == 0) return OSCAR_OK;
    if (!bf16_pool || !src_slots || !int2_pool || !dst_slots)
        return fail(OSCAR_ERR_INVALID_ARG, "device pointer is NULL");
    if (bf16_pool_pages <= 0 || int2_pool_pages <= 0)
        return fail(OSCAR_ERR_INVALID_ARG, "pool page counts must be positive");
    if (fault("launch")) return fail(OSCAR_ERR_CUDA, "injected launch failure (OSCAR_FAULT=launch)");
    cudaError_t e = oscar::launch_write(ctx->shape, oscar::layer_params(ctx, layer), ctx->num_sms, nullptr, nullptr,
                                        dst_slots, n, bf16_pool, bf16_pool_pages, src_slots, int2_pool,
                                        int2_pool_pages, ctx->dbg, &ctx->prof, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? OSCAR_OK : cuda_fail(e, "demote kernel launch");
}

size_t oscar_decode_workspace_size(const oscar_ctx_t* ctx, int batch, int max_hist) {
    if (!ctx || batch < 0 || batch > oscar::kMaxBatch || max_hist < 0) return 0;
    return oscar::plan_decode(ctx->shape, ctx->num_sms, batch, max_hist).ws_total;
}

size_t oscar_decode_shared_prefix_workspace_size(const oscar_ctx_t* ctx, int batch, int prefix_pages, int max_hist) {
    if (!ctx || batch < 0 || batch > oscar::kMaxBatch || max_hist < 0 || prefix_pages < 0) return 0;
    return oscar::plan_decode(ctx->shape, ctx->num_sms, batch, max_hist, prefix_pages).ws_total;
}

}  // extern "C"

namespace {

// Shared body of oscar_decode and oscar_decode_shared_prefix (prefix_pages = 0: no shared prefix).
oscar_status decode_call(oscar_ctx_t* ctx, int layer, const void* q, const void* int2_pool, int64_t int2_pool_pages,
                         const int32_t* prefix_table, int prefix_pages, const int32_t* int2_tables,
                         int int2_table_stride, const int32_t* hist_len, int max_hist, const void* bf16_pool,
                         int64_t bf16_pool_pages, const int32_t* bf16_tables, int bf16_table_stride,
                         const int32_t* bf16_len, float* out, void* workspace, size_t workspace_bytes, int batch,
                         void* stream) {
    oscar_status st = check_ctx_layer(ctx, layer);
    if (st != OSCAR_OK) return st;
    if (batch < 0 || max_hist < 0 || prefix_pages < 0)
        return fail(OSCAR_ERR_INVALID_ARG, "batch %d / max_hist %d / prefix_pages %d negative", batch, max_hist,
                    prefix_pages);
    if (batch == 0) return OSCAR_OK;
    if (batch > oscar::kMaxBatch)
        return fail(OSCAR_ERR_UNSUPPORTED, "batch %d above %d (one grid dimension per sequence)", batch, oscar::kMaxBatch);
    if (!q || !out || !hist_len || !bf16_len) return fail(OSCAR_ERR_INVALID_ARG, "device pointer is NULL");
    if (max_hist > 0 && (!int2_pool || !int2_tables || int2_table_stride <= 0 || int2_pool_pages <= 0))
        return fail(OSCAR_ERR_INVALID_ARG, "INT2 pool/tables missing while max_hist = %d", max_hist);
    if (prefix_pages > 0 && (!int2_pool || !prefix_table || int2_pool_pages <= 0))
        return fail(OSCAR_ERR_INVALID_ARG, "INT2 pool/prefix table missing while prefix_pages = %d", prefix_pages);
    if (!bf16_pool || !bf16_tables || bf16_table_stride <= 0 || bf16_pool_pages <= 0)
        return fail(OSCAR_ERR_INVALID_ARG, "BF16 pool/tables missing");
    if ((long long)max_hist > (long long)int2_table_stride * oscar::kPage && max_hist > 0)
        return fail(OSCAR_ERR_INVALID_ARG, "max_hist %d exceeds table stride %d pages", max_hist, int2_table_stride);
    const oscar::DecodePlan plan = oscar::plan_decode(ctx->shape, ctx->num_sms, batch, max_hist, prefix_pages);
    if (!workspace || workspace_bytes < plan.ws_total)
        return fail(OSCAR_ERR_WORKSPACE, "workspace %zu bytes, need %zu", workspace_bytes, plan.ws_total);
    if (reinterpret_cast<uintptr_t>(workspace) % 256)
        return fail(OSCAR_ERR_INVALID_ARG, "workspace is not 256-byte aligned");
    if (fault("launch")) return fail(OSCAR_ERR_CUDA, "injected launch failure (OSCAR_FAULT=launch)");
    oscar::DecodeArgs a;
    a.q = q;
    a.prefix_table = prefix_table; a.prefix_pages = prefix_pages;
    a.int2_pool = static_cast<const uint8_t*>(int2_pool); a.int2_pages = int2_pool_pages;
    a.int2_tables = int2_tables; a.int2_stride = int2_table_stride;
    a.hist_len = hist_len; a.max_hist = max_hist;
    a.bf16_pool = static_cast<const uint16_t*>(bf16_pool); a.bf16_pages = bf16_pool_pages;
    a.bf16_tables = bf16_tables; a.bf16_stride = bf16_table_stride;
    a.bf16_len = bf16_len;
    a.out = out; a.ws = workspace; a.batch = batch;
    cudaError_t e = oscar::launch_decode(ctx->shape, oscar::layer_params(ctx, layer), plan, a, ctx->dbg,
                                         &ctx->prof, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? OSCAR_OK : cuda_fail(e, "decode launch");
}

}  // namespace

extern "C" {

oscar_status oscar_decode(oscar_ctx_t* ctx, int layer, const void* q,
                          const void* int2_pool, int64_t int2_pool_pages,
                          const int32_t* int2_tables, int int2_table_stride,
                          const int32_t* hist_len, int max_hist,
                          const void* bf16_pool, int64_t bf16_pool_pages,
                          const int32_t* bf16_tables, int bf16_table_stride,
                          const int32_t* bf16_len,
                          float* out, void* workspace, size_t workspace_bytes,
                          int batch, void* stream) {
    return decode_call(ctx, layer, q, int2_pool, int2_pool_pages, nullptr, 0, int2_tables, int2_table_stride,
                       hist_len, max_hist, bf16_pool, bf16_pool_pages, bf16_tables, bf16_table_stride, bf16_len,
                       out, workspace, workspace_bytes, batch, stream);
}

oscar_status oscar_decode_shared_prefix(oscar_ctx_t* ctx, int layer, const void* q,
                                        const void* int2_pool, int64_t int2_pool_pages,
                                        const int32_t* prefix_table, int prefix_pages,
                                        const int32_t* int2_tables, int int2_table_stride,
                                        const int32_t* hist_len, int max_hist,
                                        const void* bf16_pool, int64_t bf16_pool_pages,
                                        const int32_t* bf16_tables, int bf16_table_stride,
                                        const int32_t* bf16_len,
                                        float* out, void* workspace, size_t workspace_bytes,
                                        int batch, void* stream) {
    return decode_call(ctx, layer, q, int2_pool, int2_pool_pages, prefix_table, prefix_pages, int2_tables,
                       int2_table_stride, hist_len, max_hist, bf16_pool, bf16_pool_pages, bf16_tables,
                       bf16_table_stride, bf16_len, out, workspace, workspace_bytes, batch, stream);
}

namespace {
bool calibration_shape_ok(int n, int h_q, int h_kv, int d) {
    return n >= 1 && h_kv >= 1 && h_q >= h_kv && h_q % h_kv == 0 && (d == 64 || d == 128);
}
}  // namespace

size_t oscar_calibration_workspace_size(int n, int n_q_heads, int n_kv_heads, int head_dim) {
    if (!calibration_shape_ok(n, n_q_heads, n_kv_heads, head_dim)) return 0;
    return oscar::calibration_workspace_bytes(n, n_q_heads, n_kv_heads, head_dim);
}

oscar_status oscar_calibration_targets(const float* q_cal, const float* k_cal, const float* v_cal, int n, int m,
                                       int n_q_heads, int n_kv_heads, int head_dim, double sm_scale,
                                       double* target_k, double* target_v, void* workspace, size_t workspace_bytes,
                                       void* stream) {
    if (!q_cal || !k_cal || !v_cal || !target_k || !target_v)
        return fail(OSCAR_ERR_INVALID_ARG, "device pointer is NULL");
    if (n < 1 || m < 1 || n_kv_heads < 1 || n_q_heads < n_kv_heads || n_q_heads % n_kv_heads ||
        !(sm_scale > 0.0) || !std::isfinite(sm_scale))
        return fail(OSCAR_ERR_INVALID_ARG, "n %d, m %d, heads %d/%d or sm_scale %g invalid", n, m, n_q_heads,
                    n_kv_heads, sm_scale);
    if ((head_dim != 64 && head_dim != 128) || m > oscar::kCalibMaxKeys)
        return fail(OSCAR_ERR_UNSUPPORTED, "head_dim %d or m %d (at most %d keys) unsupported", head_dim, m,
                    oscar::kCalibMaxKeys);
    const size_t need = oscar::calibration_workspace_bytes(n, n_q_heads, n_kv_heads, head_dim);
    if (!workspace || workspace_bytes < need)
        return fail(OSCAR_ERR_WORKSPACE, "workspace %zu bytes, need %zu", workspace_bytes, need);
    if (reinterpret_cast<uintptr_t>(workspace) % 256)
        return fail(OSCAR_ERR_INVALID_ARG, "workspace is not 256-byte aligned");
    cudaError_t e = oscar::launch_calibration_targets(q_cal, k_cal, v_cal, n, m, n_q_heads, n_kv_heads, head_dim,
                                                      sm_scale, target_k, target_v, static_cast<double*>(workspace),
                                                      static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? OSCAR_OK : cuda_fail(e, "calibration launch");
}

size_t oscar_int2_page_bytes(const oscar_ctx_t* ctx) {
    if (!ctx) return 0;
    const oscar::Shape& s = ctx->shape;
    return (size_t)s.h_kv * 2 * ((size_t)oscar::kPage * s.d / 4 + (size_t)oscar::kPage * (s.d / s.group) * 4);
}

size_t oscar_bf16_page_bytes(const oscar_ctx_t* ctx) {
    if (!ctx) return 0;
    const oscar::Shape& s = ctx->shape;
    return (size_t)s.h_kv * 2 * oscar::kPage * s.d * 2;
}

oscar_status oscar_profile_enable(oscar_ctx_t* ctx, int enable) {
    if (!ctx) return fail(OSCAR_ERR_INVALID_ARG, "ctx is NULL");
    ctx->prof.on = enable != 0;
    return OSCAR_OK;
}

oscar_status oscar_profile_read(oscar_ctx_t* ctx, int kernel, double* total_ms, long long* launches) {
    if (!ctx) return fail(OSCAR_ERR_INVALID_ARG, "ctx is NULL");
    if (kernel < 0 || kernel >= OSCAR_KERNEL_COUNT) return fail(OSCAR_ERR_INVALID_ARG, "kernel id %d", kernel);
    double sum = 0.0;
    long long cnt = 0;
    cudaError_t first = cudaSuccess;
    for (auto& pr : ctx->prof.pending[kernel]) {
        float ms = 0.0f;
        cudaError_t e = cudaEventSynchronize(pr.second);
        if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, pr.first, pr.second);
        if (e == cudaSuccess) { sum += ms; ++cnt; }
        else if (first == cudaSuccess) first = e;
        cudaEventDestroy(pr.first);
        cudaEventDestroy(pr.second);
    }
    ctx->prof.pending[kernel].clear();
    if (total_ms) *total_ms = sum;
    if (launches) *launches = cnt;
    return first == cudaSuccess ? OSCAR_OK : cuda_fail(first, "reading profile events");
}

oscar_status oscar_debug_error(oscar_ctx_t* ctx, int* kind, long long* index) {
    if (!ctx) return fail(OSCAR_ERR_INVALID_ARG, "ctx is NULL");
    oscar::DebugWord w{};
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpy(&w, ctx->dbg, sizeof(w), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemset(ctx->dbg, 0, sizeof(w));
    if (e != cudaSuccess) return cuda_fail(e, "reading the error word");
    if (kind) *kind = w.kind;
    if (index) *index = w.index;
    if (w.kind) return fail(OSCAR_ERR_BOUNDS, "bounds check %d failed at index %lld", w.kind, w.index);
    return OSCAR_OK;
}

}  // extern "C"
