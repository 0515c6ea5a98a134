// Internal declarations shared by the host API and the kernel translation units.
#pragma once

#include <cuda_runtime.h>
#include <atomic>
#include <cstdint>
#include <vector>

#include "../../include/oscar.h"

namespace oscar {

constexpr int kPage = 16;
constexpr int kMaxBf16 = 512;     // sink + recent upper bound
constexpr int kMaxBatch = 65535;  // sequences per decode call (one grid dimension per sequence)
constexpr float kLog2e = 1.4426950408889634f;
// The INT2 decode raises its running softmax max only when a logit passes it by more than
// 2^kSoftmaxHeadroomLog2 (log2 units), so weights stay at or below 2^8 between rescales.
constexpr int kSoftmaxHeadroomLog2 = 8;

// Opts kernel Kern into `bytes` of dynamic shared memory on the current device. The CUDA
// runtime applies the attribute per device, so it is set once for each device that launches
// the kernel (devices 0..63; a higher ordinal sets it on every call).
template <auto Kern>
cudaError_t smem_opt_in(size_t bytes) {
    static std::atomic<unsigned long long> done{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

// Per-layer device parameters. All pointers index into one allocation.
struct LayerParams {
    const float* r_k;      // [H_kv][d][d]
    const float* r_v;      // [H_kv][d][d]
    const float* r_vt;     // [H_kv][d][d], r_vt[h][i][c] = r_v[h][c][i]
    const float* t_k;      // [H_kv][d]
    const float* t_v;      // [H_kv][d]
    const float* pv_scale; // [H_kv] 2^sigma with 2^8 (2/3) max T_v 2^sigma <= 32752: keeps p s_v 2^sigma in fp16
    const float* rk_colmax;  // [H_kv] upper bound of max_c |R_k[:, c]|_2 (follows pv_scale)
    const uint16_t* r_img; // [K,V][H_kv][3][d*d] bf16 pieces of R as tensor-core operand images
    const float* r_kt;     // [H_kv][d][d], r_kt[h][c][i] = r_k[h][i][c] (exact recompute of the bulk write)
};

struct Shape {
    int h_q, h_kv, d, group, page, sink, recent;
    double sm_scale;
    int debug;
    int codebook;      // OSCAR_CODEBOOK_UNIFORM or OSCAR_CODEBOOK_LLOYD_MAX
};

// Opt-in launch timing: event pairs on the launching stream, per kernel class.
struct Profiler {
    bool on = false;
    std::vector<std::pair<cudaEvent_t, cudaEvent_t>> pending[OSCAR_KERNEL_COUNT];
};

// Records a start event at construction and a stop event at stop() on `st`.
class ProfScope {
  public:
    ProfScope(Profiler* p, int kernel, cudaStream_t st) : p_(p && p->on ? p : nullptr), k_(kernel), st_(st) {
        if (p_ && cudaEventCreate(&a_) == cudaSuccess && cudaEventCreate(&b_) == cudaSuccess)
            cudaEventRecord(a_, st_);
        else
            p_ = nullptr;
    }
    void stop() {
        if (!p_) return;
        cudaEventRecord(b_, st_);
        p_->pending[k_].push_back({a_, b_});
        p_ = nullptr;
    }
    ~ProfScope() { stop(); }

  private:
    Profiler* p_;
    int k_;
    cudaStream_t st_;
    cudaEvent_t a_ = nullptr, b_ = nullptr;
};

// Device error word: {kind, pad, index}.
struct DebugWord {
    int kind;
    int pad;
    long long index;
};

}  // namespace oscar

struct oscar_ctx {
    oscar_config_t cfg;
    oscar::Shape shape;
    int device;
    int num_sms;
    float* params;                 // all layers' parameters
    size_t params_floats;
    uint16_t* r_img;               // all layers' bf16 rotation images (tensor-core bulk write)
    size_t r_img_elems;            // per layer
    float* r_kt;                   // all layers' R_k^T, [layers][H_kv][d][d]
    std::vector<char> calibrated;  // per layer
    oscar::DebugWord* dbg;         // device error word
    oscar::Profiler prof;
};

namespace oscar {

LayerParams layer_params(const oscar_ctx* ctx, int layer);

// Records `st` and a formatted message as the calling thread's last failure; returns st.
oscar_status record_failure(oscar_status st, const char* fmt, ...);

// ---- write path (write_kernels.cu)
cudaError_t launch_write(const Shape& s, const LayerParams& p, int num_sms,
                         const void* k, const void* v, const int64_t* slots, int n,
                         const void* bf16_pool, int64_t bf16_pages, const int64_t* src_slots,
                         void* int2_pool, int64_t int2_pages, DebugWord* dbg, Profiler* prof, cudaStream_t st);

cudaError_t launch_transpose(const float* src, float* dst, int h, int d, cudaStream_t st);

// Lloyd-Max codebook write / demote (write_lm.cu), same arguments as launch_write.
cudaError_t launch_write_lm(const Shape& s, const LayerParams& p, int num_sms, const void* k, const void* v,
                            const int64_t* slots, int n, const void* bf16_pool, int64_t bf16_pages,
                            const int64_t* src_slots, void* int2_pool, int64_t int2_pages, DebugWord* dbg,
                            Profiler* prof, cudaStream_t st);

// Offline calibration targets (calib_kernels.cu): Q^T Q and (S V)^T (S V) per KV head, fp64.
constexpr int kCalibMaxKeys = 8192;                                     // m: calibration keys per head
constexpr size_t kCalibMaxSmem = (size_t)(kCalibMaxKeys + 128) * sizeof(double);
size_t calibration_workspace_bytes(int n, int h_q, int h_kv, int d);
cudaError_t launch_calibration_targets(const float* q, const float* k, const float* v, int n, int m, int h_q, int h_kv,
                                       int d, double sm_scale, double* target_k, double* target_v, double* sv_rows,
                                       cudaStream_t st);

// ---- tensor-core bulk write (write_tc.cu)
constexpr int kTcMinTokens = 512;     // below this the CUDA-core kernel is used
constexpr int kRotationPieces = 3;    // bf16 pieces of R in the operand images

// Whether a write of n tokens from k/v into int2_pool can take the tcgen05 path.
bool write_tc_eligible(const Shape& s, const void* k, const void* v, const void* int2_pool, int n);
cudaError_t launch_write_tc(const Shape& s, const LayerParams& p, int num_sms, const void* k, const void* v,
                            const int64_t* slots, int n, void* int2_pool, int64_t int2_pages, DebugWord* dbg,
                            Profiler* prof, cudaStream_t st);
// Host: the bf16 pieces of h_kv rotations r[h][i][j] (fp32) as swizzled K-major operand images,
// out[h][piece][d*d].
void build_rotation_images(const float* r, int h_kv, int d, uint16_t* out);

// ---- decode path (decode_kernels.cu)
struct DecodePlan {
    int int2_splits;        // splits over the INT2 history
    int pages_per_split;    // INT2 pages per split
    int bf16_splits;        // splits over the BF16 segment
    int bf16_pages_per_split;  // BF16 pages per BF16 split
    int prefix_pages_per_split;  // shared-prefix pages per prefix CTA (0 without a shared prefix)
    int prefix_splits;      // prefix partial slots per query head
    int n_prefix_ctas;      // prefix CTAs: prefix_splits x H_kv x sequence groups of the CTA's warp count
    int total_splits;       // partial slots per query head: prefix + INT2 + BF16
    size_t ws_partials;     // bytes of split partials
    size_t ws_qrot;         // bytes of rotated-query digits, exponents and digit sums
    size_t ws_counters;     // bytes of per-(sequence, KV head) tickets of the last-CTA merge
    bool fuse_merge;        // the split kernel merges (else the merge kernel runs)
    bool merge_per_unit;    // the merge kernel takes one (sequence, KV head) per CTA (else one query head)
    bool qprep_per_unit;    // q_prep takes one (sequence, KV head, slice) per CTA (else one query head)
    size_t ws_total;
};

DecodePlan plan_decode(const Shape& s, int num_sms, int batch, int max_hist, int prefix_pages = 0);

struct DecodeArgs {
    const void* q;
    const int32_t* prefix_table = nullptr; int prefix_pages = 0;   // shared prefix (cascade), or none
    const uint8_t* int2_pool; int64_t int2_pages;
    const int32_t* int2_tables; int int2_stride;
    const int32_t* hist_len; int max_hist;
    const uint16_t* bf16_pool; int64_t bf16_pages;
    const int32_t* bf16_tables; int bf16_stride;
    const int32_t* bf16_len;
    float* out;
    void* ws;
    int batch;
};

cudaError_t launch_decode(const Shape& s, const LayerParams& p, const DecodePlan& plan,
                          const DecodeArgs& a, DebugWord* dbg, Profiler* prof, cudaStream_t st);

}  // namespace oscar
