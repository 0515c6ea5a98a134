// oscar_decode_static_workspace: paged decode for callers that cannot allocate device memory.
//
// oscar_decode needs a caller-supplied device workspace (split partials and the
// prepared query). Some callers cannot provide one. A plain-C host engine may
// only be handed the input and output buffers of the step. A serving loop may
// forbid device allocation on its decode path because its allocator owns the
// whole memory budget, or because the step runs inside CUDA stream capture,
// where cudaMalloc is not permitted. This entry point serves those callers. Its
// scratch is one file-scope device array of fixed size. It calls no allocator
// (no cudaMalloc, no cudaFree, no library routine that allocates). It then runs
// exactly the same kernels as oscar_decode.

#include <cstdint>
#include <mutex>

#include "oscar_internal.h"

namespace {

constexpr size_t kStaticWorkspaceBytes = size_t(8) << 20;   // per device, held until process exit
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_static_workspace[kStaticWorkspaceBytes];

std::mutex g_setup_mutex;
void* g_workspace_addr[kMaxDevices];   // device address of g_static_workspace, per device

// Host code cannot pass g_static_workspace itself to a kernel: in host code that name is
// a host-side stand-in, not a device address. The address is looked up once per device,
// with that device current.
oscar_status static_workspace(int device, void** out) {
    if (device < 0 || device >= kMaxDevices)
        return oscar::record_failure(OSCAR_ERR_UNSUPPORTED, "device %d beyond the %d supported for the static workspace",
                                     device, kMaxDevices);
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_workspace_addr[device]) {
        void* ptr = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&ptr, g_static_workspace);
        if (e != cudaSuccess || !ptr)
            return oscar::record_failure(OSCAR_ERR_CUDA, "cudaGetSymbolAddress of the static workspace: %s",
                                         cudaGetErrorString(e));
        g_workspace_addr[device] = ptr;
    }
    *out = g_workspace_addr[device];
    return OSCAR_OK;
}

}  // namespace

extern "C" oscar_status oscar_decode_static_workspace(
    oscar_ctx_t* ctx, int layer, const void* q, const void* int2_pool, int64_t int2_pool_pages,
    const int32_t* int2_tables, int int2_table_stride, const int32_t* hist_len, int max_hist,
    const void* bf16_pool, int64_t bf16_pool_pages, const int32_t* bf16_tables, int bf16_table_stride,
    const int32_t* bf16_len, float* out, int batch, void* stream) {
    if (!ctx) return oscar::record_failure(OSCAR_ERR_INVALID_ARG, "ctx is NULL");
    if (batch < 0 || max_hist < 0)
        return oscar::record_failure(OSCAR_ERR_INVALID_ARG, "batch %d / max_hist %d negative", batch, max_hist);
    if (batch > oscar::kMaxBatch)
        return oscar::record_failure(OSCAR_ERR_UNSUPPORTED, "batch %d above %d (one grid dimension per sequence)",
                                     batch, oscar::kMaxBatch);
    // the array's address is the one of the context's device, which must be the current device
    int device = 0;
    cudaError_t e = cudaGetDevice(&device);
    if (e != cudaSuccess) return oscar::record_failure(OSCAR_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (device != ctx->device)
        return oscar::record_failure(OSCAR_ERR_INVALID_ARG, "current device %d is not the context's device %d",
                                     device, ctx->device);
    const size_t need = oscar_decode_workspace_size(ctx, batch, max_hist);
    if (need > kStaticWorkspaceBytes)
        return oscar::record_failure(OSCAR_ERR_WORKSPACE,
                                     "batch %d with max_hist %d needs %zu workspace bytes; the static workspace "
                                     "holds %zu: use oscar_decode with a caller workspace",
                                     batch, max_hist, need, kStaticWorkspaceBytes);
    void* ws = nullptr;
    oscar_status st = static_workspace(device, &ws);
    if (st != OSCAR_OK) return st;
    // Nothing in the workspace has to start at zero: every split writes its whole
    // partial record and the query preparation writes all of its outputs before
    // they are read, so contents left by an earlier call are never observed.
    return oscar_decode(ctx, layer, q, int2_pool, int2_pool_pages, int2_tables, int2_table_stride, hist_len, max_hist,
                        bf16_pool, bf16_pool_pages, bf16_tables, bf16_table_stride, bf16_len, out, ws,
                        kStaticWorkspaceBytes, batch, stream);
}
