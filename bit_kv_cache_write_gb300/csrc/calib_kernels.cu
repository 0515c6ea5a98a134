// Offline calibration targets on the GPU: the key target Q^T Q and the value target V^T S^T S V of
// every KV head, accumulated in fp64.
//
// Method: QbitAI article on OSCAR, section "OSCAR aligns the rotation with attention". A few
// calibration samples give, per layer and per head, the query covariance Q^T Q (which sets the key
// rotation) and the score-weighted value covariance V^T S^T S V (which sets the value rotation).
// The eigendecomposition, R = U H P and the clip thresholds then run on the host.
//
// Readings, the same as the rest of the library's calibration:
// - the key target of KV head h stacks the calibration queries of its g = H_q / H_kv query heads as
//   rows (n * g rows);
// - S is the row-wise softmax of sm_scale * Q K^T over the m calibration keys of that head, with no
//   mask;
// - V^T S^T S V = (S V)^T (S V).
//
// Work: sv_kernel writes the rows of S V (one block per query row and head), and gram_kernel forms
// X^T X for X = the query rows or the S V rows (32 x 32 output tiles, rows staged through shared
// memory 32 at a time). All arithmetic is fp64. Sizes are small (n * g x m logits per head), so
// these are plain CUDA-core kernels.

#include <cuda_runtime.h>
#include <cmath>
#include <cstdint>

#include "oscar_internal.h"

namespace oscar {
namespace {

constexpr int kTileG = 32;                 // output tile of the Gram kernel
constexpr int kRowsG = 8;                  // thread rows of the Gram kernel: 32 x 8 threads, 4 outputs each

// Row r of the key-target matrix of KV head h: query head h * g + r % g of calibration sample r / g.
struct QueryRows {
    const float* q;
    int g, h_q, d;
    __device__ double at(int h, int r, int c) const {
        return (double)q[((size_t)(r / g) * h_q + (size_t)h * g + r % g) * d + c];
    }
};

// Row r of S V for KV head h, as written by sv_kernel: [H_kv][rows][d].
struct SvRows {
    const double* sv;
    int rows, d;
    __device__ double at(int h, int r, int c) const { return sv[((size_t)h * rows + r) * d + c]; }
};

// C_h = X_h^T X_h (d x d) for every head h = blockIdx.z.
template <class Rows>
__global__ void __launch_bounds__(kTileG * kRowsG) gram_kernel(Rows x, int n_rows, int d, double* __restrict__ c) {
    __shared__ double xs[kTileG][kTileG + 1], ys[kTileG][kTileG + 1];
    const int h = blockIdx.z, i0 = blockIdx.y * kTileG, j0 = blockIdx.x * kTileG;
    const int tx = threadIdx.x % kTileG, ty = threadIdx.x / kTileG;
    double acc[kTileG / kRowsG] = {};
    for (int r0 = 0; r0 < n_rows; r0 += kTileG) {
        for (int k = ty; k < kTileG; k += kRowsG) {
            const int r = r0 + k;
            xs[k][tx] = (r < n_rows && i0 + tx < d) ? x.at(h, r, i0 + tx) : 0.0;
            ys[k][tx] = (r < n_rows && j0 + tx < d) ? x.at(h, r, j0 + tx) : 0.0;
        }
        __syncthreads();
        for (int k = 0; k < kTileG; ++k) {
            const double y = ys[k][tx];
#pragma unroll
            for (int m = 0; m < kTileG / kRowsG; ++m) acc[m] = fma(xs[k][ty + kRowsG * m], y, acc[m]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int m = 0; m < kTileG / kRowsG; ++m) {
        const int i = i0 + ty + kRowsG * m, j = j0 + tx;
        if (i < d && j < d) c[((size_t)h * d + i) * d + j] = acc[m];
    }
}

__device__ double block_reduce(double v, bool is_max, double* red) {
    const int lane = threadIdx.x % 32, warp = threadIdx.x / 32, warps = blockDim.x / 32;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const double u = __shfl_xor_sync(0xffffffffu, v, o);
        v = is_max ? fmax(v, u) : v + u;
    }
    __syncthreads();                         // red is reused across calls
    if (lane == 0) red[warp] = v;
    __syncthreads();
    double r = red[0];
    for (int w = 1; w < warps; ++w) r = is_max ? fmax(r, red[w]) : r + red[w];
    return r;
}

// Row r (= blockIdx.x) of S V for KV head h (= blockIdx.y): the scores of query row r against the m
// keys of head h, their softmax, and the weighted sum of the values. Block of d threads.
// Dynamic shared memory: m + d doubles.
__global__ void sv_kernel(const float* __restrict__ q, const float* __restrict__ k, const float* __restrict__ v,
                          int rows, int m, int g, int h_q, int h_kv, int d, double sm_scale, double* __restrict__ sv) {
    extern __shared__ double sbuf[];
    __shared__ double red[32];
    double* e = sbuf;                        // [m]
    double* qr = sbuf + m;                   // [d]
    const int r = blockIdx.x, h = blockIdx.y, t = threadIdx.x;
    const float* qp = q + ((size_t)(r / g) * h_q + (size_t)h * g + r % g) * d;
    for (int c = t; c < d; c += blockDim.x) qr[c] = (double)qp[c];
    __syncthreads();
    double mx = -INFINITY;
    for (int b = t; b < m; b += blockDim.x) {
        const float* kp = k + ((size_t)b * h_kv + h) * d;
        double s = 0.0;
        for (int c = 0; c < d; ++c) s = fma((double)kp[c], qr[c], s);
        s *= sm_scale;
        e[b] = s;
        mx = fmax(mx, s);
    }
    mx = block_reduce(mx, true, red);
    double sum = 0.0;
    for (int b = t; b < m; b += blockDim.x) {
        const double x = exp(e[b] - mx);
        e[b] = x;
        sum += x;
    }
    sum = block_reduce(sum, false, red);     // its barriers also publish every e[b]
    for (int c = t; c < d; c += blockDim.x) {
        double acc = 0.0;
        for (int b = 0; b < m; ++b) acc = fma(e[b], (double)v[((size_t)b * h_kv + h) * d + c], acc);
        sv[((size_t)h * rows + r) * d + c] = acc / sum;
    }
}

}  // namespace

size_t calibration_workspace_bytes(int n, int h_q, int h_kv, int d) {
    return (size_t)h_kv * n * (h_q / h_kv) * d * sizeof(double);
}

cudaError_t launch_calibration_targets(const float* q, const float* k, const float* v, int n, int m, int h_q, int h_kv,
                                       int d, double sm_scale, double* target_k, double* target_v, double* sv_rows,
                                       cudaStream_t st) {
    const int g = h_q / h_kv;
    const int rows = n * g;
    const dim3 gram_grid((d + kTileG - 1) / kTileG, (d + kTileG - 1) / kTileG, h_kv);
    gram_kernel<QueryRows><<<gram_grid, kTileG * kRowsG, 0, st>>>(QueryRows{q, g, h_q, d}, rows, d, target_k);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const size_t smem = (size_t)(m + d) * sizeof(double);
    const cudaError_t attr = smem_opt_in<sv_kernel>(kCalibMaxSmem);
    if (attr != cudaSuccess) return attr;
    sv_kernel<<<dim3(rows, h_kv), d, smem, st>>>(q, k, v, rows, m, g, h_q, h_kv, d, sm_scale, sv_rows);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    gram_kernel<SvRows><<<gram_grid, kTileG * kRowsG, 0, st>>>(SvRows{sv_rows, rows, d}, rows, d, target_v);
    return cudaGetLastError();
}

}  // namespace oscar
