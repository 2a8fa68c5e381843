// Masked Adam: one Adam step on the parameter entries a sparse gradient materializes.
//
// SparseAdam page (tensorplay.optim.sparse_adam.SparseAdam): the first and second moments
// and the parameter change only where the sparse gradient holds a value; every other entry
// is left untouched (defaults lr 1e-3, betas (0.9, 0.999), eps 1e-8, maximize False). The
// update is Adam's with bias-corrected moments:
//     m = b1 m + (1 - b1) g,  v = b2 v + (1 - b2) g^2,
//     p -= lr * (m / (1 - b1^t)) / (sqrt(v / (1 - b2^t)) + eps)
// evaluated in fp32 as p -= (lr / bc1) * m / (sqrt(v) / sqrt(bc2) + eps), g negated when
// maximizing. Two layouts of the gradient:
//   * values of the parameter's own sparsity pattern (the RoSA adapter: parameter, moments
//     and gradient are the nnz values of one CSR mask): entry g updates position g;
//   * a CSR gradient (row_offsets, col_idx) over a dense m x n parameter: entry k of row i
//     updates position i * n + col[k].
// Each kernel streams the gradient once and reads and writes parameter and moments once
// per materialized entry: HBM-bound.
#include "common.cuh"
#include "internal.h"

namespace spops {
namespace {

struct AdamCoef {
    float b1, b2, omb1, omb2, step_size, inv_sqrt_bc2, eps, sign;
};

__device__ __forceinline__ void adam_entry(float& p, float& m, float& v, float g, const AdamCoef& c) {
    const float d = c.sign * g;
    m = c.b1 * m + c.omb1 * d;
    v = c.b2 * v + c.omb2 * (d * d);
    const float denom = sqrtf(v) * c.inv_sqrt_bc2 + c.eps;
    p = p - c.step_size * (m / denom);
}

// Identity layout, four entries per thread with 16-byte loads where the pointers allow.
template <typename G, bool kVec>
__global__ void __launch_bounds__(256) adam_values_kernel(float* __restrict__ param, float* __restrict__ exp_avg,
                                                         float* __restrict__ exp_avg_sq, const G* __restrict__ grad,
                                                         int64_t count, AdamCoef c) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    if constexpr (kVec) {
        const int64_t n4 = count / 4;
        for (int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; q < n4; q += stride) {
            float4 p = reinterpret_cast<float4*>(param)[q];
            float4 m = reinterpret_cast<float4*>(exp_avg)[q];
            float4 v = reinterpret_cast<float4*>(exp_avg_sq)[q];
            float g[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) g[e] = Elt<G>::to_f(grad[q * 4 + e]);
            adam_entry(p.x, m.x, v.x, g[0], c);
            adam_entry(p.y, m.y, v.y, g[1], c);
            adam_entry(p.z, m.z, v.z, g[2], c);
            adam_entry(p.w, m.w, v.w, g[3], c);
            reinterpret_cast<float4*>(param)[q] = p;
            reinterpret_cast<float4*>(exp_avg)[q] = m;
            reinterpret_cast<float4*>(exp_avg_sq)[q] = v;
        }
        for (int64_t i = n4 * 4 + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < count; i += stride) {
            float p = param[i], m = exp_avg[i], v = exp_avg_sq[i];
            adam_entry(p, m, v, Elt<G>::to_f(grad[i]), c);
            param[i] = p;
            exp_avg[i] = m;
            exp_avg_sq[i] = v;
        }
    } else {
        for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < count; i += stride) {
            float p = param[i], m = exp_avg[i], v = exp_avg_sq[i];
            adam_entry(p, m, v, Elt<G>::to_f(grad[i]), c);
            param[i] = p;
            exp_avg[i] = m;
            exp_avg_sq[i] = v;
        }
    }
}

// CSR gradient over a dense parameter: a warp per row (rows visited in order, strided by
// warps), lanes over the row's entries.
template <typename G, typename I>
__global__ void __launch_bounds__(256) adam_csr_kernel(float* __restrict__ param, float* __restrict__ exp_avg,
                                                      float* __restrict__ exp_avg_sq, const G* __restrict__ grad,
                                                      const int32_t* __restrict__ ro, const I* __restrict__ col,
                                                      int32_t m, int32_t n, AdamCoef c) {
    const int lane = threadIdx.x & 31;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t i = warp; i < m; i += nwarps) {
        const int32_t k0 = ro[i], k1 = ro[i + 1];
        float* prow = param + i * n;
        float* mrow = exp_avg + i * n;
        float* vrow = exp_avg_sq + i * n;
        for (int32_t k = k0 + lane; k < k1; k += 32) {
            const int j = idx_of(col[k]);
            float p = prow[j], mm = mrow[j], v = vrow[j];
            adam_entry(p, mm, v, Elt<G>::to_f(grad[k]), c);
            prow[j] = p;
            mrow[j] = mm;
            vrow[j] = v;
        }
    }
}

AdamCoef coef(int32_t step, double lr, double beta1, double beta2, double eps, int maximize) {
    const double bc1 = 1.0 - pow(beta1, (double)step), bc2 = 1.0 - pow(beta2, (double)step);
    AdamCoef c;
    c.b1 = (float)beta1;
    c.b2 = (float)beta2;
    c.omb1 = (float)(1.0 - beta1);
    c.omb2 = (float)(1.0 - beta2);
    c.step_size = (float)(lr / bc1);
    c.inv_sqrt_bc2 = (float)(1.0 / sqrt(bc2));
    c.eps = (float)eps;
    c.sign = maximize ? -1.f : 1.f;
    return c;
}

template <typename G>
cudaError_t run_values(float* p, float* m, float* v, const void* g, int64_t count, const AdamCoef& c, cudaStream_t s) {
    const bool vec = ((uintptr_t)p | (uintptr_t)m | (uintptr_t)v) % 16 == 0;
    const int64_t work = vec ? (count + 3) / 4 : count;
    const int grid = (int)max64(1, min64((int64_t)device_props().sm_count * 8, (work + 255) / 256));
    if (vec) adam_values_kernel<G, true><<<grid, 256, 0, s>>>(p, m, v, static_cast<const G*>(g), count, c);
    else adam_values_kernel<G, false><<<grid, 256, 0, s>>>(p, m, v, static_cast<const G*>(g), count, c);
    count_launches(1);
    return cudaGetLastError();
}

template <typename G, typename I>
cudaError_t run_csr(float* p, float* m1, float* v, const void* g, const int32_t* ro, const void* col, int32_t m,
                    int32_t n, const AdamCoef& c, cudaStream_t s) {
    const int grid = (int)max64(1, min64((int64_t)device_props().sm_count * 8, ((int64_t)m + 7) / 8));
    adam_csr_kernel<G, I><<<grid, 256, 0, s>>>(p, m1, v, static_cast<const G*>(g), ro, static_cast<const I*>(col), m,
                                               n, c);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_masked_adam(int gdt, float* param, float* exp_avg, float* exp_avg_sq, const void* grad,
                               int64_t count, int32_t step, double lr, double beta1, double beta2, double eps,
                               int maximize, cudaStream_t s) {
    if (count <= 0) return cudaSuccess;
    const AdamCoef c = coef(step, lr, beta1, beta2, eps, maximize);
    if (gdt == kF32) return run_values<float>(param, exp_avg, exp_avg_sq, grad, count, c, s);
    if (gdt == kF16) return run_values<__half>(param, exp_avg, exp_avg_sq, grad, count, c, s);
    return run_values<__nv_bfloat16>(param, exp_avg, exp_avg_sq, grad, count, c, s);
}

cudaError_t launch_masked_adam_csr(int gdt, int it, float* param, float* exp_avg, float* exp_avg_sq, const void* grad,
                                   const int32_t* ro, const void* col, int32_t m, int32_t n, int32_t step, double lr,
                                   double beta1, double beta2, double eps, int maximize, cudaStream_t s) {
    if (m <= 0) return cudaSuccess;
    const AdamCoef c = coef(step, lr, beta1, beta2, eps, maximize);
    if (gdt == kF32)
        return it == kIdx16 ? run_csr<float, uint16_t>(param, exp_avg, exp_avg_sq, grad, ro, col, m, n, c, s)
                            : run_csr<float, int32_t>(param, exp_avg, exp_avg_sq, grad, ro, col, m, n, c, s);
    if (gdt == kF16)
        return it == kIdx16 ? run_csr<__half, uint16_t>(param, exp_avg, exp_avg_sq, grad, ro, col, m, n, c, s)
                            : run_csr<__half, int32_t>(param, exp_avg, exp_avg_sq, grad, ro, col, m, n, c, s);
    return it == kIdx16 ? run_csr<__nv_bfloat16, uint16_t>(param, exp_avg, exp_avg_sq, grad, ro, col, m, n, c, s)
                        : run_csr<__nv_bfloat16, int32_t>(param, exp_avg, exp_avg_sq, grad, ro, col, m, n, c, s);
}

}  // namespace spops
