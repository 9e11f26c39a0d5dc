// Gate preparation from raw projections (FlashQLA PR #1, host-gating and
// in-kernel-gating commits): g = -exp(A_log) * softplus(a + dt_bias) with
// softplus(x) = x for x > 20 else log(1 + exp(x)); beta = sigmoid(b), doubled
// for the negative-eigenvalue variant.  One thread per (token, value-head);
// HBM-bound elementwise work.
#include "common.cuh"
#include "launch.h"

namespace gdr {
namespace {

template <typename T>
__global__ void gating_kernel(const T* __restrict__ a, const float* __restrict__ dt_bias,
                              const float* __restrict__ A_log, const T* __restrict__ b,
                              float* __restrict__ g, T* __restrict__ beta, int64_t n, int Hv,
                              float beta_mul) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    const int h = (int)(i % Hv);
    const float x = to_f(a[i]) + dt_bias[h];
    const float sp = x > 20.f ? x : log1pf(expf(x));
    g[i] = -expf(A_log[h]) * sp;
    beta[i] = from_f<T>(beta_mul / (1.f + expf(-to_f(b[i]))));
}

}  // namespace

cudaError_t launch_gating(const GatingArgs& a, cudaStream_t stream) {
    const int64_t n = a.T * a.Hv;
    const unsigned blocks = (unsigned)((n + 255) / 256);
    const float mul = (a.flags & 2) ? 2.f : 1.f;
    KernelTimer kt("gating", stream);
    if (a.dtype == 0)
        gating_kernel<__nv_bfloat16><<<blocks, 256, 0, stream>>>(
            static_cast<const __nv_bfloat16*>(a.a), a.dt_bias, a.A_log,
            static_cast<const __nv_bfloat16*>(a.b), a.g, static_cast<__nv_bfloat16*>(a.beta), n, a.Hv, mul);
    else
        gating_kernel<float><<<blocks, 256, 0, stream>>>(
            static_cast<const float*>(a.a), a.dt_bias, a.A_log, static_cast<const float*>(a.b), a.g,
            static_cast<float*>(a.beta), n, a.Hv, mul);
    return cudaGetLastError();
}

}  // namespace gdr
