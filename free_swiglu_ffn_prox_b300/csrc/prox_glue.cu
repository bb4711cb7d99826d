// prox_glue.cu -- residual + RMS normalisation between stacked FFN layers.
// No page defines this glue; the plain reading of a pre-norm residual stream
// without a learned gain:  z = x + y,  x_next = bf16_rne(z / sqrt(mean(z^2) + eps)).
#include "prox_internal.cuh"

namespace prox {
namespace {

constexpr int kThreads = 1024;

__global__ void __launch_bounds__(kThreads)
k_residual_rmsnorm(const uint16_t* __restrict__ x, const float* __restrict__ y, float eps,
                   uint16_t* __restrict__ x_next, int d) {
    __shared__ float wsum[kThreads / 32];
    float ss = 0.0f;
    for (int i = threadIdx.x; i < d; i += kThreads) {
        const float z = __uint_as_float((uint32_t)x[i] << 16) + y[i];
        ss = fmaf(z, z, ss);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((threadIdx.x & 31) == 0) wsum[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.0f;
    for (int w = 0; w < kThreads / 32; ++w) tot += wsum[w];
    const float inv = 1.0f / sqrtf(tot / (float)d + eps);
    for (int i = threadIdx.x; i < d; i += kThreads) {
        const float z = __uint_as_float((uint32_t)x[i] << 16) + y[i];
        x_next[i] = __bfloat16_as_ushort(__float2bfloat16_rn(z * inv));
    }
}

}  // namespace

cudaError_t launch_residual_rmsnorm(int d, const uint16_t* x, const float* y, float eps,
                                    uint16_t* x_next, cudaStream_t stream) {
    k_residual_rmsnorm<<<1, kThreads, 0, stream>>>(x, y, eps, x_next, d);
    return cudaGetLastError();
}

}  // namespace prox
