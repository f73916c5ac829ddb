// harness.cu -- the step that chains MoE layers in the multi-layer workloads (not part of the
// routed-expert layer itself): x_next = bf16(RMSNorm(x + y)), unit weight.
#include "moe_internal.cuh"

namespace fp4moe {

namespace {

constexpr int kNormThreads = 256;

// One block per token.  v = x + y in fp32 (both bf16), mean of v^2 by a fixed-order block
// reduction, x_next = bf16_RNE(v / sqrt(mean + eps)).
__global__ void __launch_bounds__(kNormThreads) residual_rmsnorm_kernel(int d, const uint16_t* __restrict__ x,
                                                                      const uint16_t* __restrict__ y, float eps,
                                                                      uint16_t* __restrict__ out) {
    __shared__ float red[kNormThreads / 32];
    const size_t base = (size_t)blockIdx.x * d;
    float ss = 0.f;
    for (int i = threadIdx.x; i < d; i += kNormThreads) {
        const float v = bf16_to_f32(x[base + i]) + bf16_to_f32(y[base + i]);
        ss = fmaf(v, v, ss);
    }
    ss = warp_sum(ss);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kNormThreads / 32; ++w) tot += red[w];
    const float inv = 1.0f / sqrtf(tot / (float)d + eps);
    for (int i = threadIdx.x; i < d; i += kNormThreads) {
        const float v = bf16_to_f32(x[base + i]) + bf16_to_f32(y[base + i]);
        out[base + i] = f32_to_bf16(v * inv);
    }
}

}  // namespace

int launch_residual_rmsnorm(int T, int d, const uint16_t* x, const uint16_t* y, float eps, uint16_t* out, cudaStream_t st) {
    if (T == 0) return MOE_OK;
    residual_rmsnorm_kernel<<<T, kNormThreads, 0, st>>>(d, x, y, eps, out);
    note_launch(1);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_LAUNCH;
}

}  // namespace fp4moe
