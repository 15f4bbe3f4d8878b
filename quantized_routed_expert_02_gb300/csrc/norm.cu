// Pre-FFN RMSNorm of each token row, for the multi-launch paths (the
// single-token fused kernel applies it inside its own x staging).
//
// forward_qwen3_moe.rs (aprender-serve 0.35.0), step 2f of forward_qwen3_moe
// and step 2g of forward_single_qwen3_moe_with_cache: the MoE FFN consumes
// ffn_input = rms_norm(hidden, ffn_norm_weight, eps), read as
//     xn[i] = x[i] / sqrt(mean(x^2) + eps) * gamma[i]  (fp32 in, fp32 out).
#include "common.cuh"
#include "kernels.cuh"

namespace moeq4k {

namespace {
constexpr int kNormThreads = 256;
}

// One CTA per token row: strided float4 partial sums of squares, a fixed
// warp-shuffle tree, then the eight warp sums in order; every element is
// scaled as (x * gamma) * inv.
__global__ void __launch_bounds__(kNormThreads) rmsnorm_kernel(const float *__restrict__ x,
                                                               const float *__restrict__ gamma,
                                                               float eps, int H,
                                                               float *__restrict__ xn) {
    pdl_enter();
    __shared__ float part[kNormThreads / 32];
    __shared__ float inv_sh;
    const int t = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float4 *xr = reinterpret_cast<const float4 *>(x + size_t(t) * H);
    float ss = 0.f;
    for (int i = threadIdx.x; i < H / 4; i += kNormThreads) {
        const float4 v = __ldg(xr + i);
        ss = fmaf(v.x, v.x, ss);
        ss = fmaf(v.y, v.y, ss);
        ss = fmaf(v.z, v.z, ss);
        ss = fmaf(v.w, v.w, ss);
    }
    ss = warp_sum(ss);
    if (lane == 0) part[warp] = ss;
    __syncthreads();
    if (threadIdx.x == 0) {
        float s = 0.f;
        for (int w = 0; w < kNormThreads / 32; ++w) s += part[w];
        inv_sh = 1.0f / sqrtf(s / float(H) + eps);
    }
    __syncthreads();
    const float inv = inv_sh;
    const float4 *g4 = reinterpret_cast<const float4 *>(gamma);
    float4 *out = reinterpret_cast<float4 *>(xn + size_t(t) * H);
    for (int i = threadIdx.x; i < H / 4; i += kNormThreads) {
        const float4 v = __ldg(xr + i), g = __ldg(g4 + i);
        out[i] = make_float4(v.x * g.x * inv, v.y * g.y * inv, v.z * g.z * inv, v.w * g.w * inv);
    }
}

cudaError_t launch_rmsnorm(const float *x, const float *gamma, float eps, int T, int H, float *xn,
                           cudaStream_t s) {
    launch_pdl(rmsnorm_kernel, dim3(T), dim3(kNormThreads), size_t(0), s, x, gamma, eps, H, xn);
    return cudaGetLastError();
}

}  // namespace moeq4k
