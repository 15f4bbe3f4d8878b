// Router: fp32 logits, softmax over all experts, top-k, renormalisation.
//
// forward_qwen3_moe_cuda_traced.rs (aprender-serve 0.34.0), doc of
// forward_qwen3_moe_cuda_traced_with_plan: the router stage is the k
// post-softmax, renormalised top-k weights of a token.  Softmax is monotone,
// so the top-k of p is the top-k of the logits; after renormalisation the
// full-softmax denominator cancels and w_j = exp(l_j - l_max) / sum over the
// selected slots of exp(l - l_max).
#include "common.cuh"
#include "kernels.cuh"

namespace moeq4k {

// ---------------------------------------------------------------------------
// Logits: one warp per expert row of Wr, a tile of kTT tokens per CTA.  Each
// lane walks the row in float4 steps, so a warp reads 512 contiguous bytes
// of Wr and of every x row per step.
// ---------------------------------------------------------------------------
template <int kTT>
__global__ void __launch_bounds__(256) router_logits_kernel(const float *__restrict__ x,
                                                            const float *__restrict__ Wr,
                                                            const float *__restrict__ bias,
                                                            int T, int H, int E,
                                                            float *__restrict__ logits) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = blockIdx.x * 8 + warp;
    const int t0 = blockIdx.y * kTT;
    if (e >= E) return;
    const float4 *wr = reinterpret_cast<const float4 *>(Wr + size_t(e) * H);
    float acc[kTT];
#pragma unroll
    for (int i = 0; i < kTT; ++i) acc[i] = 0.f;
    const int n4 = H >> 2;
    for (int c = lane; c < n4; c += 32) {
        float4 a = __ldg(wr + c);
#pragma unroll
        for (int i = 0; i < kTT; ++i) {
            if (t0 + i < T) {
                float4 b = __ldg(reinterpret_cast<const float4 *>(x + size_t(t0 + i) * H) + c);
                acc[i] = fmaf(a.x, b.x, acc[i]);
                acc[i] = fmaf(a.y, b.y, acc[i]);
                acc[i] = fmaf(a.z, b.z, acc[i]);
                acc[i] = fmaf(a.w, b.w, acc[i]);
            }
        }
    }
    const float b = bias ? bias[e] : 0.f;
#pragma unroll
    for (int i = 0; i < kTT; ++i) {
        float s = warp_sum(acc[i]);
        if (lane == 0 && t0 + i < T) logits[size_t(t0 + i) * E + e] = s + b;
    }
}

// ---------------------------------------------------------------------------
// Top-k + renormalise: one warp per token.  Lane L holds logits of experts
// L, L+32, ...; k rounds of a warp-wide arg-max with the order (value
// descending, index ascending).
// ---------------------------------------------------------------------------
__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
    return v > bv || (v == bv && i < bi);
}

__global__ void __launch_bounds__(256) router_topk_kernel(const float *__restrict__ logits,
                                                          int T, int E, int k,
                                                          int32_t *__restrict__ idx,
                                                          float *__restrict__ w) {
    constexpr int kPer = kMaxE / 32;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * 8 + warp;
    if (t >= T) return;
    float v[kPer];
    bool taken[kPer];
#pragma unroll
    for (int s = 0; s < kPer; ++s) {
        int e = lane + 32 * s;
        v[s] = (e < E) ? logits[size_t(t) * E + e] : -INFINITY;
        taken[s] = (e >= E);
    }
    float sel_v = 0.f;   // lane j keeps slot j's logit
    int sel_i = 0;
    float vmax = 0.f;
    for (int j = 0; j < k; ++j) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
#pragma unroll
        for (int s = 0; s < kPer; ++s) {
            int e = lane + 32 * s;
            if (!taken[s] && better(v[s], e, bv, bi)) {
                bv = v[s];
                bi = e;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (better(ov, oi, bv, bi)) {
                bv = ov;
                bi = oi;
            }
        }
#pragma unroll
        for (int s = 0; s < kPer; ++s)
            if (bi == lane + 32 * s) taken[s] = true;
        if (j == 0) vmax = bv;
        if (lane == j) {
            sel_v = bv;
            sel_i = bi;
        }
    }
    float ex = (lane < k) ? expf(sel_v - vmax) : 0.f;
    float z = warp_sum(ex);
    if (lane < k) {
        idx[size_t(t) * k + lane] = sel_i;
        w[size_t(t) * k + lane] = ex / z;
    }
}

cudaError_t launch_router(const float *x, const float *Wr, const float *bias, int T, int H, int E,
                          int k, int32_t *idx, float *w, float *logits, cudaStream_t s) {
    dim3 blk(256);
    if (T <= 2) {
        dim3 grid((E + 7) / 8, (T + 1) / 2);
        router_logits_kernel<2><<<grid, blk, 0, s>>>(x, Wr, bias, T, H, E, logits);
    } else {
        dim3 grid((E + 7) / 8, (T + 7) / 8);
        router_logits_kernel<8><<<grid, blk, 0, s>>>(x, Wr, bias, T, H, E, logits);
    }
    router_topk_kernel<<<(T + 7) / 8, blk, 0, s>>>(logits, T, E, k, idx, w);
    return cudaGetLastError();
}

}  // namespace moeq4k
