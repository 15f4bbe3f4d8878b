// Router: fp32 logits, softmax over all experts, top-k, renormalisation.
//
// forward_qwen3_moe_cuda_traced.rs (aprender-serve 0.34.0), doc of
// forward_qwen3_moe_cuda_traced_with_plan: the router stage is the k
// post-softmax, renormalised top-k weights of a token.  Softmax is monotone,
// so the top-k of p is the top-k of the logits; after renormalisation the
// full-softmax denominator cancels and w_j = exp(l_j - l_max) / sum over the
// selected slots of exp(l - l_max).
#include "async_copy.cuh"
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
    pdl_enter();
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
// 3..255 tokens: a CTA stages kXT tokens of x in shared memory (coalesced),
// then each warp takes one expert row of Wr, requests its share of the row
// in batches of four float4 per lane before any arithmetic, and dots it with
// the staged tokens (fixed per-lane order, then a warp sum).
// ---------------------------------------------------------------------------
constexpr int kXT = 8;  // tokens per CTA
constexpr int kRouterTileSmemMax = 128 * 1024;  // x tile of up to H = 4096

__global__ void __launch_bounds__(256) router_tile_kernel(const float *__restrict__ x,
                                                          const float *__restrict__ Wr,
                                                          const float *__restrict__ bias, int T,
                                                          int H, int E, float *__restrict__ logits) {
    pdl_enter();
    extern __shared__ __align__(16) float xt[];  // [kXT][H]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t0 = blockIdx.y * kXT, n4 = H >> 2;
    for (int i = threadIdx.x; i < kXT * n4; i += blockDim.x) {
        const int tok = i / n4, c = i - tok * n4;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (t0 + tok < T) v = __ldg(reinterpret_cast<const float4 *>(x + size_t(t0 + tok) * H) + c);
        reinterpret_cast<float4 *>(xt)[i] = v;
    }
    __syncthreads();
    const int e = blockIdx.x * 8 + warp;
    if (e >= E) return;
    const float4 *wr = reinterpret_cast<const float4 *>(Wr + size_t(e) * H);
    const float4 *x4 = reinterpret_cast<const float4 *>(xt);
    float acc[kXT];
#pragma unroll
    for (int t = 0; t < kXT; ++t) acc[t] = 0.f;
    for (int c0 = lane; c0 < n4; c0 += 4 * 32) {
        float4 a[4];
#pragma unroll
        for (int b = 0; b < 4; ++b)
            if (c0 + 32 * b < n4) a[b] = __ldg(wr + c0 + 32 * b);
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const int c = c0 + 32 * b;
            if (c >= n4) break;
#pragma unroll
            for (int t = 0; t < kXT; ++t) {
                const float4 v = x4[t * n4 + c];
                acc[t] = fmaf(a[b].x, v.x, acc[t]);
                acc[t] = fmaf(a[b].y, v.y, acc[t]);
                acc[t] = fmaf(a[b].z, v.z, acc[t]);
                acc[t] = fmaf(a[b].w, v.w, acc[t]);
            }
        }
    }
    const float b = bias ? bias[e] : 0.f;
#pragma unroll
    for (int t = 0; t < kXT; ++t) {
        const float sum = warp_sum(acc[t]);
        if (lane == 0 && t0 + t < T) logits[size_t(t0 + t) * E + e] = sum + b;
    }
}

// ---------------------------------------------------------------------------
// Top-k + renormalise: one warp per token.  Lane L holds logits of experts
// L, L+32, ...; k rounds of a warp-wide arg-max with the order (value
// descending, index ascending).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) router_topk_kernel(const float *__restrict__ logits,
                                                          int T, int E, int k,
                                                          int32_t *__restrict__ idx,
                                                          float *__restrict__ w) {
    pdl_enter();
    const int warp = threadIdx.x >> 5;
    const int t = blockIdx.x * 8 + warp;
    if (t >= T) return;
    warp_topk(logits + size_t(t) * E, E, k, idx + size_t(t) * k, w + size_t(t) * k);
}

// ---------------------------------------------------------------------------
// One or two tokens: one CTA per expert row, each thread a strided share of
// the row (float4 steps), reduced in a fixed order (warp shuffles, then the
// eight warp sums in order), so every row of Wr is read by 256 threads at
// once.  The last CTA to store its logits ranks them (top-k + renormalise):
// one launch for the whole router.
// ---------------------------------------------------------------------------
template <int kTT>
__global__ void __launch_bounds__(256) router_row_kernel(const float *__restrict__ x,
                                                         const float *__restrict__ Wr,
                                                         const float *__restrict__ bias, int T,
                                                         int H, int E, int k,
                                                         float *__restrict__ logits,
                                                         int32_t *__restrict__ idx,
                                                         float *__restrict__ w, WsHeader *hdr) {
    pdl_enter();
    __shared__ float part[kTT][8];
    __shared__ float lg[kTT][kMaxE];
    __shared__ int last;
    const int e = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float4 *wr = reinterpret_cast<const float4 *>(Wr + size_t(e) * H);
    float acc[kTT];
#pragma unroll
    for (int i = 0; i < kTT; ++i) acc[i] = 0.f;
    for (int c = threadIdx.x; c < H / 4; c += blockDim.x) {
        const float4 a = __ldg(wr + c);
#pragma unroll
        for (int i = 0; i < kTT; ++i) {
            if (i < T) {
                const float4 b = __ldg(reinterpret_cast<const float4 *>(x + size_t(i) * H) + c);
                acc[i] = fmaf(a.x, b.x, acc[i]);
                acc[i] = fmaf(a.y, b.y, acc[i]);
                acc[i] = fmaf(a.z, b.z, acc[i]);
                acc[i] = fmaf(a.w, b.w, acc[i]);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < kTT; ++i) {
        const float s = warp_sum(acc[i]);
        if (lane == 0) part[i][warp] = s;
    }
    __syncthreads();
    if (threadIdx.x < kTT && int(threadIdx.x) < T) {
        const int i = threadIdx.x;
        float s = 0.f;
        for (int ww = 0; ww < 8; ++ww) s += part[i][ww];
        logits[size_t(i) * E + e] = s + (bias ? bias[e] : 0.f);
        __threadfence();  // the logit is visible GPU-wide before this CTA is counted
    }
    __syncthreads();
    // The count starts every call at 0 (moe_workspace_init, then the ranking
    // CTA of each call sets it back), so exactly the last CTA to count itself
    // sees gridDim.x - 1 and every other logit is stored by then.  A count at
    // or past gridDim.x means the header was never initialised (or was
    // overwritten): that is recorded, and no CTA ranks logits it cannot
    // trust; the count stays off until the workspace is re-initialised.
    if (threadIdx.x == 0) {
        const unsigned long long prev = atomicAdd(&hdr->router_rows, 1ull);
        last = prev == gridDim.x - 1;
        if (prev >= gridDim.x)
            record_status(hdr, MOE_ERR_INTERNAL, 500000000 + int(prev % 1000000ull));
    }
    __syncthreads();
    if (!last) return;
    __threadfence();
    for (int i = threadIdx.x; i < T * E; i += blockDim.x) lg[i / E][i % E] = __ldcg(logits + i);
    __syncthreads();
    if (warp < T) warp_topk(&lg[warp][0], E, k, idx + size_t(warp) * k, w + size_t(warp) * k);
    if (threadIdx.x == 0) atomicExch(&hdr->router_rows, 0ull);  // every CTA has counted itself
}

// ---------------------------------------------------------------------------
// Large batches: logits of 32 tokens x all E experts per CTA as a shared-
// memory-tiled fp32 GEMM (each thread a 4 x 4 register tile, K in chunks of
// 32, double-buffered), then the top-k of each token by one warp from the
// CTA's logits in shared memory.
// ---------------------------------------------------------------------------
constexpr int kRT = 32;   // tokens per CTA
constexpr int kRE = 128;  // experts per pass
constexpr int kRK = 32;   // K per chunk
constexpr int kRouterBigSmem = int(sizeof(float)) * (2 * kRK * kRT + 2 * kRK * kRE + kRT * (kMaxE + 1));

__global__ void __launch_bounds__(256) router_big_kernel(const float *__restrict__ x,
                                                         const float *__restrict__ Wr,
                                                         const float *__restrict__ bias, int T,
                                                         int H, int E, int k,
                                                         int32_t *__restrict__ idx,
                                                         float *__restrict__ w) {
    pdl_enter();
    // dynamic shared memory: xs[2][kRK][kRT], ws[2][kRK][kRE] (k-major), lg[kRT][kMaxE + 1]
    extern __shared__ __align__(16) float rsm[];
    float (*xs)[kRK][kRT] = reinterpret_cast<float (*)[kRK][kRT]>(rsm);
    float (*ws)[kRK][kRE] = reinterpret_cast<float (*)[kRK][kRE]>(rsm + 2 * kRK * kRT);
    float (*lg)[kMaxE + 1] = reinterpret_cast<float (*)[kMaxE + 1]>(rsm + 2 * kRK * kRT + 2 * kRK * kRE);
    const int tid = threadIdx.x, ty = tid >> 5, tx = tid & 31;
    const int t0 = blockIdx.x * kRT;
    const int nchunk = H / kRK;
    for (int e0 = 0; e0 < E; e0 += kRE) {
        float acc[4][4] = {};
        auto load = [&](int c, int buf) {
            // x: 32 tokens x 32 k = 256 float4, one per thread
            {
                const int t = tid >> 3, q = tid & 7;
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (t0 + t < T) v = __ldg(reinterpret_cast<const float4 *>(x + size_t(t0 + t) * H + c * kRK) + q);
                xs[buf][4 * q + 0][t] = v.x;
                xs[buf][4 * q + 1][t] = v.y;
                xs[buf][4 * q + 2][t] = v.z;
                xs[buf][4 * q + 3][t] = v.w;
            }
            // Wr: 128 experts x 32 k = 1024 float4, four per thread
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int f = tid + 256 * r, e = f >> 3, q = f & 7;
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (e0 + e < E) v = __ldg(reinterpret_cast<const float4 *>(Wr + size_t(e0 + e) * H + c * kRK) + q);
                ws[buf][4 * q + 0][e] = v.x;
                ws[buf][4 * q + 1][e] = v.y;
                ws[buf][4 * q + 2][e] = v.z;
                ws[buf][4 * q + 3][e] = v.w;
            }
        };
        load(0, 0);
        __syncthreads();
        for (int c = 0; c < nchunk; ++c) {
            const int buf = c & 1;
            if (c + 1 < nchunk) load(c + 1, buf ^ 1);
            // two-level sum: a fresh partial per 32-wide chunk keeps the fp32
            // rounding of the 2048-term dot products small
            float part[4][4] = {};
#pragma unroll 8
            for (int kk = 0; kk < kRK; ++kk) {
                const float4 a = *reinterpret_cast<const float4 *>(&xs[buf][kk][ty * 4]);
                const float4 b = *reinterpret_cast<const float4 *>(&ws[buf][kk][tx * 4]);
                const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) part[i][j] = fmaf(av[i], bv[j], part[i][j]);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] += part[i][j];
            __syncthreads();
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int e = e0 + tx * 4 + j;
                if (e < E) lg[ty * 4 + i][e] = acc[i][j] + (bias ? bias[e] : 0.f);
            }
        __syncthreads();
    }
    // top-k: warp ty takes tokens ty, ty+8, ty+16, ty+24
    for (int i = ty; i < kRT; i += 8) {
        const int t = t0 + i;
        if (t < T) warp_topk(&lg[i][0], E, k, idx + size_t(t) * k, w + size_t(t) * k);
    }
}

cudaError_t init_router() {
    cudaError_t err = cudaFuncSetAttribute(router_big_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           kRouterBigSmem);
    if (err != cudaSuccess) return err;
    err = cudaFuncSetAttribute(router_tile_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kRouterTileSmemMax);
    if (err != cudaSuccess) return err;
    return cudaSuccess;
}

cudaError_t launch_router(const float *x, const float *Wr, const float *bias, int T, int H, int E,
                          int k, int32_t *idx, float *w, float *logits, WsHeader *hdr,
                          cudaStream_t s) {
    dim3 blk(256);
    // T >= 256, E <= 128: tensor cores (three-pass TF32, router_tc.cu)
    if (router_tc_supported(T, H, E))
        return launch_router_tc(x, Wr, bias, T, H, E, k, idx, w, hdr, 1000000000ull, s);
    if (T >= 256) {
        launch_pdl(router_big_kernel, dim3((T + kRT - 1) / kRT), dim3(blk), size_t(kRouterBigSmem), s, x, Wr, bias, T, H, E, k, idx, w);
        return cudaGetLastError();
    }
    if (T <= 2) {
        launch_pdl(router_row_kernel<2>, dim3(E), dim3(blk), size_t(0), s, x, Wr, bias, T, H, E, k, logits, idx, w, hdr);
        return cudaGetLastError();
    }
    if (size_t(kXT) * H * sizeof(float) <= size_t(kRouterTileSmemMax)) {
        dim3 grid((E + 7) / 8, (T + kXT - 1) / kXT);
        launch_pdl(router_tile_kernel, dim3(grid), dim3(blk), size_t(size_t(kXT) * H * sizeof(float)), s, x, Wr, bias, T, H, E, logits);
    } else {
        dim3 grid((E + 7) / 8, (T + 7) / 8);
        launch_pdl(router_logits_kernel<8>, dim3(grid), dim3(blk), size_t(0), s, x, Wr, bias, T, H, E, logits);
    }
    launch_pdl(router_topk_kernel, dim3((T + 7) / 8), dim3(blk), size_t(0), s, logits, T, E, k, idx, w);
    return cudaGetLastError();
}

}  // namespace moeq4k
