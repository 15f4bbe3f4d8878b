// Single token, rows streamed from HBM: the layer for one token when its
// expert rows do not fit the fused kernel's shared-memory slots (the
// Qwen3-235B-A22B shape: 85 MB of Q4_K rows per token).
//
// forward_qwen3_moe.rs (aprender-serve 0.35.0), step 2h of
// forward_single_qwen3_moe_with_cache: each of the token's k experts computes
// h_j = SiLU(Wg[e_j] x) * (Wu[e_j] x), its down projection o_j = Wd[e_j] h_j,
// and y = sum_j w_j o_j in slot order.  Two launches after the router:
//   gate/up  persistent CTAs stage x once (padded, with 32-element sums) and
//            take (slot, row) items; a warp loads the whole gate and up row
//            (lane L: sub-block pair L%4 of blocks L/4, L/4+8, ...) before
//            any arithmetic, so every warp keeps ~6 KB of reads in flight;
//   down     persistent CTAs stage the k vectors h_j; a warp takes an output
//            row r, loads row r of four experts' down matrices at a time
//            (fewer for rows longer than 2048) and folds o_j into
//            y[r] = sum_j w_j o_j in slot order, so no o buffer and no
//            separate combine pass exist.
// Weights are read once per call with read-only 16-byte loads; the dot
// products are fp32 (one byte-permute and one FMA per weight).
#include "common.cuh"
#include "kernels.cuh"

namespace moeq4k {
namespace dst {

constexpr int kGuThreads = 256;
constexpr int kGuBlocksPerSm = 2;
constexpr int kDnThreads = 512;
constexpr int kDnPairsInFlight = 4;  // per lane: slots x blocks of down rows loaded together

// Padded shared-memory vector: 4 floats of padding after every 64, so the
// lanes of a warp reading 64-element units 64 floats apart hit distinct banks.
__device__ __forceinline__ int padded(int i) { return i + ((i >> 6) << 2); }
__host__ __device__ inline int padded_len(int n) { return n + (n >> 4); }

// 1 + q/128 as fp32 from byte i of v, where v's bytes are 0x80 | q.
__device__ __forceinline__ float one_plus_q(uint32_t v, int i) {
    return __uint_as_float(__byte_perm(v, 0x3F000000u, 0x7044u | (uint32_t(i) << 8)));
}

__device__ __forceinline__ float u6f(uint32_t v) { return __uint_as_float(0x4B000000u | v) - 8388608.0f; }

// The 48 bytes a lane needs for sub-blocks 2c and 2c+1 of one block: the
// block head and the 32 code bytes qs[32c .. 32c+31].
struct Pair {
    uint4 head, qa, qb;
};

__device__ __forceinline__ Pair load_pair(const uint8_t *blk, int c) {
    Pair p;
    p.head = ldg_nc_v4(blk);
    p.qa = ldg_nc_v4(blk + 16 + 32 * c);
    p.qb = ldg_nc_v4(blk + 32 + 32 * c);
    return p;
}

// sum over sub-blocks 2c, 2c+1 of (d sc q - dmin m) x: `xs` points at the
// block's element 64c of the padded vector, `s2` at its two 32-element sums.
// The codes enter as 1 + q/128, so sum(q x) = 128 (sum((1 + q/128) x) - sum(x)).
__device__ __forceinline__ float pair_dot(const Pair &P, int c, const float *xs, const float *s2) {
    const uint32_t w[8] = {P.qa.x, P.qa.y, P.qa.z, P.qa.w, P.qb.x, P.qb.y, P.qb.z, P.qb.w};
    float a0 = 0.f, a1 = 0.f, b0 = 0.f, b1 = 0.f;
#pragma unroll
    for (int wi = 0; wi < 8; ++wi) {
        const uint32_t lo = (w[wi] & 0x0F0F0F0Fu) | 0x80808080u;
        const uint32_t hi = ((w[wi] >> 4) & 0x0F0F0F0Fu) | 0x80808080u;
        const float4 xl = *reinterpret_cast<const float4 *>(xs + 4 * wi);
        const float4 xh = *reinterpret_cast<const float4 *>(xs + 32 + 4 * wi);
        a0 = fmaf(one_plus_q(lo, 0), xl.x, a0);
        a1 = fmaf(one_plus_q(lo, 1), xl.y, a1);
        a0 = fmaf(one_plus_q(lo, 2), xl.z, a0);
        a1 = fmaf(one_plus_q(lo, 3), xl.w, a1);
        b0 = fmaf(one_plus_q(hi, 0), xh.x, b0);
        b1 = fmaf(one_plus_q(hi, 1), xh.y, b1);
        b0 = fmaf(one_plus_q(hi, 2), xh.z, b0);
        b1 = fmaf(one_plus_q(hi, 3), xh.w, b1);
    }
    // scales and mins of sub-blocks 2c (j0) and 2c+1 (j1)
    const uint4 &h = P.head;
    const int j0 = 2 * c, j1 = 2 * c + 1;
    uint32_t sc0, m0, sc1, m1;
    if (c < 2) {
        sc0 = (h.y >> (8 * j0)) & 63u;
        m0 = (h.z >> (8 * j0)) & 63u;
        sc1 = (h.y >> (8 * j1)) & 63u;
        m1 = (h.z >> (8 * j1)) & 63u;
    } else {
        const int a = j0 - 4, b = j1 - 4;
        sc0 = ((h.w >> (8 * a)) & 15u) | (((h.y >> (8 * a + 6)) & 3u) << 4);
        m0 = ((h.w >> (8 * a + 4)) & 15u) | (((h.z >> (8 * a + 6)) & 3u) << 4);
        sc1 = ((h.w >> (8 * b)) & 15u) | (((h.y >> (8 * b + 6)) & 3u) << 4);
        m1 = ((h.w >> (8 * b + 4)) & 15u) | (((h.z >> (8 * b + 6)) & 3u) << 4);
    }
    const float2 dd = q4k_d_dmin(h);
    const float dm = dd.x * 128.0f;
    const float A0 = dm * u6f(sc0), A1 = dm * u6f(sc1);
    const float B0 = dd.y * u6f(m0), B1 = dd.y * u6f(m1);
    const float slo = s2[0], shi = s2[1];
    float acc = A0 * ((a0 + a1) - slo);
    acc = fmaf(-B0, slo, acc);
    acc = fmaf(A1, (b0 + b1) - shi, acc);
    acc = fmaf(-B1, shi, acc);
    return acc;
}

// Stage n floats of `src` into the padded vector `dst` and their 32-element
// sums into `sum32` (one warp per run, fixed order).  Ends synchronised.
__device__ __forceinline__ void stage_vector(const float *__restrict__ src, int n, float *dst,
                                             float *sum32) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    for (int i = threadIdx.x; i < n / 4; i += blockDim.x)
        *reinterpret_cast<float4 *>(dst + padded(4 * i)) = reinterpret_cast<const float4 *>(src)[i];
    __syncthreads();
    for (int r = warp; r < n / 32; r += nw) {
        const float s = warp_sum(dst[padded(32 * r + lane)]);
        if (lane == 0) sum32[r] = s;
    }
    __syncthreads();
}

// The token's expert ids, -1 for one outside [0, E) (recorded once; the
// slot is skipped).
__device__ __forceinline__ void load_experts(const int32_t *idx, int k, int E, int *eid,
                                             WsHeader *hdr) {
    for (int j = threadIdx.x; j < k; j += blockDim.x) {
        int e = idx[j];
        if (e < 0 || e >= E) {
            if (blockIdx.x == 0) record_status(hdr, MOE_ERR_EXPERT_RANGE, e);
            e = -1;
        }
        eid[j] = e;
    }
}

// h[j*I + r] = SiLU(Wg[e_j][r] . x) * (Wu[e_j][r] . x).  NB = blocks per
// lane (ceil(H / 2048)).
template <int NB>
__global__ void __launch_bounds__(kGuThreads, kGuBlocksPerSm)
    stream_gateup_kernel(const float *__restrict__ x, const uint8_t *__restrict__ gate,
                         const uint8_t *__restrict__ up, const int32_t *__restrict__ idx, int k,
                         int E, int H, int I, float *__restrict__ h, WsHeader *hdr) {
    extern __shared__ __align__(16) float sm[];
    float *xs = sm;
    float *s32 = xs + padded_len(H);
    int *eid = reinterpret_cast<int *>(s32 + H / 32);
    load_experts(idx, k, E, eid, hdr);
    stage_vector(x, H, xs, s32);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    const int nsb = H / kQK;
    const size_t row_bytes = size_t(nsb) * kBlockBytes, mat = size_t(I) * row_bytes;
    const int c = lane & 3, s0 = lane >> 2;
    const int items = k * I;
    for (int it = blockIdx.x * nw + warp; it < items; it += gridDim.x * nw) {
        const int j = it / I, r = it - j * I;
        const int e = eid[j];
        if (e < 0) continue;  // uniform over the warp
        const uint8_t *grow = gate + size_t(e) * mat + size_t(r) * row_bytes;
        const uint8_t *urow = up + size_t(e) * mat + size_t(r) * row_bytes;
        Pair pg[NB], pu[NB];
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            const int s = s0 + 8 * b;
            if (s < nsb) {
                pg[b] = load_pair(grow + size_t(s) * kBlockBytes, c);
                pu[b] = load_pair(urow + size_t(s) * kBlockBytes, c);
            }
        }
        float g = 0.f, u = 0.f;
#pragma unroll
        for (int b = 0; b < NB; ++b) {
            const int s = s0 + 8 * b;
            if (s < nsb) {
                const float *xv = xs + padded(s * kQK + 64 * c);
                const float *sv = s32 + s * 8 + 2 * c;
                g += pair_dot(pg[b], c, xv, sv);
                u += pair_dot(pu[b], c, xv, sv);
            }
        }
        g = warp_sum(g);
        u = warp_sum(u);
        if (lane == 0) h[size_t(j) * I + r] = silu_mul(g, u);
    }
}

// y[r] = sum_j w_j (Wd[e_j][r] . h_j), j = 0..k-1 in order (the same fused
// multiply-adds as the combine of the batched path).  NB = blocks per lane
// (ceil(I / 2048)).
template <int NB>
__global__ void __launch_bounds__(kDnThreads, 1)
    stream_down_kernel(const float *__restrict__ h, const uint8_t *__restrict__ down,
                       const int32_t *__restrict__ idx, const float *__restrict__ w, int k, int E,
                       int H, int I, float *__restrict__ y, WsHeader *hdr) {
    extern __shared__ __align__(16) float sm[];
    const int plen = padded_len(I), runs = I / 32;
    float *hs = sm;                       // [k][plen]
    float *s32 = hs + size_t(k) * plen;   // [k][runs]
    float *wj = s32 + size_t(k) * runs;   // [k]
    int *eid = reinterpret_cast<int *>(wj + k);
    load_experts(idx, k, E, eid, hdr);
    for (int j = threadIdx.x; j < k; j += blockDim.x) wj[j] = w[j];
    for (int j = 0; j < k; ++j) stage_vector(h + size_t(j) * I, I, hs + size_t(j) * plen, s32 + size_t(j) * runs);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    const int nsb = I / kQK;
    const size_t row_bytes = size_t(nsb) * kBlockBytes, mat = size_t(H) * row_bytes;
    const int c = lane & 3, s0 = lane >> 2;
    for (int r = blockIdx.x * nw + warp; r < H; r += gridDim.x * nw) {
        float acc = 0.f;
        constexpr int kSlots = kDnPairsInFlight / NB > 0 ? kDnPairsInFlight / NB : 1;
        for (int j0 = 0; j0 < k; j0 += kSlots) {
            Pair P[kSlots][NB];
#pragma unroll
            for (int jj = 0; jj < kSlots; ++jj) {
                const int j = j0 + jj;
                const int e = j < k ? eid[j] : -1;
                if (e < 0) continue;
                const uint8_t *row = down + size_t(e) * mat + size_t(r) * row_bytes;
#pragma unroll
                for (int b = 0; b < NB; ++b) {
                    const int s = s0 + 8 * b;
                    if (s < nsb) P[jj][b] = load_pair(row + size_t(s) * kBlockBytes, c);
                }
            }
#pragma unroll
            for (int jj = 0; jj < kSlots; ++jj) {
                const int j = j0 + jj;
                const int e = j < k ? eid[j] : -1;
                if (e < 0) continue;  // uniform over the warp
                float part = 0.f;
#pragma unroll
                for (int b = 0; b < NB; ++b) {
                    const int s = s0 + 8 * b;
                    if (s < nsb)
                        part += pair_dot(P[jj][b], c, hs + size_t(j) * plen + padded(s * kQK + 64 * c),
                                         s32 + size_t(j) * runs + s * 8 + 2 * c);
                }
                acc = fmaf(wj[j], warp_sum(part), acc);
            }
        }
        if (lane == 0) y[r] = acc;
    }
}

size_t gateup_smem(int H, int k) { return sizeof(float) * (padded_len(H) + H / 32) + sizeof(int) * k; }
size_t down_smem(int I, int k) {
    return sizeof(float) * size_t(k) * (padded_len(I) + I / 32 + 1) + sizeof(int) * k;
}

}  // namespace dst

namespace {
int g_stream_smem_optin[64];
}

cudaError_t init_decode_stream(int dev) {
    using namespace dst;
    int optin = 0;
    cudaError_t err = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (err != cudaSuccess) return err;
    g_stream_smem_optin[dev] = optin;
    const void *fns[] = {reinterpret_cast<const void *>(stream_down_kernel<1>),
                         reinterpret_cast<const void *>(stream_down_kernel<2>),
                         reinterpret_cast<const void *>(stream_down_kernel<4>)};
    for (const void *f : fns) {
        err = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
        if (err != cudaSuccess) return err;
    }
    return cudaSuccess;
}

bool decode_stream_supported(int dev, int T, int H, int E, int k, int I) {
    using namespace dst;
    if (T != 1 || H % kQK != 0 || I % kQK != 0 || H > 8192 || I > 8192) return false;
    const size_t optin = size_t(g_stream_smem_optin[dev]);
    return gateup_smem(H, k) <= 48 * 1024 && down_smem(I, k) <= optin;
}

cudaError_t launch_decode_stream(const float *x, const int32_t *idx, const float *w,
                                 const uint8_t *gate, const uint8_t *up, const uint8_t *down,
                                 int H, int E, int k, int I, float *y, float *hbuf, WsHeader *hdr,
                                 int num_sms, cudaStream_t s) {
    using namespace dst;
    const int nbh = (H / kQK + 7) / 8, nbi = (I / kQK + 7) / 8;
    const size_t sg = gateup_smem(H, k), sd = down_smem(I, k);
    const int gg = num_sms * kGuBlocksPerSm;
    if (nbh <= 1)
        stream_gateup_kernel<1><<<gg, kGuThreads, sg, s>>>(x, gate, up, idx, k, E, H, I, hbuf, hdr);
    else if (nbh <= 2)
        stream_gateup_kernel<2><<<gg, kGuThreads, sg, s>>>(x, gate, up, idx, k, E, H, I, hbuf, hdr);
    else
        stream_gateup_kernel<4><<<gg, kGuThreads, sg, s>>>(x, gate, up, idx, k, E, H, I, hbuf, hdr);
    if (nbi <= 1)
        stream_down_kernel<1><<<num_sms, kDnThreads, sd, s>>>(hbuf, down, idx, w, k, E, H, I, y, hdr);
    else if (nbi <= 2)
        stream_down_kernel<2><<<num_sms, kDnThreads, sd, s>>>(hbuf, down, idx, w, k, E, H, I, y, hdr);
    else
        stream_down_kernel<4><<<num_sms, kDnThreads, sd, s>>>(hbuf, down, idx, w, k, E, H, I, y, hdr);
    return cudaGetLastError();
}

}  // namespace moeq4k
