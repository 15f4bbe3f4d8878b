// The expert FFN with Q8_K activations: every activation vector that meets
// a Q4_K matrix (x before gate/up, h before down) is first quantised per
// block of 256 values to signed 8-bit codes with one fp32 scale, and the
// products are integer dot products.
//
// qwen3_moe_dispatch.rs (aprender-serve 0.70.2), doc of cpu_reference: the
// production CPU path runs the layer on Q8_K activations; the fp32-activation
// path is the other scope of the same forward.  The page names the format
// only; the arithmetic taken here (one scale d = amax / 127 per 256 values,
// codes rounded half to even from v * (127 / amax), fp32 throughout) is the
// plainest reading of it, and every step is fp32 so the codes are decided
// exactly as the host-side statement of the format decides them.
//
// Launches (all with programmatic dependent launch):
//   q8k_quantize_kernel  x [T, H] -> codes, block scales, sub-block code sums
//   q8k_gateup_kernel    warp per (slot, row): g, u integer dots, h = SiLU(g) u
//   q8k_quantize_kernel  h [T*k, I] -> codes, scales, sums
//   q8k_down_kernel      warp per (token, row): y = sum_j w_j (Wd[e_j] . h_j)
// A Q4_K sub-block pair (64 weights: 32 code bytes, low nibbles = sub-block
// 2c, high = 2c+1) against 64 codes is 16 dp4a; the block scales are applied
// in fp32 per sub-block: d8 (d4 sc P - dmin m S), P the integer dot, S the
// sub-block's code sum.
#include <algorithm>

#include "common.cuh"
#include "kernels.cuh"

namespace moeq4k {
namespace q8 {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

// One warp per 256-value block: lane L holds values 8L..8L+7.
__global__ void __launch_bounds__(kThreads) q8k_quantize_kernel(const float *__restrict__ v,
                                                                long nblocks,
                                                                int8_t *__restrict__ q,
                                                                float *__restrict__ d,
                                                                int32_t *__restrict__ sums) {
    pdl_enter();
    const int lane = threadIdx.x & 31;
    const long nwarps = long(gridDim.x) * kWarps;
    for (long b = long(blockIdx.x) * kWarps + (threadIdx.x >> 5); b < nblocks; b += nwarps) {
        const float4 *src = reinterpret_cast<const float4 *>(v + b * kQK) + 2 * lane;
        const float4 a = src[0], c = src[1];
        const float vals[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(vals[i]));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        int codes[8];
        if (amax == 0.f) {
#pragma unroll
            for (int i = 0; i < 8; ++i) codes[i] = 0;
            if (lane == 0) d[b] = 0.f;
        } else {
            // the scale and each product rounded once to fp32 (no contraction)
            const float s = __fdiv_rn(127.f, amax);
            if (lane == 0) d[b] = __fdiv_rn(amax, 127.f);
#pragma unroll
            for (int i = 0; i < 8; ++i) codes[i] = __float2int_rn(__fmul_rn(vals[i], s));
        }
        uint2 packed;
        packed.x = (uint32_t(codes[0]) & 255u) | (uint32_t(codes[1]) & 255u) << 8 |
                   (uint32_t(codes[2]) & 255u) << 16 | (uint32_t(codes[3]) & 255u) << 24;
        packed.y = (uint32_t(codes[4]) & 255u) | (uint32_t(codes[5]) & 255u) << 8 |
                   (uint32_t(codes[6]) & 255u) << 16 | (uint32_t(codes[7]) & 255u) << 24;
        reinterpret_cast<uint2 *>(q + b * kQK)[lane] = packed;
        // sub-block j (32 values) = lanes 4j..4j+3
        int sum = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) sum += codes[i];
        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
        sum += __shfl_xor_sync(0xffffffffu, sum, 2);
        if ((lane & 3) == 0) sums[b * (kQK / 32) + (lane >> 2)] = sum;
    }
}

// d8 * (d4 sc P - dmin m S) for one sub-block pair of one Q4_K row: the 32
// code bytes `cw` (8 words), the block head, sub-block pair c (0..3) of the
// block, the vector's 64 codes `xw` (16 words: 8 for sub-block 2c, then 8
// for 2c+1), its two sub-block sums and its block scale.
__device__ __forceinline__ float pair_dot_q8k(const uint4 &head, int c, const uint32_t cw[8],
                                              const uint32_t xw[16], int s_lo, int s_hi,
                                              float d8) {
    int p_lo = 0, p_hi = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        p_lo = __dp4a(int(cw[i] & 0x0F0F0F0Fu), int(xw[i]), p_lo);
        p_hi = __dp4a(int((cw[i] >> 4) & 0x0F0F0F0Fu), int(xw[8 + i]), p_hi);
    }
    float sc0, m0, sc1, m1;
    q4k_scale_min(head, 2 * c, sc0, m0);
    q4k_scale_min(head, 2 * c + 1, sc1, m1);
    const float2 dd = q4k_d_dmin(head);
    const float lo = dd.x * sc0 * float(p_lo) - dd.y * m0 * float(s_lo);
    const float hi = dd.x * sc1 * float(p_hi) - dd.y * m1 * float(s_hi);
    return d8 * (lo + hi);
}

__device__ __forceinline__ void load_codes(const uint8_t *p, uint32_t w[8]) {
    const uint4 a = ldg_nc_v4(p), b = ldg_nc_v4(p + 16);
    w[0] = a.x, w[1] = a.y, w[2] = a.z, w[3] = a.w, w[4] = b.x, w[5] = b.y, w[6] = b.z, w[7] = b.w;
}

__device__ __forceinline__ void load_vec(const int8_t *p, uint32_t w[16]) {
    const uint4 *s = reinterpret_cast<const uint4 *>(p);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint4 v = __ldg(s + i);
        w[4 * i] = v.x, w[4 * i + 1] = v.y, w[4 * i + 2] = v.z, w[4 * i + 3] = v.w;
    }
}

// h[p, r] = SiLU(g) u for slot p (token p / k, expert idx[p]) and row r, one
// warp per (p, r); lanes over the H / 64 sub-block pairs of the gate and up
// rows.  A slot with an expert index outside [0, E) gets h = 0 (and the
// status records it).
__global__ void __launch_bounds__(kThreads) q8k_gateup_kernel(
    const int8_t *__restrict__ xq, const float *__restrict__ xd, const int32_t *__restrict__ xs,
    const int32_t *__restrict__ idx, const uint8_t *__restrict__ gate,
    const uint8_t *__restrict__ up, int T, int H, int E, int k, int I, float *__restrict__ h,
    WsHeader *hdr) {
    pdl_enter();
    const int lane = threadIdx.x & 31;
    const int npairs = H / 64, nsb = H / kQK;
    const size_t row_bytes = size_t(nsb) * kBlockBytes, mat = size_t(I) * row_bytes;
    const long items = long(T) * k * I;
    const long nwarps = long(gridDim.x) * kWarps;
    for (long it = long(blockIdx.x) * kWarps + (threadIdx.x >> 5); it < items; it += nwarps) {
        const long p = it / I;
        const int r = int(it - p * I);
        const int t = int(p / k);
        const int e = idx[p];
        if (e < 0 || e >= E) {
            if (lane == 0) {
                h[p * I + r] = 0.f;
                if (r == 0) record_status(hdr, MOE_ERR_EXPERT_RANGE, e);
            }
            continue;
        }
        const uint8_t *grow = gate + size_t(e) * mat + size_t(r) * row_bytes;
        const uint8_t *urow = up + size_t(e) * mat + size_t(r) * row_bytes;
        const int8_t *xv = xq + size_t(t) * H;
        float g = 0.f, u = 0.f;
        for (int pc = lane; pc < npairs; pc += 32) {
            const int b = pc >> 2, c = pc & 3;
            const size_t boff = size_t(b) * kBlockBytes;
            const uint4 gh = ldg_nc_v4(grow + boff), uh = ldg_nc_v4(urow + boff);
            uint32_t gw[8], uw[8], xw[16];
            load_codes(grow + boff + 16 + 32 * c, gw);
            load_codes(urow + boff + 16 + 32 * c, uw);
            load_vec(xv + 64 * pc, xw);
            const int sb = t * (H / 32) + 2 * pc;
            const int s_lo = __ldg(xs + sb), s_hi = __ldg(xs + sb + 1);
            const float d8 = __ldg(xd + size_t(t) * nsb + b);
            g += pair_dot_q8k(gh, c, gw, xw, s_lo, s_hi, d8);
            u += pair_dot_q8k(uh, c, uw, xw, s_lo, s_hi, d8);
        }
        g = warp_sum(g);
        u = warp_sum(u);
        if (lane == 0) h[p * I + r] = silu_mul(g, u);
    }
}

// y[t, r] = sum over the k slots of w_j (Wd[e_j] row r . h_j), one warp per
// (t, r); lanes over the k * I / 64 units (slot j, sub-block pair c), each
// unit's dot weighted by w_j, then one fixed-order warp sum.
__global__ void __launch_bounds__(kThreads) q8k_down_kernel(
    const int8_t *__restrict__ hq, const float *__restrict__ hd, const int32_t *__restrict__ hs,
    const int32_t *__restrict__ idx, const float *__restrict__ w, const uint8_t *__restrict__ down,
    int T, int H, int E, int k, int I, float *__restrict__ y) {
    pdl_enter();
    const int lane = threadIdx.x & 31;
    const int npairs = I / 64, nsb = I / kQK;
    const size_t row_bytes = size_t(nsb) * kBlockBytes, mat = size_t(H) * row_bytes;
    const long items = long(T) * H;
    const int units = k * npairs;
    const long nwarps = long(gridDim.x) * kWarps;
    for (long it = long(blockIdx.x) * kWarps + (threadIdx.x >> 5); it < items; it += nwarps) {
        const int t = int(it / H);
        const int r = int(it - long(t) * H);
        float acc = 0.f;
        for (int un = lane; un < units; un += 32) {
            const int j = un / npairs, pc = un - j * npairs;
            const long p = long(t) * k + j;
            const int e = idx[p];
            if (e < 0 || e >= E) continue;  // recorded by the gate/up launch
            const int b = pc >> 2, c = pc & 3;
            const uint8_t *drow = down + size_t(e) * mat + size_t(r) * row_bytes + size_t(b) * kBlockBytes;
            const uint4 head = ldg_nc_v4(drow);
            uint32_t cw[8], xw[16];
            load_codes(drow + 16 + 32 * c, cw);
            load_vec(hq + size_t(p) * I + 64 * pc, xw);
            const int sb = int(p * (I / 32)) + 2 * pc;
            acc += __ldg(w + p) *
                   pair_dot_q8k(head, c, cw, xw, __ldg(hs + sb), __ldg(hs + sb + 1),
                                __ldg(hd + size_t(p) * nsb + b));
        }
        acc = warp_sum(acc);
        if (lane == 0) y[it] = acc;
    }
}

}  // namespace q8

cudaError_t launch_q8k_quantize(const float *v, long rows, int n, int8_t *q, float *d,
                                int32_t *sums, int num_sms, cudaStream_t s) {
    const long nblocks = rows * (n / kQK);
    const long grid = std::min<long>((nblocks + q8::kWarps - 1) / q8::kWarps, long(num_sms) * 16);
    launch_pdl(q8::q8k_quantize_kernel, dim3(unsigned(std::max<long>(grid, 1))),
               dim3(q8::kThreads), size_t(0), s, v, nblocks, q, d, sums);
    return cudaGetLastError();
}

cudaError_t launch_q8k_ffn(const float *x, const int32_t *idx, const float *w, const uint8_t *gate,
                           const uint8_t *up, const uint8_t *down, int T, int H, int E, int k,
                           int I, float *y, int8_t *xq, float *xd, int32_t *xs, float *hbuf,
                           int8_t *hq, float *hd, int32_t *hs, WsHeader *hdr, int num_sms,
                           cudaStream_t s) {
    const long pairs = long(T) * k;
    cudaError_t err = launch_q8k_quantize(x, T, H, xq, xd, xs, num_sms, s);
    if (err != cudaSuccess) return err;
    const long gu_items = pairs * I;
    const long gu_grid = std::min<long>((gu_items + q8::kWarps - 1) / q8::kWarps, long(num_sms) * 64);
    launch_pdl(q8::q8k_gateup_kernel, dim3(unsigned(gu_grid)), dim3(q8::kThreads), size_t(0), s,
               xq, xd, xs, idx, gate, up, T, H, E, k, I, hbuf, hdr);
    err = launch_q8k_quantize(hbuf, pairs, I, hq, hd, hs, num_sms, s);
    if (err != cudaSuccess) return err;
    const long dn_items = long(T) * H;
    const long dn_grid = std::min<long>((dn_items + q8::kWarps - 1) / q8::kWarps, long(num_sms) * 64);
    launch_pdl(q8::q8k_down_kernel, dim3(unsigned(dn_grid)), dim3(q8::kThreads), size_t(0), s, hq, hd,
               hs, idx, w, down, T, H, E, k, I, y);
    return cudaGetLastError();
}

}  // namespace moeq4k
