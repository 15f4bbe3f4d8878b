// Expert FFN over Q4_K blocks: gate+up with the SwiGLU epilogue, down, and
// the slot-ordered combine.
//
// forward_qwen3_moe.rs (aprender-serve 0.35.0), step 2h of
// forward_single_qwen3_moe_with_cache: each selected expert computes
// SiLU(gate x) * (up x) and its down projection; the outputs are weighted by
// the renormalised router weights and summed.  The weights are consumed in
// place (fused dequant + matvec, doc of forward_qwen3_moe).
//
// Work is split into (active expert, block of 8 rows) items; a CTA of 8
// warps takes one item at a time, one row per warp, and runs that row for
// every token routed to the expert, so each weight byte is fetched from HBM
// once per call.  Inside a warp, lane L decodes the 16-byte code chunk
// L % 8 of block 4*i + L/8 of the row (32 weights: 16 of sub-block 2c and 16
// of sub-block 2c+1, c = (L%8)/2) and takes d, dmin and the 6-bit scales
// from the block's 16-byte head.
#include "common.cuh"
#include "kernels.cuh"

namespace moeq4k {

constexpr int kRowsPerItem = 8;  // one row per warp
constexpr int kTokGroup = 4;     // activation rows staged in shared memory at a time

// Stage `n` activation rows (row ids from `rows_of`) into shared memory with
// their 16-element partial sums (needed for the dmin * m term).
template <typename RowPtr>
__device__ __forceinline__ void stage_rows(float *vs, float *vsum, int n, int len, RowPtr row_ptr) {
    const int len4 = len >> 2;
    for (int i = 0; i < n; ++i) {
        const float4 *src = reinterpret_cast<const float4 *>(row_ptr(i));
        float4 *dst = reinterpret_cast<float4 *>(vs + i * len);
        for (int c = threadIdx.x; c < len4; c += blockDim.x) dst[c] = src[c];
    }
    __syncthreads();
    const int runs = len >> 4;
    for (int i = 0; i < n; ++i) {
        for (int r = threadIdx.x; r < runs; r += blockDim.x) {
            const float *v = vs + i * len + 16 * r;
            float s = 0.f;
#pragma unroll
            for (int b = 0; b < 16; ++b) s += v[b];
            vsum[i * runs + r] = s;
        }
    }
    __syncthreads();
}

// A slot id read back from the permutation, checked against [0, npairs):
// an id outside it is recorded and replaced by 0 so no access leaves the
// buffers (the write of its result is skipped by the caller).
__device__ __forceinline__ int checked_pair(int p, int npairs, WsHeader *hdr, int site) {
    if (p < 0 || p >= npairs) {
        record_status(hdr, MOE_ERR_INTERNAL, site + (p & 0xffffff));
        return 0;
    }
    return p;
}

// Partial dot product of one lane's share of a Q4_K row with staged vector
// `v` (length len = nsb*256, with 16-element partial sums `vsum`).
__device__ __forceinline__ float row_part(const uint8_t *row, int nsb, int lane, const float *v,
                                          const float *vsum) {
    const int cq = lane & 7;        // 16-byte code chunk inside the block
    const int c = cq >> 1;          // 32-byte group: sub-blocks 2c, 2c+1
    const int l0 = (cq & 1) * 16;   // first position inside the sub-block
    float acc = 0.f;
    for (int s = lane >> 3; s < nsb; s += 4) {
        const uint8_t *blk = row + size_t(s) * kBlockBytes;
        uint4 head = ldg_nc_v4(blk);
        uint4 q = ldg_nc_v4(blk + 16 + 16 * cq);
        float2 dd = q4k_d_dmin(head);
        float sc0, m0, sc1, m1;
        q4k_scale_min(head, 2 * c, sc0, m0);
        q4k_scale_min(head, 2 * c + 1, sc1, m1);
        const int base = s * kQK + 64 * c + l0;
        float lo, hi;
        chunk_dot(q, v + base, v + base + 32, lo, hi);
        const float slo = vsum[base >> 4], shi = vsum[(base + 32) >> 4];
        acc += dd.x * (sc0 * lo + sc1 * hi) - dd.y * (m0 * slo + m1 * shi);
    }
    return acc;
}

// gate+up+SwiGLU: h[p, r] = SiLU(Wg[e][r] . x[t]) * (Wu[e][r] . x[t]) for every
// slot p = t*k + j routed to expert e.
__global__ void __launch_bounds__(256) gateup_kernel(const float *__restrict__ x,
                                                     const uint8_t *__restrict__ gate,
                                                     const uint8_t *__restrict__ up,
                                                     const int32_t *__restrict__ offs,
                                                     const int32_t *__restrict__ perm,
                                                     const int32_t *__restrict__ active,
                                                     const int32_t *__restrict__ nactive,
                                                     int H, int I, int k, int E, int npairs,
                                                     float *__restrict__ h, WsHeader *hdr) {
    pdl_enter();
    extern __shared__ float smem[];
    float *xs = smem;                         // [kTokGroup][H]
    float *xsum = smem + kTokGroup * H;       // [kTokGroup][H/16]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nsb = H / kQK;
    const int nrb = I / kRowsPerItem;
    int na = *nactive;
    if (na < 0 || na > E) {
        if (blockIdx.x == 0 && threadIdx.x == 0) record_status(hdr, MOE_ERR_INTERNAL, 500000000 + (na & 0xffffff));
        na = 0;
    }
    const int items = na * nrb;
    const size_t mat_bytes = size_t(I) * nsb * kBlockBytes;
    for (int it = blockIdx.x; it < items; it += gridDim.x) {
        const int e = active[it / nrb];
        if (e < 0 || e >= E) {
            if (threadIdx.x == 0) record_status(hdr, MOE_ERR_INTERNAL, 100000000 + (e & 0xffffff));
            continue;
        }
        const int r = (it % nrb) * kRowsPerItem + warp;
        const int p0 = offs[e], n_e = offs[e + 1] - p0;
        if (p0 < 0 || n_e < 0 || p0 + n_e > npairs) {
            if (threadIdx.x == 0) record_status(hdr, MOE_ERR_INTERNAL, 200000000 + (p0 & 0xffffff));
            continue;
        }
        const uint8_t *grow = gate + e * mat_bytes + size_t(r) * nsb * kBlockBytes;
        const uint8_t *urow = up + e * mat_bytes + size_t(r) * nsb * kBlockBytes;
        for (int g0 = 0; g0 < n_e; g0 += kTokGroup) {
            const int ng = min(kTokGroup, n_e - g0);
            __syncthreads();
            stage_rows(xs, xsum, ng, H, [&](int i) {
                return x + size_t(checked_pair(perm[p0 + g0 + i], npairs, hdr, 300000000) / k) * H;
            });
            for (int i = 0; i < ng; ++i) {
                float g = warp_sum(row_part(grow, nsb, lane, xs + i * H, xsum + i * (H >> 4)));
                float u = warp_sum(row_part(urow, nsb, lane, xs + i * H, xsum + i * (H >> 4)));
                const int p = perm[p0 + g0 + i];
                if (lane == 0 && p >= 0 && p < npairs) h[size_t(p) * I + r] = silu_mul(g, u);
            }
        }
    }
}

// down: o[p, r] = Wd[e][r] . h[p] for every slot p routed to expert e.
__global__ void __launch_bounds__(256) down_kernel(const float *__restrict__ h,
                                                   const uint8_t *__restrict__ down,
                                                   const int32_t *__restrict__ offs,
                                                   const int32_t *__restrict__ perm,
                                                   const int32_t *__restrict__ active,
                                                   const int32_t *__restrict__ nactive,
                                                   int H, int I, int E, int npairs,
                                                   float *__restrict__ o, WsHeader *hdr) {
    pdl_enter();
    extern __shared__ float smem[];
    float *hs = smem;                         // [kTokGroup][I]
    float *hsum = smem + kTokGroup * I;       // [kTokGroup][I/16]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nsb = I / kQK;
    const int nrb = H / kRowsPerItem;
    int na = *nactive;
    if (na < 0 || na > E) {
        if (blockIdx.x == 0 && threadIdx.x == 0) record_status(hdr, MOE_ERR_INTERNAL, 510000000 + (na & 0xffffff));
        na = 0;
    }
    const int items = na * nrb;
    const size_t mat_bytes = size_t(H) * nsb * kBlockBytes;
    for (int it = blockIdx.x; it < items; it += gridDim.x) {
        const int e = active[it / nrb];
        if (e < 0 || e >= E) {
            if (threadIdx.x == 0) record_status(hdr, MOE_ERR_INTERNAL, 110000000 + (e & 0xffffff));
            continue;
        }
        const int r = (it % nrb) * kRowsPerItem + warp;
        const int p0 = offs[e], n_e = offs[e + 1] - p0;
        if (p0 < 0 || n_e < 0 || p0 + n_e > npairs) {
            if (threadIdx.x == 0) record_status(hdr, MOE_ERR_INTERNAL, 210000000 + (p0 & 0xffffff));
            continue;
        }
        const uint8_t *drow = down + e * mat_bytes + size_t(r) * nsb * kBlockBytes;
        for (int g0 = 0; g0 < n_e; g0 += kTokGroup) {
            const int ng = min(kTokGroup, n_e - g0);
            __syncthreads();
            stage_rows(hs, hsum, ng, I, [&](int i) {
                return h + size_t(checked_pair(perm[p0 + g0 + i], npairs, hdr, 310000000)) * I;
            });
            for (int i = 0; i < ng; ++i) {
                float v = warp_sum(row_part(drow, nsb, lane, hs + i * I, hsum + i * (I >> 4)));
                const int p = perm[p0 + g0 + i];
                if (lane == 0 && p >= 0 && p < npairs) o[size_t(p) * H + r] = v;
            }
        }
    }
}

// y[t, :] = sum_j w[t,j] * o[t*k+j, :], j = 0..k-1 in order; slots with an
// expert index outside [0,E) are skipped.  The epilogue then copies token
// cap_t's row out and adds the residual stream.
__global__ void __launch_bounds__(256) combine_kernel(const float *__restrict__ o,
                                                      const int32_t *__restrict__ idx,
                                                      const float *__restrict__ w, int T, int H,
                                                      int E, int k, float *__restrict__ y,
                                                      const OutEpilogue ep) {
    pdl_enter();
    const int h4 = H >> 2;
    const size_t total = size_t(T) * h4;
    for (size_t i = blockIdx.x * size_t(blockDim.x) + threadIdx.x; i < total;
         i += size_t(gridDim.x) * blockDim.x) {
        const int t = int(i / h4), c = int(i % h4);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        // eight slots at a time: every index, weight and output row of the
        // group is requested before the first multiply-add, which then run in
        // slot order (a slot with an index outside [0, E) adds nothing)
        for (int j0 = 0; j0 < k; j0 += 8) {
            bool ok[8];
            float wj[8];
            float4 v[8];
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                const int j = j0 + jj;
                const int e = j < k ? idx[size_t(t) * k + j] : -1;
                ok[jj] = e >= 0 && e < E;
                wj[jj] = ok[jj] ? w[size_t(t) * k + j] : 0.f;
            }
#pragma unroll
            for (int jj = 0; jj < 8; ++jj)
                v[jj] = ok[jj] ? reinterpret_cast<const float4 *>(o + (size_t(t) * k + j0 + jj) * H)[c]
                               : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                if (!ok[jj]) continue;
                acc.x = fmaf(wj[jj], v[jj].x, acc.x);
                acc.y = fmaf(wj[jj], v[jj].y, acc.y);
                acc.z = fmaf(wj[jj], v[jj].z, acc.z);
                acc.w = fmaf(wj[jj], v[jj].w, acc.w);
            }
        }
        if (ep.capture != nullptr && t == ep.cap_t) reinterpret_cast<float4 *>(ep.capture)[c] = acc;
        if (ep.residual != nullptr) {
            const float4 r = reinterpret_cast<const float4 *>(ep.residual + size_t(t) * H)[c];
            acc = make_float4(r.x + acc.x, r.y + acc.y, r.z + acc.z, r.w + acc.w);
        }
        reinterpret_cast<float4 *>(y + size_t(t) * H)[c] = acc;
    }
}

cudaError_t launch_combine(const float *obuf, const int32_t *idx, const float *w, int T, int H,
                           int E, int k, float *y, const OutEpilogue &ep, int num_sms,
                           cudaStream_t s) {
    const size_t total = size_t(T) * (H / 4);
    const size_t g3s = (total + 255) / 256, g3cap = size_t(num_sms) * 16;
    launch_pdl(combine_kernel, dim3(int(g3s < g3cap ? g3s : g3cap)), dim3(256), size_t(0), s, obuf, idx, w, T, H, E, k, y, ep);
    return cudaGetLastError();
}

cudaError_t init_expert_ffn() {
    const int max_smem = int(sizeof(float) * kTokGroup * (kMaxHI + kMaxHI / 16));
    cudaError_t err = cudaFuncSetAttribute(gateup_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
    if (err != cudaSuccess) return err;
    return cudaFuncSetAttribute(down_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
}

cudaError_t launch_expert_ffn(const float *x, const int32_t *idx, const float *w,
                              const uint8_t *gate, const uint8_t *up, const uint8_t *down, int T,
                              int H, int E, int k, int I, float *y, const int32_t *offs,
                              const int32_t *perm, const int32_t *active, const int32_t *nactive,
                              float *hbuf, float *obuf, WsHeader *hdr, const OutEpilogue &ep,
                              int num_sms, cudaStream_t s) {
    const int max_active = min(E, T * k);
    const size_t smem_gu = sizeof(float) * kTokGroup * (H + H / 16);
    const size_t smem_dn = sizeof(float) * kTokGroup * (I + I / 16);
    const int cap = num_sms * 8;
    int g1 = min(max_active * (I / kRowsPerItem), cap);
    launch_pdl(gateup_kernel, dim3(g1), dim3(256), size_t(smem_gu), s, x, gate, up, offs, perm, active, nactive, H, I, k, E,
                                           T * k, hbuf, hdr);
    int g2 = min(max_active * (H / kRowsPerItem), cap);
    launch_pdl(down_kernel, dim3(g2), dim3(256), size_t(smem_dn), s, hbuf, down, offs, perm, active, nactive, H, I, E, T * k,
                                         obuf, hdr);
    const size_t total = size_t(T) * (H / 4);
    const size_t g3s = (total + 255) / 256, g3cap = size_t(num_sms) * 16;
    int g3 = int(g3s < g3cap ? g3s : g3cap);
    launch_pdl(combine_kernel, dim3(g3), dim3(256), size_t(0), s, obuf, idx, w, T, H, E, k, y, ep);
    return cudaGetLastError();
}

}  // namespace moeq4k
