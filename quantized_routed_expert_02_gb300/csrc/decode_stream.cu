// Single token, rows streamed from HBM: the layer for one token when its
// expert rows do not fit the fused kernel's shared-memory slots (the
// Qwen3-235B-A22B shape: 85 MB of Q4_K rows per token).
//
// forward_qwen3_moe.rs (aprender-serve 0.35.0), step 2h of
// forward_single_qwen3_moe_with_cache: each of the token's k experts computes
// h_j = SiLU(Wg[e_j] x) * (Wu[e_j] x), its down projection o_j = Wd[e_j] h_j,
// and y = sum_j w_j o_j in slot order.  Two launches after the router, each
// with one persistent CTA per SM:
//   gate/up  x becomes integer digit planes in shared memory; thread t keeps
//            the digits of unit t % (H/64) of x (a sub-block pair: 64
//            elements) in registers and, round after round, loads that
//            unit's 48 bytes of one gate row and one up row (the next
//            round's loads issued before this round's arithmetic), dots them
//            with dp4a, and leaves the partial sums in shared memory, where
//            one warp per row adds them in a fixed order;
//   down     the concatenated h_1..h_k (k*I/64 units) as digit planes; a
//            warp per output row r, lanes over the units (a unit belongs to
//            one slot j and dots row r of Wd[e_j]), all of a lane's row bytes
//            requested before its arithmetic, the digits read from shared
//            memory at the dot; y[r] = sum over units of w_j times the unit's
//            dot, one fixed-order warp sum: no o buffer, no combine pass and
//            no CTA-wide barrier after the staging.
// Shapes the digit layout does not cover (H not a power of two, or k*I/64
// above the CTA's 512 threads) take fp32 fallbacks with the same results up
// to rounding: warp per (slot, row) for gate/up, warp per output row for
// down.  Weights are read once per call with read-only 16-byte loads.
#include "common.cuh"
#include "kernels.cuh"
#include "q4k_dot.cuh"

namespace moeq4k {
namespace dst {

constexpr int kGuThreads = 256;
constexpr int kGuBlocksPerSm = 2;
constexpr int kDnThreads = 512;
constexpr int kDnPairsInFlight = 4;  // per lane: slots x blocks of down rows loaded together
constexpr int kDgThreads = 512;      // digit kernels: one thread per unit of the vector

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

__device__ __forceinline__ float pair_dot(const Pair &P, int c, const float *xs, const float *s2) {
    return moeq4k::pair_dot(P.head, P.qa, P.qb, c, xs, s2);
}

__device__ __forceinline__ float pair_dot_digits(const Pair &P, int c, const XDigits &X) {
    return moeq4k::pair_dot_digits(P.head, P.qa, P.qb, c, X);
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

// The CTA's contiguous share [*lo, *hi) of n work units.
__device__ __forceinline__ void cta_share(int n, int *lo, int *hi) {
    const int per = (n + gridDim.x - 1) / gridDim.x;
    *lo = min(n, int(blockIdx.x) * per);
    *hi = min(n, *lo + per);
}

// h[j*I + r] = SiLU(Wg[e_j][r] . x) * (Wu[e_j][r] . x).  NB = blocks per
// lane (ceil(H / 2048)).
template <int NB>
__global__ void __launch_bounds__(kGuThreads, kGuBlocksPerSm)
    stream_gateup_kernel(const float *__restrict__ x, const uint8_t *__restrict__ gate,
                         const uint8_t *__restrict__ up, const int32_t *__restrict__ idx, int k,
                         int E, int H, int I, float *__restrict__ h, WsHeader *hdr) {
    pdl_enter();
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
                       int H, int I, float *__restrict__ y, WsHeader *hdr, const OutEpilogue ep) {
    pdl_enter();
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
        if (lane == 0) y[r] = epilogue_value(ep, 0, H, r, acc);
    }
}

// A vector of n floats (n a multiple of 128) as three digit planes (n bytes
// each, unit-major 16-byte chunks: plane_offset), a scale and a sum per
// 32-element run.  Warps take 128-element chunks, lane l elements 4l..4l+3.
__device__ __forceinline__ void stage_digits(const float *__restrict__ src, int n, uint8_t *planes,
                                             float *scales, float *sums) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    const int nunits = n >> 6, nch = n >> 7;
    constexpr int kBatch = 4;  // chunks a warp loads before converting any
    for (int base = warp; base < nch; base += kBatch * nw) {
        float4 v[kBatch];
#pragma unroll
        for (int t = 0; t < kBatch; ++t) {
            const int ch = base + t * nw;
            if (ch < nch) v[t] = __ldg(reinterpret_cast<const float4 *>(src + 128 * ch + 4 * lane));
        }
#pragma unroll
        for (int t = 0; t < kBatch; ++t) {
            const int ch = base + t * nw;
            if (ch >= nch) break;  // uniform over the warp
            const int e0 = 128 * ch + 4 * lane;
            uint32_t wa, wb, wc;
            float sum;
            const float sc = run_digits4(v[t], lane, wa, wb, wc, sum);
            const int off = plane_offset(e0, nunits);
            *reinterpret_cast<uint32_t *>(planes + off) = wa;
            *reinterpret_cast<uint32_t *>(planes + n + off) = wb;
            *reinterpret_cast<uint32_t *>(planes + 2 * n + off) = wc;
            if ((lane & 7) == 0) {
                scales[e0 >> 5] = sc;
                sums[e0 >> 5] = sum;
            }
        }
    }
}

// h[j*I + r] = SiLU(Wg[e_j][r] . x) * (Wu[e_j][r] . x) with x as digits.
// UX = H/64 units (a power of two <= 512); Q = 512/UX items per round.
__global__ void __launch_bounds__(kDgThreads, 1)
    stream_gateup_digits_kernel(const float *__restrict__ x, const uint8_t *__restrict__ gate,
                                const uint8_t *__restrict__ up, const int32_t *__restrict__ idx,
                                int k, int E, int H, int I, float *__restrict__ h, WsHeader *hdr) {
    pdl_enter();
    extern __shared__ __align__(16) uint8_t smd[];
    const int UX = H >> 6, Q = kDgThreads / UX;
    uint8_t *planes = smd;                                      // 3H bytes
    float *xscale = reinterpret_cast<float *>(smd + 3 * H);     // H/32
    float *xsum = xscale + H / 32;                              // H/32
    float *P = xsum + H / 32;                                   // [2][Q][2][UX]
    int *eid = reinterpret_cast<int *>(P + 2 * kDgThreads * 2);  // [k]
    load_experts(idx, k, E, eid, hdr);
    __syncthreads();

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, nw = blockDim.x >> 5;
    const int u = tid % UX, q = tid / UX, sb = u >> 2, c = u & 3;
    const size_t row_bytes = size_t(H / kQK) * kBlockBytes, mat = size_t(I) * row_bytes;
    int it0, it1;
    cta_share(k * I, &it0, &it1);
    const int rounds = (it1 - it0 + Q - 1) / Q;

    // this thread's item of round rd: its gate and up bytes, if any
    auto load = [&](int rd, Pair &pg, Pair &pu) -> bool {
        const int item = it0 + rd * Q + q;
        if (item >= it1) return false;
        const int j = item / I, r = item - j * I, e = eid[j];
        if (e < 0) return false;
        const size_t off = size_t(e) * mat + size_t(r) * row_bytes + size_t(sb) * kBlockBytes;
        pg = load_pair(gate + off, c);
        pu = load_pair(up + off, c);
        return true;
    };
    // the first round's rows are requested before x is converted
    Pair cg, cu, ng, nu;
    bool have = rounds > 0 && load(0, cg, cu);
    stage_digits(x, H, planes, xscale, xsum);
    __syncthreads();
    XDigits X;
    load_digits(X, planes, H, UX, u, xscale, xsum);
    for (int rd = 0; rd < rounds; ++rd) {
        const bool have_next = rd + 1 < rounds && load(rd + 1, ng, nu);
        float g = 0.f, v = 0.f;
        if (have) {
            g = pair_dot_digits(cg, c, X);
            v = pair_dot_digits(cu, c, X);
        }
        float *Pb = P + (rd & 1) * (kDgThreads * 2);
        Pb[(2 * q) * UX + u] = g;
        Pb[(2 * q + 1) * UX + u] = v;
        __syncthreads();  // also orders the reuse of the other buffer two rounds on
        for (int qq = warp; qq < Q; qq += nw) {
            const int item = it0 + rd * Q + qq;
            if (item >= it1) break;
            const int j = item / I, r = item - j * I;
            if (eid[j] < 0) continue;
            float gs = 0.f, us = 0.f;
            for (int uu = lane; uu < UX; uu += 32) {
                gs += Pb[(2 * qq) * UX + uu];
                us += Pb[(2 * qq + 1) * UX + uu];
            }
            gs = warp_sum(gs);
            us = warp_sum(us);
            if (lane == 0) h[size_t(j) * I + r] = silu_mul(gs, us);
        }
        cg = ng;
        cu = nu;
        have = have_next;
    }
}

// Dot of sub-blocks 2c and 2c+1 of one block with unit u of a digit vector
// read straight from the shared planes (the digits of a unit are not kept in
// registers: a lane visits several units per row).  Same integer sums and
// scalings as pair_dot_digits.
__device__ __forceinline__ float pair_dot_digits_smem(const Pair &P, int c, const uint8_t *planes,
                                                      int plane_bytes, int nunits, int u,
                                                      const float *scales, const float *sums) {
    const uint32_t w[8] = {P.qa.x, P.qa.y, P.qa.z, P.qa.w, P.qb.x, P.qb.y, P.qb.z, P.qb.w};
    int a0 = 0, b0 = 0, c0 = 0, a1 = 0, b1 = 0, c1 = 0;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        // chunk `half` holds the low sub-block's elements 16 half ..; chunk
        // 2 + half the high sub-block's
        const uint8_t *lo_ch = planes + (half * nunits + u) * 16;
        const uint8_t *hi_ch = planes + ((2 + half) * nunits + u) * 16;
        const uint4 la = *reinterpret_cast<const uint4 *>(lo_ch);
        const uint4 lb = *reinterpret_cast<const uint4 *>(lo_ch + plane_bytes);
        const uint4 lc = *reinterpret_cast<const uint4 *>(lo_ch + 2 * plane_bytes);
        const uint4 ha = *reinterpret_cast<const uint4 *>(hi_ch);
        const uint4 hb = *reinterpret_cast<const uint4 *>(hi_ch + plane_bytes);
        const uint4 hc = *reinterpret_cast<const uint4 *>(hi_ch + 2 * plane_bytes);
        const uint32_t da[4] = {la.x, la.y, la.z, la.w}, db[4] = {lb.x, lb.y, lb.z, lb.w},
                       dc[4] = {lc.x, lc.y, lc.z, lc.w};
        const uint32_t ea[4] = {ha.x, ha.y, ha.z, ha.w}, eb[4] = {hb.x, hb.y, hb.z, hb.w},
                       ec[4] = {hc.x, hc.y, hc.z, hc.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t q = w[4 * half + i];
            const uint32_t lo = q & 0x0F0F0F0Fu, hi = q & 0xF0F0F0F0u;
            a0 = dp4a_us(lo, da[i], a0);
            b0 = dp4a_us(lo, db[i], b0);
            c0 = dp4a_us(lo, dc[i], c0);
            a1 = dp4a_us(hi, ea[i], a1);
            b1 = dp4a_us(hi, eb[i], b1);
            c1 = dp4a_us(hi, ec[i], c1);
        }
    }
    const int r0 = (64 * u) >> 5;
    const float qx0 = scales[r0] * fmaf(float(c0), 1.0f / 254.0f, float(254 * a0 + b0));
    const float qx1 = scales[r0 + 1] * 0.0625f * fmaf(float(c1), 1.0f / 254.0f, float(254 * a1 + b1));
    float A0, B0, A1, B1;
    pair_scales(P.head, c, 1.0f, A0, B0, A1, B1);
    float acc = A0 * qx0;
    acc = fmaf(-B0, sums[r0], acc);
    acc = fmaf(A1, qx1, acc);
    acc = fmaf(-B1, sums[r0 + 1], acc);
    return acc;
}

// y[r] = sum over the n/64 units u of the concatenated h digits of
// w_{j(u)} * (unit u of row r of Wd[e_j] . h_j): a warp per output row,
// lanes over units (unit lane + 32 g), all of a lane's G units requested
// before any arithmetic; one fixed-order warp sum per row.  The CTA's rows
// are a contiguous share, so its warps read consecutive rows of every
// expert at once.  No CTA-wide barrier after the staging.
template <int G>
__global__ void __launch_bounds__(kDgThreads, 1)
    stream_down_rows_kernel(const float *__restrict__ h, const uint8_t *__restrict__ down,
                            const int32_t *__restrict__ idx, const float *__restrict__ w, int k,
                            int E, int H, int I, float *__restrict__ y, WsHeader *hdr,
                            const OutEpilogue ep) {
    pdl_enter();
    extern __shared__ __align__(16) uint8_t smd[];
    const int n = k * I, UD = n >> 6, upr = I >> 6;
    uint8_t *planes = smd;                                      // 3n bytes
    float *hscale = reinterpret_cast<float *>(smd + 3 * size_t(n));
    float *hsum = hscale + n / 32;
    float *wj = hsum + n / 32;                                  // [k]
    int *eid = reinterpret_cast<int *>(wj + k);                 // [k]
    load_experts(idx, k, E, eid, hdr);
    for (int j = threadIdx.x; j < k; j += blockDim.x) wj[j] = w[j];
    stage_digits(h, n, planes, hscale, hsum);
    __syncthreads();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
    const size_t row_bytes = size_t(I / kQK) * kBlockBytes, mat = size_t(H) * row_bytes;
    int r0, r1;
    cta_share(H, &r0, &r1);
    for (int r = r0 + warp; r < r1; r += nw) {
        float acc = 0.f;
        for (int u0 = 0; u0 < UD; u0 += 32 * G) {
            Pair P[G];
            bool ok[G];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const int u = u0 + lane + 32 * g;
                const int j = u / upr, uin = u - j * upr;
                ok[g] = u < UD && eid[min(j, k - 1)] >= 0;
                if (ok[g])
                    P[g] = load_pair(down + size_t(eid[j]) * mat + size_t(r) * row_bytes +
                                         size_t(uin >> 2) * kBlockBytes,
                                     uin & 3);
            }
#pragma unroll
            for (int g = 0; g < G; ++g) {
                if (!ok[g]) continue;
                const int u = u0 + lane + 32 * g;
                const int j = u / upr, uin = u - j * upr;
                acc = fmaf(wj[j], pair_dot_digits_smem(P[g], uin & 3, planes, n, UD, u, hscale, hsum),
                           acc);
            }
        }
        acc = warp_sum(acc);
        if (lane == 0) y[r] = epilogue_value(ep, 0, H, r, acc);
    }
}

bool gateup_digits_ok(int H) { return H >= 256 && H <= 64 * kDgThreads && (H & (H - 1)) == 0; }
bool down_digits_ok(int k, int I) { return size_t(k) * I <= size_t(64) * 512; }
size_t gateup_digits_smem(int H, int k) {
    return 3 * size_t(H) + sizeof(float) * (H / 16 + 4 * kDgThreads) + sizeof(int) * k;
}
size_t down_digits_smem(int k, int I) {
    const size_t n = size_t(k) * I;
    return 3 * n + sizeof(float) * (n / 16 + k) + sizeof(int) * k;
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
    const void *rows[] = {reinterpret_cast<const void *>(stream_down_rows_kernel<1>),
                          reinterpret_cast<const void *>(stream_down_rows_kernel<2>),
                          reinterpret_cast<const void *>(stream_down_rows_kernel<4>),
                          reinterpret_cast<const void *>(stream_down_rows_kernel<6>)};
    for (const void *f : rows) {
        err = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
        if (err != cudaSuccess) return err;
    }
    return cudaSuccess;
}

bool decode_stream_supported(int dev, int T, int H, int E, int k, int I) {
    using namespace dst;
    if (T != 1 || H % kQK != 0 || I % kQK != 0 || H > 8192 || I > 8192) return false;
    const size_t optin = size_t(g_stream_smem_optin[dev]);
    const bool gu = gateup_digits_ok(H) ? gateup_digits_smem(H, k) <= 48 * 1024
                                        : gateup_smem(H, k) <= 48 * 1024;
    const bool dn = down_digits_ok(k, I) ? down_digits_smem(k, I) <= optin : down_smem(I, k) <= optin;
    return gu && dn;
}

cudaError_t launch_decode_stream(const float *x, const int32_t *idx, const float *w,
                                 const uint8_t *gate, const uint8_t *up, const uint8_t *down,
                                 int H, int E, int k, int I, float *y, float *hbuf, WsHeader *hdr,
                                 const OutEpilogue &ep, int num_sms, cudaStream_t s) {
    using namespace dst;
    const int nbh = (H / kQK + 7) / 8, nbi = (I / kQK + 7) / 8;
    const size_t sg = gateup_smem(H, k), sd = down_smem(I, k);
    const int gg = num_sms * kGuBlocksPerSm;
    if (gateup_digits_ok(H))
        launch_pdl(stream_gateup_digits_kernel, dim3(num_sms), dim3(kDgThreads),
                   gateup_digits_smem(H, k), s, x, gate, up, idx, k, E, H, I, hbuf, hdr);
    else if (nbh <= 1)
        launch_pdl(stream_gateup_kernel<1>, dim3(gg), dim3(kGuThreads), size_t(sg), s, x, gate, up, idx, k, E, H, I, hbuf, hdr);
    else if (nbh <= 2)
        launch_pdl(stream_gateup_kernel<2>, dim3(gg), dim3(kGuThreads), size_t(sg), s, x, gate, up, idx, k, E, H, I, hbuf, hdr);
    else
        launch_pdl(stream_gateup_kernel<4>, dim3(gg), dim3(kGuThreads), size_t(sg), s, x, gate, up, idx, k, E, H, I, hbuf, hdr);
    if (down_digits_ok(k, I)) {
        const int ud = k * I / 64;  // units per output row; lanes take ceil(ud / 32) each
        const size_t sdd = down_digits_smem(k, I);
        if (ud <= 32)
            launch_pdl(stream_down_rows_kernel<1>, dim3(num_sms), dim3(kDgThreads), size_t(sdd), s, hbuf, down, idx, w, k, E, H, I, y, hdr, ep);
        else if (ud <= 64)
            launch_pdl(stream_down_rows_kernel<2>, dim3(num_sms), dim3(kDgThreads), size_t(sdd), s, hbuf, down, idx, w, k, E, H, I, y, hdr, ep);
        else if (ud <= 128)
            launch_pdl(stream_down_rows_kernel<4>, dim3(num_sms), dim3(kDgThreads), size_t(sdd), s, hbuf, down, idx, w, k, E, H, I, y, hdr, ep);
        else if (ud <= 192)
            launch_pdl(stream_down_rows_kernel<6>, dim3(num_sms), dim3(kDgThreads), size_t(sdd), s, hbuf, down, idx, w, k, E, H, I, y, hdr, ep);
        else  // four units per lane in flight, looping over the rest (a wider
              // batch of loads per lane would spill at the 128-register cap)
            launch_pdl(stream_down_rows_kernel<4>, dim3(num_sms), dim3(kDgThreads), size_t(sdd), s, hbuf, down, idx, w, k, E, H, I, y, hdr, ep);
    }
    else if (nbi <= 1)
        launch_pdl(stream_down_kernel<1>, dim3(num_sms), dim3(kDnThreads), size_t(sd), s, hbuf, down, idx, w, k, E, H, I, y, hdr, ep);
    else if (nbi <= 2)
        launch_pdl(stream_down_kernel<2>, dim3(num_sms), dim3(kDnThreads), size_t(sd), s, hbuf, down, idx, w, k, E, H, I, y, hdr, ep);
    else
        launch_pdl(stream_down_kernel<4>, dim3(num_sms), dim3(kDnThreads), size_t(sd), s, hbuf, down, idx, w, k, E, H, I, y, hdr, ep);
    return cudaGetLastError();
}

}  // namespace moeq4k
