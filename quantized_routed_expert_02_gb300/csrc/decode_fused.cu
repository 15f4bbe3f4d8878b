// Single-token decode of the whole routed-expert layer in one persistent
// kernel: router -> top-k -> gate/up + SwiGLU -> down -> slot-ordered combine.
//
// forward_qwen3_moe.rs (aprender-serve 0.35.0), step 2h of
// forward_single_qwen3_moe_with_cache: one token's MoE FFN is the gate x up
// SwiGLU of each selected expert weighted by the softmax-normalised top-k
// router weights; forward_qwen3_moe_cuda_traced.rs (aprender-serve 0.34.0),
// doc of forward_qwen3_moe_cuda_traced_with_plan: the router stage is the k
// post-softmax, renormalised weights and the output stage is [H].
//
// Design (one CTA of 16 warps per SM, cooperative launch so every CTA is
// resident):
//  1. Every CTA stages x in shared memory and computes a share of the E
//     router logits (Wr read with an L2 evict-last policy: it is re-read by
//     every token, unlike the expert bytes, which are read evict-first).
//  2. Grid barrier; every CTA reads the E logits and runs the same top-k and
//     renormalisation, so all CTAs know the k experts without a broadcast.
//  3. The k*I gate/up row pairs are split evenly over the CTAs and, inside a
//     CTA, over its warps.  Each warp streams its own rows into a private
//     ring of shared-memory slots with 16-byte cp.async copies (every lane
//     issues, so hundreds of requests per SM are in flight; one commit group
//     per row, waited with cp.async.wait_group), decodes nibbles and 6-bit scales
//     in registers, does fp32 FMAs against x in shared memory, and writes
//     h = SiLU(g) * u to the workspace.  When the CTA's down rows (its share
//     of the H output rows, for all k experts) fit beside the rings, all
//     threads prefetch them right after the first gate/up rows.
//  4. Grid barrier; each CTA stages h of all k slots, then for each of its
//     output rows computes o_j = Wd[e_j][row] . h_j for j = 0..k-1 and
//     y = sum_j w_j o_j in slot order: deterministic, no atomics.
// The grid barrier is a monotonic 64-bit arrival counter (release add,
// acquire polling), so it needs no reset between calls or graph replays.
// The grid-barrier wait is bounded by a global-timer deadline; on expiry the
// kernel records MOE_ERR_TIMEOUT, stops computing and lets its copies land
// before returning.  (Copy completion needs no bound: loads always finish.)
#include <algorithm>

#include "async_copy.cuh"
#include "common.cuh"
#include "kernels.cuh"

namespace moeq4k {
namespace fused {

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kMaxNbw = 8;         // ring slots per warp
constexpr int kHeadBytes = 4096;   // small shared arrays

// Optional phase timeline for profiling builds (-DMOEQ4K_TIMELINE): thread 0
// of each CTA stamps the global timer at phase boundaries into the
// workspace's per-slot output region, which this path does not otherwise use.
#ifdef MOEQ4K_TIMELINE
#define TL_STAMP(p, i) ((p).timeline[blockIdx.x * 16 + (i)] = global_timer_ns())
#else
#define TL_STAMP(p, i) ((void)0)
#endif

struct Params {
    const float *x, *Wr, *bias;
    const int32_t *idx_in;
    const float *w_in;
    int32_t *idx_out;
    float *w_out;
    const uint8_t *gate, *up, *down;
    float *y, *logits, *hbuf;
    WsHeader *hdr;
    int H, E, k, I;
    int router_on;
    int nbw, slot_bytes, ring_off;
    int down_resident, down_off;  // CTA's down rows prefetched into [down_off, ...)
    int withhold;                 // test hook: extra arrivals the grid barrier waits for
    unsigned long long wait_ns;   // bound of the grid-barrier waits
    unsigned long long *timeline; // profiling builds only
};

// Padded shared-memory vector: 4 floats of padding after every 64, so the
// 8 lanes of a quarter-warp reading 16-float runs that are 64 floats apart
// hit distinct banks.
__device__ __forceinline__ int padded(int i) { return i + ((i >> 6) << 2); }
__host__ __device__ inline int padded_len(int n) { return n + (n >> 4); }

// 1 + q/128 as fp32 from byte i of v, where v's bytes are 0x80 | q.
__device__ __forceinline__ float one_plus_q(uint32_t v, int i) {
    return __uint_as_float(__byte_perm(v, 0x3F000000u, 0x7044u | (uint32_t(i) << 8)));
}

// sum_b (1 + q_lo[b]/128) x_lo[b] and the same for the high nibbles, for one
// 16-byte code chunk; x_lo = xs[0..15], x_hi = xs[32..47].
__device__ __forceinline__ void chunk_acc(const uint4 &q, const float *xs, float &alo, float &ahi) {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int wi = 0; wi < 4; ++wi) {
        const uint32_t lo = (w[wi] & 0x0F0F0F0Fu) | 0x80808080u;
        const uint32_t hi = ((w[wi] >> 4) & 0x0F0F0F0Fu) | 0x80808080u;
        const float4 xl = *reinterpret_cast<const float4 *>(xs + 4 * wi);
        const float4 xh = *reinterpret_cast<const float4 *>(xs + 32 + 4 * wi);
        alo = fmaf(one_plus_q(lo, 0), xl.x, alo);
        alo = fmaf(one_plus_q(lo, 1), xl.y, alo);
        alo = fmaf(one_plus_q(lo, 2), xl.z, alo);
        alo = fmaf(one_plus_q(lo, 3), xl.w, alo);
        ahi = fmaf(one_plus_q(hi, 0), xh.x, ahi);
        ahi = fmaf(one_plus_q(hi, 1), xh.y, ahi);
        ahi = fmaf(one_plus_q(hi, 2), xh.z, ahi);
        ahi = fmaf(one_plus_q(hi, 3), xh.w, ahi);
    }
}

__device__ __forceinline__ float u6_to_float(uint32_t v) {
    return __uint_as_float(0x4B000000u | v) - 8388608.0f;
}

// One lane's share of a Q4_K row (nsb blocks in shared memory at `row`)
// dotted with the padded vector `vec` (16-element run sums in `vsum`).  Lane
// L takes code chunk L%8 of blocks L/8, L/8+4, ...
template <int NSB>
__device__ __forceinline__ float row_lane_dot(const uint8_t *row, int nsb_rt, const float *vec,
                                              const float *vsum, int lane) {
    const int nsb = NSB > 0 ? NSB : nsb_rt;
    const int cq = lane & 7, c = cq >> 1, hf = cq & 1;
    const bool upper = c >= 2;  // sub-blocks 4..7 keep their high scale bits elsewhere
    const int j0 = 2 * c, j1 = 2 * c + 1;
    float acc = 0.f;
#pragma unroll(NSB > 8 ? 2 : 4)
    for (int s = lane >> 3; s < nsb; s += 4) {
        const uint8_t *blk = row + s * kBlockBytes;
        const uint4 head = *reinterpret_cast<const uint4 *>(blk);
        const uint4 q = *reinterpret_cast<const uint4 *>(blk + 16 + 16 * cq);
        const int base = s * kQK + 64 * c + 16 * hf;
        const float *xs = vec + padded(base);
        float alo = 0.f, ahi = 0.f;
        chunk_acc(q, xs, alo, ahi);
        const float slo = vsum[base >> 4], shi = vsum[(base >> 4) + 2];
        uint32_t sc0, m0, sc1, m1;
        if (!upper) {
            sc0 = (head.y >> (8 * j0)) & 63u;
            m0 = (head.z >> (8 * j0)) & 63u;
            sc1 = (head.y >> (8 * j1)) & 63u;
            m1 = (head.z >> (8 * j1)) & 63u;
        } else {
            const int a = j0 - 4, b = j1 - 4;
            sc0 = ((head.w >> (8 * a)) & 15u) | (((head.y >> (8 * a + 6)) & 3u) << 4);
            m0 = ((head.w >> (8 * a + 4)) & 15u) | (((head.z >> (8 * a + 6)) & 3u) << 4);
            sc1 = ((head.w >> (8 * b)) & 15u) | (((head.y >> (8 * b + 6)) & 3u) << 4);
            m1 = ((head.w >> (8 * b + 4)) & 15u) | (((head.z >> (8 * b + 6)) & 3u) << 4);
        }
        const float2 dd = __half22float2(*reinterpret_cast<const __half2 *>(&head.x));
        const float d128 = dd.x * 128.0f;
        const float A0 = d128 * u6_to_float(sc0), A1 = d128 * u6_to_float(sc1);
        const float B0 = dd.y * u6_to_float(m0), B1 = dd.y * u6_to_float(m1);
        // d*sc*sum(q x) - dmin*m*sum(x), with sum(q x) = 128*(acc - sum(x))
        acc = fmaf(A0, alo - slo, acc);
        acc = fmaf(-B0, slo, acc);
        acc = fmaf(A1, ahi - shi, acc);
        acc = fmaf(-B1, shi, acc);
    }
    return acc;
}

// Contribution of one 16-byte code chunk (chunk cq of the block at `blk`)
// to a row dot product with the padded vector `vec` / run sums `vsum`; the
// block is block `s` of its row.
__device__ __forceinline__ float block_chunk_dot(const uint8_t *blk, int s, int cq, const float *vec,
                                                 const float *vsum) {
    const int c = cq >> 1, hf = cq & 1;
    const uint4 head = *reinterpret_cast<const uint4 *>(blk);
    const uint4 q = *reinterpret_cast<const uint4 *>(blk + 16 + 16 * cq);
    const int base = s * kQK + 64 * c + 16 * hf;
    float alo = 0.f, ahi = 0.f;
    chunk_acc(q, vec + padded(base), alo, ahi);
    const float slo = vsum[base >> 4], shi = vsum[(base >> 4) + 2];
    const int j0 = 2 * c, j1 = 2 * c + 1;
    uint32_t sc0, m0, sc1, m1;
    if (c < 2) {
        sc0 = (head.y >> (8 * j0)) & 63u;
        m0 = (head.z >> (8 * j0)) & 63u;
        sc1 = (head.y >> (8 * j1)) & 63u;
        m1 = (head.z >> (8 * j1)) & 63u;
    } else {
        const int a = j0 - 4, b = j1 - 4;
        sc0 = ((head.w >> (8 * a)) & 15u) | (((head.y >> (8 * a + 6)) & 3u) << 4);
        m0 = ((head.w >> (8 * a + 4)) & 15u) | (((head.z >> (8 * a + 6)) & 3u) << 4);
        sc1 = ((head.w >> (8 * b)) & 15u) | (((head.y >> (8 * b + 6)) & 3u) << 4);
        m1 = ((head.w >> (8 * b + 4)) & 15u) | (((head.z >> (8 * b + 6)) & 3u) << 4);
    }
    const float2 dd = __half22float2(*reinterpret_cast<const __half2 *>(&head.x));
    const float d128 = dd.x * 128.0f;
    float acc = (d128 * u6_to_float(sc0)) * (alo - slo);
    acc = fmaf(-dd.y * u6_to_float(m0), slo, acc);
    acc = fmaf(d128 * u6_to_float(sc1), ahi - shi, acc);
    acc = fmaf(-dd.y * u6_to_float(m1), shi, acc);
    return acc;
}

// Scale and min of sub-blocks 2c and 2c+1 of a block head, as d*sc*128 and
// dmin*m (the 128 undoes the 1 + q/128 encoding of the codes).
__device__ __forceinline__ void pair_scales(const uint4 &head, int c, float &A0, float &B0, float &A1,
                                            float &B1) {
    const int j0 = 2 * c, j1 = 2 * c + 1;
    uint32_t sc0, m0, sc1, m1;
    if (c < 2) {
        sc0 = (head.y >> (8 * j0)) & 63u;
        m0 = (head.z >> (8 * j0)) & 63u;
        sc1 = (head.y >> (8 * j1)) & 63u;
        m1 = (head.z >> (8 * j1)) & 63u;
    } else {
        const int a = j0 - 4, b = j1 - 4;
        sc0 = ((head.w >> (8 * a)) & 15u) | (((head.y >> (8 * a + 6)) & 3u) << 4);
        m0 = ((head.w >> (8 * a + 4)) & 15u) | (((head.z >> (8 * a + 6)) & 3u) << 4);
        sc1 = ((head.w >> (8 * b)) & 15u) | (((head.y >> (8 * b + 6)) & 3u) << 4);
        m1 = ((head.w >> (8 * b + 4)) & 15u) | (((head.z >> (8 * b + 6)) & 3u) << 4);
    }
    const float2 dd = __half22float2(*reinterpret_cast<const __half2 *>(&head.x));
    const float d128 = dd.x * 128.0f;
    A0 = d128 * u6_to_float(sc0);
    A1 = d128 * u6_to_float(sc1);
    B0 = dd.y * u6_to_float(m0);
    B1 = dd.y * u6_to_float(m1);
}

// Dot of sub-blocks 2c (low nibbles of qs[32c..32c+31]) and 2c+1 (high
// nibbles) of one block with the padded vector: `xs` points at the block's
// element 64c (32 x values for 2c, then 32 for 2c+1), `s2` at the two
// 32-element sums.  Four independent accumulators keep the FMA chains short.
__device__ __forceinline__ float pair_dot(const uint8_t *blk, int c, const float *xs,
                                          const float *s2) {
    const uint4 head = *reinterpret_cast<const uint4 *>(blk);
    const uint4 qa = *reinterpret_cast<const uint4 *>(blk + 16 + 32 * c);
    const uint4 qb = *reinterpret_cast<const uint4 *>(blk + 32 + 32 * c);
    const uint32_t w[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
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
    float A0, B0, A1, B1;
    pair_scales(head, c, A0, B0, A1, B1);
    const float slo = s2[0], shi = s2[1];
    // d*sc*sum(q x) - dmin*m*sum(x), with sum(q x) = 128*(acc - sum(x))
    float acc = A0 * ((a0 + a1) - slo);
    acc = fmaf(-B0, slo, acc);
    acc = fmaf(A1, (b0 + b1) - shi, acc);
    acc = fmaf(-B1, shi, acc);
    return acc;
}

// One lane's share of a Q4_K row in shared memory: lane L takes sub-block
// pair L%4 of blocks L/4, L/4+8, ...  `vec` is the padded vector, `sum32`
// its 32-element sums.
template <int NSB>
__device__ __forceinline__ float row_dot_pairs(const uint8_t *row, int nsb_rt, const float *vec,
                                               const float *sum32, int lane) {
    const int nsb = NSB > 0 ? NSB : nsb_rt;
    const int c = lane & 3;
    float acc = 0.f;
#pragma unroll
    for (int s = lane >> 2; s < nsb; s += 8)
        acc += pair_dot(row + s * kBlockBytes, c, vec + padded(s * kQK + 64 * c),
                        sum32 + s * 8 + 2 * c);
    return acc;
}

// Sum each 32-float run of the padded vector(s) into sum32; run q starts at
// logical element 32*(q % runs_per_vec) of vector q / runs_per_vec.
__device__ __forceinline__ void run_sums32(const float *vec, float *sum32, int count,
                                           int runs_per_vec, int vec_stride) {
    for (int q = threadIdx.x; q < count; q += kThreads) {
        const int j = q / runs_per_vec, c = 32 * (q % runs_per_vec);
        const float *v = vec + j * vec_stride + padded(c);
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int b = 0; b < 32; b += 2) {
            s0 += v[b];
            s1 += v[b + 1];
        }
        sum32[q] = s0 + s1;
    }
}

// Sum each 16-float run of `count` runs of the padded vector(s) into vsum.
// Run q starts at logical element 16*(q % runs_per_vec) of vector q / runs_per_vec.
__device__ __forceinline__ void run_sums(const float *vec, float *vsum, int count, int runs_per_vec,
                                         int vec_stride) {
    for (int q = threadIdx.x; q < count; q += kThreads) {
        const int j = q / runs_per_vec, c = 16 * (q % runs_per_vec);
        const float *v = vec + j * vec_stride + padded(c);
        float s = 0.f;
#pragma unroll
        for (int b = 0; b < 16; ++b) s += v[b];
        vsum[q] = s;
    }
}

// Grid barrier on a monotonic arrival counter: arrive (release), then wait
// (acquire) until the counter reaches `target`.  All threads of the CTA call
// it; returns false on time-out.
__device__ __forceinline__ bool grid_sync(WsHeader *hdr, unsigned long long target,
                                          uint64_t deadline, int *flag, bool publish_cta) {
    __syncthreads();
    if (threadIdx.x == 0) {
        // the release add publishes this thread's writes; other threads'
        // writes (ordered before it by the CTA barrier) get a full fence
        if (publish_cta) __threadfence();
        red_release_add_u64(&hdr->bar_arrivals, 1ull);
        bool ok = true;
        while (ld_acquire_u64(&hdr->bar_arrivals) < target) {
            if (global_timer_ns() > deadline) {
                ok = false;
                break;
            }
            __nanosleep(20);
        }
        *flag = ok ? 0 : 1;
    }
    __syncthreads();
    return *flag == 0;
}


template <int NSB_H, int NSB_I>
__global__ void __launch_bounds__(kThreads, 1) decode_fused_kernel(const Params p) {
    extern __shared__ __align__(128) uint8_t smem[];
    unsigned long long *base_sh = reinterpret_cast<unsigned long long *>(smem);
    int *sel_e = reinterpret_cast<int *>(base_sh + 1);
    float *sel_w = reinterpret_cast<float *>(sel_e + 32);
    int *flags = reinterpret_cast<int *>(sel_w + 32);  // [0] barrier result, [1] abort
    float *red = reinterpret_cast<float *>(flags + 4); // partial sums, then logits + ranks (2*kMaxE)
    float *vec = reinterpret_cast<float *>(smem + kHeadBytes);
    const int H = p.H, E = p.E, k = p.k, I = p.I;
    const int vec_pad = max(padded_len(H), k * padded_len(I));
    float *vsum = vec + vec_pad;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint64_t deadline = global_timer_ns() + p.wait_ns;
    const unsigned nblk = gridDim.x;
    const int nsb_h = H / kQK, nsb_i = I / kQK;
    const int row_gu = nsb_h * kBlockBytes, row_dn = nsb_i * kBlockBytes;
    const size_t mat_gu = size_t(I) * row_gu, mat_dn = size_t(H) * row_dn;
    const int nbw = p.nbw;
    uint8_t *ring = smem + p.ring_off + size_t(warp) * nbw * p.slot_bytes;

    if (threadIdx.x == 0) {
        TL_STAMP(p, 0);
        // this call's barrier rounds: every call adds 2 arrivals per CTA, and
        // fewer than 2*nblk arrivals of this call can precede this read
        const unsigned long long c0 = ld_acquire_u64(&p.hdr->bar_arrivals);
        *base_sh = c0 - c0 % (2ull * nblk);
        flags[1] = 0;
    }
    // ---------------- 1. router logits (a share per CTA), grid barrier.
    // The CTA's first logit is computed while x is staged: x and the router
    // row are requested together, so their latencies overlap.
    const uint64_t pol_last = l2_policy_evict_last();
    {
        const int e = blockIdx.x;
        const bool logit = p.router_on && e < E;
        const float *wr = p.Wr + size_t(logit ? e : 0) * H;
        float a = 0.f;
        for (int i = threadIdx.x; i < (H >> 2); i += kThreads) {
            const float4 x4 = __ldg(reinterpret_cast<const float4 *>(p.x) + i);
            if (logit) {
                const float4 w4 = ldg_f4_policy(wr + 4 * i, pol_last);
                a = fmaf(w4.x, x4.x, a);
                a = fmaf(w4.y, x4.y, a);
                a = fmaf(w4.z, x4.z, a);
                a = fmaf(w4.w, x4.w, a);
            }
            *reinterpret_cast<float4 *>(vec + padded(4 * i)) = x4;
        }
        a = warp_sum(a);
        if (lane == 0) red[warp] = a;
        __syncthreads();
        if (logit && threadIdx.x == 0) {
            float sum = 0.f;
            for (int w = 0; w < kWarps; ++w) sum += red[w];
            p.logits[e] = sum + (p.bias ? p.bias[e] : 0.f);
        }
        run_sums32(vec, vsum, H >> 5, H >> 5, 0);
        __syncthreads();
    }
    const unsigned long long base = *base_sh;
    if (threadIdx.x == 0) TL_STAMP(p, 1);

    if (p.router_on) {
        for (int e = blockIdx.x + nblk; e < E; e += nblk) {
            const float *wr = p.Wr + size_t(e) * H;
            float a = 0.f;
            for (int i = threadIdx.x; i < (H >> 2); i += kThreads) {
                const float4 w4 = ldg_f4_policy(wr + 4 * i, pol_last);
                const float4 x4 = *reinterpret_cast<const float4 *>(vec + padded(4 * i));
                a = fmaf(w4.x, x4.x, a);
                a = fmaf(w4.y, x4.y, a);
                a = fmaf(w4.z, x4.z, a);
                a = fmaf(w4.w, x4.w, a);
            }
            a = warp_sum(a);
            if (lane == 0) red[warp] = a;
            __syncthreads();
            if (threadIdx.x == 0) {
                float s = 0.f;
                for (int w = 0; w < kWarps; ++w) s += red[w];
                p.logits[e] = s + (p.bias ? p.bias[e] : 0.f);
            }
            __syncthreads();
        }
        if (threadIdx.x == 0) TL_STAMP(p, 2);
        if (!grid_sync(p.hdr, base + nblk + p.withhold, deadline, flags, false)) {
            if (threadIdx.x == 0) record_status(p.hdr, MOE_ERR_TIMEOUT, 1);
            cp_async_wait_all();
            return;  // no output written
        }
    } else if (threadIdx.x == 0) {
        red_release_add_u64(&p.hdr->bar_arrivals, 1ull);  // keep 2 arrivals per call
    }
    if (threadIdx.x == 0) TL_STAMP(p, 8);

    // ---------------- 2. top-k + renormalise, by rank: every CTA ranks the E
    // logits in the order (value descending, index ascending); the logit of
    // rank j < k is slot j.  G threads share the comparisons of one logit.
    if (p.router_on) {
        float *lsm = red;                     // E logits (red is free again)
        int *rank = reinterpret_cast<int *>(lsm + kMaxE);
        for (int e = threadIdx.x; e < E; e += kThreads) {
            float v = __ldcg(p.logits + e);
            lsm[e] = (v == v) ? v : -INFINITY;   // a NaN never ranks first
            rank[e] = 0;
        }
        __syncthreads();
        const int G = max(1, kThreads / E);      // threads per logit
        const int per = (E + G - 1) / G;         // comparisons per thread
        for (int t = threadIdx.x; t < E * G; t += kThreads) {
            const int e = t / G, part = t % G;
            const float ve = lsm[e];
            int cnt = 0;
            const int b0 = part * per, b1 = min(E, b0 + per);
            for (int o = b0; o < b1; ++o) {
                const float vo = lsm[o];
                cnt += (vo > ve || (vo == ve && o < e)) ? 1 : 0;
            }
            if (cnt) atomicAdd(rank + e, cnt);
        }
        __syncthreads();
        for (int e = threadIdx.x; e < E; e += kThreads) {
            const int r = rank[e];
            if (r < k) sel_e[r] = e;
        }
        __syncthreads();
        if (warp == 0) {
            const float l = (lane < k) ? lsm[sel_e[lane]] : 0.f;
            const float l0 = lsm[sel_e[0]];
            const float ex = (lane < k) ? expf(l - l0) : 0.f;
            const float z = warp_sum(ex);
            if (lane < k) {
                sel_w[lane] = ex / z;
                if (blockIdx.x == 0) {
                    p.idx_out[lane] = sel_e[lane];
                    p.w_out[lane] = ex / z;
                }
            }
        }
    } else if (warp == 0 && lane < k) {
        const int e = p.idx_in[lane];
        sel_e[lane] = e;
        sel_w[lane] = p.w_in[lane];
        if (blockIdx.x == 0 && (e < 0 || e >= E)) record_status(p.hdr, MOE_ERR_EXPERT_RANGE, e);
    }
    __syncthreads();
    if (threadIdx.x == 0) TL_STAMP(p, 3);

    // ---------------- 3. gate/up rows: per-warp cp.async rings
    const int U = k * I;
    const int u0 = int((long long)U * blockIdx.x / nblk);
    const int u1 = int((long long)U * (blockIdx.x + 1) / nblk);
    const int r0 = int((long long)H * blockIdx.x / nblk);
    const int r1 = int((long long)H * (blockIdx.x + 1) / nblk);
    const int R = r1 - r0;
    const int n_gu = u1 - u0;
    const int n_mine = n_gu > warp ? (n_gu - warp + kWarps - 1) / kWarps : 0;  // rows warp+16i
    const uint64_t pol = l2_policy_evict_first();
    const int n16_gu = row_gu >> 4, n16_dn = row_dn >> 4;

    // issue the copies of this warp's i-th gate/up row pair into its ring slot
    auto issue_gu = [&](int i) {
        const int u = u0 + warp + kWarps * i, j = u / I, r = u % I;
        const int e = sel_e[j];
        uint8_t *dst = ring + (i % nbw) * p.slot_bytes;
        if (e >= 0 && e < E) {
            const uint8_t *g = p.gate + e * mat_gu + size_t(r) * row_gu;
            const uint8_t *uu = p.up + e * mat_gu + size_t(r) * row_gu;
            for (int c = lane; c < 2 * n16_gu; c += 32) {
                const uint8_t *src = c < n16_gu ? g + 16 * c : uu + 16 * (c - n16_gu);
                cp_async_16(dst + 16 * c, src, pol);
            }
        }
        cp_async_commit();
    };
    // issue the copies of this warp's i-th down row (all k experts) into a ring slot
    auto issue_dn = [&](int i, int slot) {
        const int r = r0 + warp + kWarps * i;
        uint8_t *dst = ring + slot * p.slot_bytes;
        for (int c = lane; c < k * n16_dn; c += 32) {
            const int j = c / n16_dn, w16 = c % n16_dn;
            const int e = sel_e[j];
            if (e >= 0 && e < E)
                cp_async_16(dst + 16 * c, p.down + e * mat_dn + size_t(r) * row_dn + 16 * w16, pol);
        }
        cp_async_commit();
    };

    const int first = min(nbw, n_mine);
    for (int i = 0; i < first; ++i) issue_gu(i);
    uint8_t *dbuf = smem + p.down_off;
    if (p.down_resident) {
        // the CTA's R output rows of all k experts: k contiguous ranges
        const int per_j = R * n16_dn;
        for (int c = threadIdx.x; c < k * per_j; c += kThreads) {
            const int j = c / per_j, w16 = c % per_j;
            const int e = sel_e[j];
            if (e >= 0 && e < E)
                cp_async_16(dbuf + 16 * c, p.down + e * mat_dn + size_t(r0) * row_dn + 16 * w16, pol);
        }
        cp_async_commit();  // one group after the first gate/up rows
    }

    for (int i = 0; i < n_mine; ++i) {
        const int slot = i % nbw;
        // groups committed after row i: the rows issued beyond it, plus the
        // down prefetch when it went in after the first rows
        const int later = min(nbw - 1, n_mine - 1 - i) + ((p.down_resident && i < first) ? 1 : 0);
        cp_async_wait_pending(later);
        __syncwarp();
        if (threadIdx.x == 0 && i == 0) TL_STAMP(p, 9);
        const int u = u0 + warp + kWarps * i, j = u / I, r = u % I;
        const int e = sel_e[j];
        if (e >= 0 && e < E) {
            const uint8_t *src = ring + slot * p.slot_bytes;
            const float g = warp_sum(row_dot_pairs<NSB_H>(src, nsb_h, vec, vsum, lane));
            const float uu = warp_sum(row_dot_pairs<NSB_H>(src + row_gu, nsb_h, vec, vsum, lane));
            if (lane == 0) p.hbuf[size_t(j) * I + r] = silu_mul(g, uu);
        }
        __syncwarp();
        if (i + nbw < n_mine) issue_gu(i + nbw);
    }
    if (threadIdx.x == 0) TL_STAMP(p, 4);

    // ---------------- 4. h complete everywhere -> down rows + combine
    if (!grid_sync(p.hdr, base + 2ull * nblk + p.withhold, deadline, flags, true)) {
        if (threadIdx.x == 0) record_status(p.hdr, MOE_ERR_TIMEOUT, 4);
        flags[1] = 1;
    }
    __syncthreads();
    if (threadIdx.x == 0) TL_STAMP(p, 5);
    if (flags[1] == 0) {
        const int ip = padded_len(I);
        for (int q = threadIdx.x; q < (k * I) >> 5; q += kThreads) {  // one 32-float run each
            const int j = (32 * q) / I, c = (32 * q) % I;
            const float4 *src = reinterpret_cast<const float4 *>(p.hbuf) + 8 * q;
            float4 v[8];
#pragma unroll
            for (int b = 0; b < 8; ++b) v[b] = __ldcg(src + b);
            float *dst = vec + j * ip + padded(c);
            float s0 = 0.f, s1 = 0.f;
#pragma unroll
            for (int b = 0; b < 8; b += 2) {
                *reinterpret_cast<float4 *>(dst + 4 * b) = v[b];
                *reinterpret_cast<float4 *>(dst + 4 * b + 4) = v[b + 1];
                s0 += (v[b].x + v[b].y) + (v[b].z + v[b].w);
                s1 += (v[b + 1].x + v[b + 1].y) + (v[b + 1].z + v[b + 1].w);
            }
            vsum[q] = s0 + s1;
        }
        __syncthreads();
        if (threadIdx.x == 0) TL_STAMP(p, 6);

        const int n_rows = R > warp ? (R - warp + kWarps - 1) / kWarps : 0;  // rows warp+16i
        if (p.down_resident) {
            cp_async_wait_all();  // this thread's share of the prefetch
            __syncthreads();      // everyone's share
        }
        if (threadIdx.x == 0) TL_STAMP(p, 10);
        const int first_dn = p.down_resident ? 0 : min(nbw, n_rows);
        for (int i = 0; i < first_dn; ++i) issue_dn(i, i % nbw);
        for (int i = 0; i < n_rows; ++i) {
            const int rr = warp + kWarps * i;  // row inside the CTA's share
            const uint8_t *src;
            size_t jstride;
            if (p.down_resident) {
                src = dbuf + size_t(rr) * row_dn;
                jstride = size_t(R) * row_dn;
            } else {
                cp_async_wait_pending(min(nbw - 1, n_rows - 1 - i));
                __syncwarp();
                src = ring + (i % nbw) * p.slot_bytes;
                jstride = row_dn;
            }
            // k experts x nsb_i blocks x 8 chunks, spread over the 32 lanes in a
            // fixed order; each chunk's partial dot is weighted by its slot's
            // router weight, then one warp reduction gives y (deterministic)
            float yacc = 0.f;
            const int per_j = (NSB_I > 0 ? NSB_I : nsb_i) * 4;   // (block, pair) units per slot
            const int nunits = k * per_j;
            for (int t = lane; t < nunits; t += 32) {
                const int j = t / per_j, rem = t - j * per_j;
                const int sb = rem >> 2, c = rem & 3;
                const int e = sel_e[j];
                if (e < 0 || e >= E) continue;
                const float part = pair_dot(src + j * jstride + sb * kBlockBytes, c,
                                            vec + j * ip + padded(sb * kQK + 64 * c),
                                            vsum + j * (I >> 5) + sb * 8 + 2 * c);
                yacc = fmaf(sel_w[j], part, yacc);
            }
            yacc = warp_sum(yacc);
            if (lane == 0) p.y[r0 + rr] = yacc;
            __syncwarp();
            if (!p.down_resident && i + nbw < n_rows) issue_dn(i + nbw, (i + nbw) % nbw);
        }
    }
    // every copy this thread issued must land before the CTA's shared memory goes away
    cp_async_wait_all();
    if (threadIdx.x == 0) TL_STAMP(p, 7);
}

}  // namespace fused

namespace {

struct FusedConfig {
    int nbw = 0, slot_bytes = 0, ring_off = 0, down_resident = 0, down_off = 0, smem = 0;
};

bool fused_config(int H, int E, int k, int I, int nblk, int max_smem, FusedConfig &c) {
    using namespace fused;
    if (E > kMaxE || k > kMaxK || nblk < 1) return false;
    const int row_gu = (H / kQK) * kBlockBytes, row_dn = (I / kQK) * kBlockBytes;
    const int vec_pad = std::max(padded_len(H), k * padded_len(I));
    const int vec_sum = std::max(H, k * I) / 16;
    const int vec_end = int(align256(size_t(kHeadBytes) + sizeof(float) * size_t(vec_pad + vec_sum)));
    const int rmax = (H + nblk - 1) / nblk;
    const int down_bytes = int(align256(size_t(k) * rmax * row_dn));
    // A: the CTA's down rows resident, rings hold gate/up row pairs
    int slot = (2 * row_gu + 127) / 128 * 128;
    int nbw = (max_smem - vec_end - down_bytes) / (kWarps * slot);
    // Only shapes whose down rows fit resident take this kernel.  The variant
    // that streams down rows through the per-warp rings after the second
    // barrier (needed by the Qwen3-235B-A22B shape) raised an illegal
    // instruction on GB300 and is not launched; those shapes run the
    // multi-kernel path.
    if (nbw < 2) return false;
    c.down_resident = 1;
    c.down_off = vec_end;
    c.ring_off = vec_end + down_bytes;
    nbw = std::min(nbw, kMaxNbw);
    if (nbw < 1) return false;
    c.nbw = nbw;
    c.slot_bytes = slot;
    c.smem = c.ring_off + kWarps * nbw * slot;
    return c.smem <= max_smem;
}

template <int A, int B>
void *kernel_ptr() {
    return reinterpret_cast<void *>(&fused::decode_fused_kernel<A, B>);
}

void *pick_kernel(int H, int I) {
    const int a = H / kQK, b = I / kQK;
    if (a == 8 && b == 3) return kernel_ptr<8, 3>();
    if (a == 1 && b == 1) return kernel_ptr<1, 1>();
    if (a == 8 && b == 4) return kernel_ptr<8, 4>();
    return kernel_ptr<0, 0>();
}

int g_fused_max_smem[64];
int g_fused_blocks[64];

}  // namespace

cudaError_t init_decode_fused(int dev, int num_sms) {
    int optin = 0;
    cudaError_t err = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (err != cudaSuccess) return err;
    g_fused_max_smem[dev] = optin;
    void *ks[] = {kernel_ptr<8, 3>(), kernel_ptr<1, 1>(), kernel_ptr<8, 4>(), kernel_ptr<0, 0>()};
    for (void *kp : ks) {
        err = cudaFuncSetAttribute(kp, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
        if (err != cudaSuccess) return err;
    }
    g_fused_blocks[dev] = num_sms;
    return cudaSuccess;
}

bool decode_fused_supported(int dev, int T, int H, int E, int k, int I) {
    if (T != 1) return false;
    FusedConfig c;
    return fused_config(H, E, k, I, g_fused_blocks[dev], g_fused_max_smem[dev], c);
}

cudaError_t launch_decode_fused(int dev, const float *x, const float *Wr, const float *bias,
                                const int32_t *idx_in, const float *w_in, int32_t *idx_out,
                                float *w_out, const uint8_t *gate, const uint8_t *up,
                                const uint8_t *down, int H, int E, int k, int I, float *y,
                                float *logits, float *hbuf, WsHeader *hdr, int withhold,
                                unsigned long long wait_ns, cudaStream_t s) {
    FusedConfig c;
    if (!fused_config(H, E, k, I, g_fused_blocks[dev], g_fused_max_smem[dev], c))
        return cudaErrorInvalidValue;
    fused::Params p;
    p.x = x;
    p.Wr = Wr;
    p.bias = bias;
    p.idx_in = idx_in;
    p.w_in = w_in;
    p.idx_out = idx_out;
    p.w_out = w_out;
    p.gate = gate;
    p.up = up;
    p.down = down;
    p.y = y;
    p.logits = logits;
    p.hbuf = hbuf;
    p.hdr = hdr;
    p.H = H;
    p.E = E;
    p.k = k;
    p.I = I;
    p.router_on = (Wr != nullptr) ? 1 : 0;
    p.nbw = c.nbw;
    p.slot_bytes = c.slot_bytes;
    p.ring_off = c.ring_off;
    p.down_resident = c.down_resident;
    p.down_off = c.down_off;
    p.withhold = withhold;
    p.wait_ns = wait_ns;
    p.timeline = reinterpret_cast<unsigned long long *>(hbuf + size_t(k) * I);

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(g_fused_blocks[dev]);
    cfg.blockDim = dim3(fused::kThreads);
    cfg.dynamicSmemBytes = c.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void *args[] = {&p};
    return cudaLaunchKernelExC(&cfg, pick_kernel(H, I), args);
}

}  // namespace moeq4k
