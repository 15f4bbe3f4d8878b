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
// Design (one CTA per SM, cooperative launch so every CTA is resident):
//  1. Every CTA stages x in shared memory and computes a share of the E
//     router logits (Wr read with an L2 evict-last policy: it is re-read by
//     every token, unlike the expert bytes).
//  2. Grid barrier; every CTA reads the E logits and runs the same top-k and
//     renormalisation, so all CTAs know the k experts without a broadcast.
//  3. A producer warp streams this CTA's share of the selected experts' Q4_K
//     rows into a ring of shared-memory slots with 1-D bulk copies (TMA
//     engine, mbarrier completion, L2 evict-first policy): first the
//     gate/up row pairs (slot j, row r), then the down rows of the CTA's
//     output rows for all k experts.  At T=1 the share of the Qwen3-30B-A3B
//     shape (~140 KB) fits in the ring entirely, so every byte is requested
//     up front and HBM sees the whole 21 MB at once.
//  4. Consumer warps decode rows as they land (nibbles and 6-bit scales in
//     registers, fp32 FMA against x in shared memory) and write
//     h = SiLU(g) * u to the workspace.
//  5. Grid barrier; each CTA stages h of all k slots, then for each of its
//     output rows computes o_j = Wd[e_j][row] . h_j for j = 0..k-1 and
//     y = sum_j w_j o_j in slot order, so the combine is deterministic and
//     needs no atomics.
// Every wait (mbarrier, grid barrier) is bounded by a global-timer deadline;
// on expiry the kernel records MOE_ERR_TIMEOUT and returns after draining
// its own copies.
#include <algorithm>

#include "async_copy.cuh"
#include "common.cuh"
#include "kernels.cuh"

namespace moeq4k {
namespace fused {

constexpr int kConsWarps = 16;
constexpr int kConsThreads = kConsWarps * 32;
constexpr int kThreads = kConsThreads + 32;  // + one producer warp
constexpr int kMaxSlots = 64;
constexpr int kHeadBytes = 2048;             // barriers + small arrays

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
    int nslots, slot_bytes, ring_off;
    int withhold;                 // test hook: extra arrivals the grid barrier waits for
    unsigned long long wait_ns;   // bound of every wait
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
// dotted with the padded vector `vec` (run sums in `vsum`).  Lane L takes
// code chunk L%8 of blocks L/8, L/8+4, ...
template <int NSB>
__device__ __forceinline__ float row_lane_dot(const uint8_t *row, int nsb_rt, const float *vec,
                                              const float *vsum, int lane) {
    const int nsb = NSB > 0 ? NSB : nsb_rt;
    const int cq = lane & 7, c = cq >> 1, hf = cq & 1;
    // sub-blocks 2c and 2c+1: shifts into the packed scale words
    const bool upper = c >= 2;
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

// Stage `n` floats from global `src` (row-major, 16-byte aligned) into the
// padded shared vector and its 16-element run sums; consumer threads only.
__device__ __forceinline__ void stage_vector(const float *src, int n, bool coherent, float *vec,
                                             float *vsum) {
    for (int i = threadIdx.x; i < (n >> 2); i += kConsThreads) {
        const float4 v = coherent ? __ldcg(reinterpret_cast<const float4 *>(src) + i)
                                  : __ldg(reinterpret_cast<const float4 *>(src) + i);
        *reinterpret_cast<float4 *>(vec + padded(4 * i)) = v;
    }
    named_bar_sync(1, kConsThreads);
    for (int r = threadIdx.x; r < (n >> 4); r += kConsThreads) {
        const float *v = vec + padded(16 * r);
        float s = 0.f;
#pragma unroll
        for (int b = 0; b < 16; ++b) s += v[b];
        vsum[r] = s;
    }
    named_bar_sync(1, kConsThreads);
}

// Grid barrier over the consumer threads of every CTA (sense by generation
// counter, self-resetting so it works across graph replays).  Returns false
// if the wait ran past the deadline.
__device__ __forceinline__ bool grid_barrier(WsHeader *hdr, unsigned expected, uint64_t deadline,
                                             int *flag) {
    named_bar_sync(1, kConsThreads);
    if (threadIdx.x == 0) {
        volatile unsigned *genp = &hdr->bar_gen;
        const unsigned g = *genp;
        __threadfence();
        const unsigned prev = atomicAdd(&hdr->bar_count, 1u);
        bool ok = true;
        if (prev == expected - 1) {
            atomicExch(&hdr->bar_count, 0u);
            __threadfence();
            atomicAdd(&hdr->bar_gen, 1u);
        } else {
            while (*genp == g) {
                if (global_timer_ns() > deadline) {
                    ok = false;
                    break;
                }
                __nanosleep(32);
            }
        }
        __threadfence();
        *flag = ok ? 0 : 1;
    }
    named_bar_sync(1, kConsThreads);
    return *flag == 0;
}

__device__ __forceinline__ bool better(float v, int i, float bv, int bi) {
    return v > bv || (v == bv && i < bi);
}

template <int NSB_H, int NSB_I>
__device__ __forceinline__ void consumer_phases(const Params &p, uint64_t *full, uint64_t *empty,
                                                const int *sel_e, const float *sel_w, int *flags,
                                                float *vec, float *vsum, uint8_t *ring,
                                                uint64_t deadline, int u0, int n_gu, int r0,
                                                int F) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int E = p.E, k = p.k, I = p.I, NS = p.nslots;
    const unsigned nblk = gridDim.x;
    const int nsb_h = p.H / kQK, nsb_i = I / kQK;
    const int row_gu = nsb_h * kBlockBytes, row_dn = nsb_i * kBlockBytes;
    // consumers: gate/up row pairs
    bool alive = true;
    for (int f = warp; f < n_gu; f += kConsWarps) {
        const int slot = f % NS;
        if (!mbar_wait(full + slot, (f / NS) & 1, deadline)) {
            if (lane == 0) record_status(p.hdr, MOE_ERR_TIMEOUT, 3);
            alive = false;
            break;
        }
        const int u = u0 + f, j = u / I, r = u % I;
        const int e = sel_e[j];
        if (e >= 0 && e < E) {
            const uint8_t *src = ring + size_t(slot) * p.slot_bytes;
            const float g = warp_sum(row_lane_dot<NSB_H>(src, nsb_h, vec, vsum, lane));
            const float uu = warp_sum(row_lane_dot<NSB_H>(src + row_gu, nsb_h, vec, vsum, lane));
            if (lane == 0) p.hbuf[size_t(j) * I + r] = silu_mul(g, uu);
        }
        __syncwarp();
        fence_proxy_async_smem();
        if (lane == 0) mbar_arrive(empty + slot);
    }
    if (!alive) flags[1] = 1;

    // h of every slot must be complete before the down rows
    if (!grid_barrier(p.hdr, nblk + p.withhold, deadline, flags)) {
        if (threadIdx.x == 0) record_status(p.hdr, MOE_ERR_TIMEOUT, 4);
        flags[1] = 1;
    }
    const bool run = flags[1] == 0;
    if (run) {
        // h for all k slots -> padded vector (slot j at j * padded_len(I))
        const int ip = padded_len(I);
        for (int i = threadIdx.x; i < (k * I) >> 2; i += kConsThreads) {
            const int j = (4 * i) / I, c = (4 * i) % I;
            const float4 v = __ldcg(reinterpret_cast<const float4 *>(p.hbuf) + i);
            *reinterpret_cast<float4 *>(vec + j * ip + padded(c)) = v;
        }
        named_bar_sync(1, kConsThreads);
        for (int q = threadIdx.x; q < (k * I) >> 4; q += kConsThreads) {
            const int j = (16 * q) / I, c = (16 * q) % I;
            const float *v = vec + j * ip + padded(c);
            float s = 0.f;
#pragma unroll
            for (int b = 0; b < 16; ++b) s += v[b];
            vsum[q] = s;
        }
        named_bar_sync(1, kConsThreads);
    }

    // down rows + slot-ordered combine
    for (int f = n_gu + warp; f < F; f += kConsWarps) {
        const int slot = f % NS;
        if (!mbar_wait(full + slot, (f / NS) & 1, deadline)) {
            if (lane == 0) record_status(p.hdr, MOE_ERR_TIMEOUT, 5);
            break;
        }
        if (run) {
            const int r = r0 + (f - n_gu);
            const uint8_t *src = ring + size_t(slot) * p.slot_bytes;
            const int ip = padded_len(I);
            float yacc = 0.f;
            for (int j = 0; j < k; ++j) {
                const int e = sel_e[j];
                if (e < 0 || e >= E) continue;
                const float o = warp_sum(row_lane_dot<NSB_I>(src + j * row_dn, nsb_i,
                                                              vec + j * ip, vsum + j * (I >> 4),
                                                              lane));
                yacc = fmaf(sel_w[j], o, yacc);
            }
            if (lane == 0) p.y[r] = yacc;
        }
        __syncwarp();
        fence_proxy_async_smem();
        if (lane == 0) mbar_arrive(empty + slot);
    }
}

template <int NSB_H, int NSB_I>
__global__ void __launch_bounds__(kThreads, 1) decode_fused_kernel(const Params p) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *empty = full + kMaxSlots;
    int *sel_e = reinterpret_cast<int *>(empty + kMaxSlots);
    float *sel_w = reinterpret_cast<float *>(sel_e + 32);
    float *red = sel_w + 32;
    int *flags = reinterpret_cast<int *>(red + 32);  // [0] barrier result, [1] abort, [2] fills issued
    float *vec = reinterpret_cast<float *>(smem + kHeadBytes);
    const int H = p.H, E = p.E, k = p.k, I = p.I;
    const int vec_pad = max(padded_len(H), k * padded_len(I));
    float *vsum = vec + vec_pad;
    uint8_t *ring = smem + p.ring_off;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool producer = warp == kConsWarps;
    const uint64_t deadline = global_timer_ns() + p.wait_ns;
    const unsigned nblk = gridDim.x;
    const int nsb_h = H / kQK, nsb_i = I / kQK;
    const int row_gu = nsb_h * kBlockBytes, row_dn = nsb_i * kBlockBytes;
    const size_t mat_gu = size_t(I) * row_gu, mat_dn = size_t(H) * row_dn;

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.nslots; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
        }
        flags[1] = 0;
        flags[2] = 0;
        fence_mbar_init();
    }
    // x -> padded shared vector (consumers); the producer waits below
    if (!producer) stage_vector(p.x, H, false, vec, vsum);
    __syncthreads();

    // ---------------- 1. router logits (a share per CTA), grid barrier
    if (p.router_on) {
        if (!producer) {
            const uint64_t pol = l2_policy_evict_last();
            for (int e = blockIdx.x; e < E; e += nblk) {
                const float *wr = p.Wr + size_t(e) * H;
                float a = 0.f;
                for (int i = threadIdx.x; i < (H >> 2); i += kConsThreads) {
                    const float4 w4 = ldg_f4_policy(wr + 4 * i, pol);
                    const float4 x4 = *reinterpret_cast<const float4 *>(vec + padded(4 * i));
                    a = fmaf(w4.x, x4.x, a);
                    a = fmaf(w4.y, x4.y, a);
                    a = fmaf(w4.z, x4.z, a);
                    a = fmaf(w4.w, x4.w, a);
                }
                a = warp_sum(a);
                if (lane == 0) red[warp] = a;
                named_bar_sync(1, kConsThreads);
                if (threadIdx.x == 0) {
                    float s = 0.f;
                    for (int w = 0; w < kConsWarps; ++w) s += red[w];
                    p.logits[e] = s + (p.bias ? p.bias[e] : 0.f);
                }
                named_bar_sync(1, kConsThreads);
            }
            if (!grid_barrier(p.hdr, nblk + p.withhold, deadline, flags)) {
                if (threadIdx.x == 0) {
                    record_status(p.hdr, MOE_ERR_TIMEOUT, 1);
                    flags[1] = 1;
                }
            }
        }
        __syncthreads();
        if (flags[1]) return;  // nothing issued yet: safe to leave
    }

    // ---------------- 2. top-k + renormalise (warp 0 of every CTA)
    if (warp == 0) {
        if (p.router_on) {
            constexpr int kPer = kMaxE / 32;
            float v[kPer];
            bool taken[kPer];
#pragma unroll
            for (int s = 0; s < kPer; ++s) {
                const int e = lane + 32 * s;
                v[s] = (e < E) ? __ldcg(p.logits + e) : -INFINITY;
                taken[s] = e >= E;
            }
            float sel_v = 0.f, vmax = 0.f;
            int sel_i = 0;
            for (int j = 0; j < k; ++j) {
                float bv = -INFINITY;
                int bi = 0x7fffffff;
#pragma unroll
                for (int s = 0; s < kPer; ++s) {
                    const int e = lane + 32 * s;
                    if (!taken[s] && better(v[s], e, bv, bi)) {
                        bv = v[s];
                        bi = e;
                    }
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
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
            const float ex = (lane < k) ? expf(sel_v - vmax) : 0.f;
            const float z = warp_sum(ex);
            if (lane < k) {
                sel_e[lane] = sel_i;
                sel_w[lane] = ex / z;
                if (blockIdx.x == 0) {
                    p.idx_out[lane] = sel_i;
                    p.w_out[lane] = ex / z;
                }
            }
        } else if (lane < k) {
            const int e = p.idx_in[lane];
            sel_e[lane] = e;
            sel_w[lane] = p.w_in[lane];
            if (blockIdx.x == 0 && (e < 0 || e >= E)) record_status(p.hdr, MOE_ERR_EXPERT_RANGE, e);
        }
    }
    __syncthreads();

    // ---------------- 3/4/5. streamed expert rows
    const int U = k * I;                                   // gate/up row pairs
    const int u0 = int((long long)U * blockIdx.x / nblk);
    const int u1 = int((long long)U * (blockIdx.x + 1) / nblk);
    const int r0 = int((long long)H * blockIdx.x / nblk);
    const int r1 = int((long long)H * (blockIdx.x + 1) / nblk);
    const int n_gu = u1 - u0, n_dn = r1 - r0;
    const int F = n_gu + n_dn;
    const int NS = p.nslots;

    if (producer) {
        if (lane == 0) {
            const uint64_t pol = l2_policy_evict_first();
            int f = 0;
            for (; f < F; ++f) {
                const int slot = f % NS;
                if (f >= NS) {
                    if (!mbar_wait(empty + slot, ((f / NS) - 1) & 1, deadline)) {
                        record_status(p.hdr, MOE_ERR_TIMEOUT, 2);
                        flags[1] = 1;
                        break;
                    }
                }
                uint8_t *dst = ring + size_t(slot) * p.slot_bytes;
                if (f < n_gu) {
                    const int u = u0 + f, j = u / I, r = u % I;
                    const int e = sel_e[j];
                    if (e >= 0 && e < E) {
                        mbar_arrive_expect_tx(full + slot, 2 * row_gu);
                        bulk_copy_g2s(dst, p.gate + e * mat_gu + size_t(r) * row_gu, row_gu,
                                      full + slot, pol);
                        bulk_copy_g2s(dst + row_gu, p.up + e * mat_gu + size_t(r) * row_gu, row_gu,
                                      full + slot, pol);
                    } else {
                        mbar_arrive(full + slot);
                    }
                } else {
                    const int r = r0 + (f - n_gu);
                    uint32_t bytes = 0;
                    for (int j = 0; j < k; ++j) {
                        const int e = sel_e[j];
                        if (e >= 0 && e < E) bytes += row_dn;
                    }
                    if (bytes) {
                        mbar_arrive_expect_tx(full + slot, bytes);
                        for (int j = 0; j < k; ++j) {
                            const int e = sel_e[j];
                            if (e >= 0 && e < E)
                                bulk_copy_g2s(dst + j * row_dn,
                                              p.down + e * mat_dn + size_t(r) * row_dn, row_dn,
                                              full + slot, pol);
                        }
                    } else {
                        mbar_arrive(full + slot);
                    }
                }
            }
            flags[2] = f;
        }
    } else {
        consumer_phases<NSB_H, NSB_I>(p, full, empty, sel_e, sel_w, flags, vec, vsum, ring,
                                      deadline, u0, n_gu, r0, F);
    }
    __syncthreads();
    // After a time-out some issued fills may never have been waited for:
    // drain them (bounded) so no bulk copy lands after the CTA has exited.
    if (threadIdx.x == 0 && flags[1]) {
        const int issued = flags[2];
        const uint64_t dl = global_timer_ns() + p.wait_ns;
        for (int f = max(0, issued - NS); f < issued; ++f) mbar_wait(full + f % NS, (f / NS) & 1, dl);
    }
}

}  // namespace fused

namespace {

struct FusedConfig {
    int nslots = 0, slot_bytes = 0, ring_off = 0, smem = 0;
};

bool fused_config(int H, int E, int k, int I, int max_smem, FusedConfig &c) {
    using namespace fused;
    const int row_gu = (H / kQK) * kBlockBytes, row_dn = (I / kQK) * kBlockBytes;
    const int vec_pad = std::max(padded_len(H), k * padded_len(I));
    const int vec_sum = std::max(H, k * I) / 16;
    c.ring_off = int(align256(size_t(kHeadBytes) + sizeof(float) * size_t(vec_pad + vec_sum)));
    c.slot_bytes = int((std::max(2 * row_gu, k * row_dn) + 127) / 128 * 128);
    const int avail = max_smem - c.ring_off;
    c.nslots = std::min(kMaxSlots, avail / c.slot_bytes);
    c.smem = c.ring_off + c.nslots * c.slot_bytes;
    return c.nslots >= 4 && E <= kMaxE && k <= kMaxK;
}

template <int A, int B>
void *kernel_ptr() {
    return reinterpret_cast<void *>(&fused::decode_fused_kernel<A, B>);
}

void *pick_kernel(int H, int I) {
    const int a = H / kQK, b = I / kQK;
    if (a == 8 && b == 3) return kernel_ptr<8, 3>();
    if (a == 16 && b == 6) return kernel_ptr<16, 6>();
    if (a == 1 && b == 1) return kernel_ptr<1, 1>();
    if (a == 8 && b == 4) return kernel_ptr<8, 4>();
    return kernel_ptr<0, 0>();
}

}  // namespace

// Per-device limits for the fused kernel (set by init_decode_fused).
static int g_fused_max_smem[64];
static int g_fused_blocks[64];

cudaError_t init_decode_fused(int dev, int num_sms) {
    int optin = 0;
    cudaError_t err = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (err != cudaSuccess) return err;
    g_fused_max_smem[dev] = optin;
    void *ks[] = {kernel_ptr<8, 3>(), kernel_ptr<16, 6>(), kernel_ptr<1, 1>(), kernel_ptr<8, 4>(),
                  kernel_ptr<0, 0>()};
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
    return fused_config(H, E, k, I, g_fused_max_smem[dev], c);
}

cudaError_t launch_decode_fused(int dev, const float *x, const float *Wr, const float *bias,
                                const int32_t *idx_in, const float *w_in, int32_t *idx_out,
                                float *w_out, const uint8_t *gate, const uint8_t *up,
                                const uint8_t *down, int H, int E, int k, int I, float *y,
                                float *logits, float *hbuf, WsHeader *hdr, int withhold,
                                unsigned long long wait_ns, cudaStream_t s) {
    FusedConfig c;
    if (!fused_config(H, E, k, I, g_fused_max_smem[dev], c)) return cudaErrorInvalidValue;
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
    p.nslots = c.nslots;
    p.slot_bytes = c.slot_bytes;
    p.ring_off = c.ring_off;
    p.withhold = withhold;
    p.wait_ns = wait_ns;

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
