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
//  1. Every CTA stages x in shared memory (applying the pre-FFN RMSNorm when
//     a norm weight is given) and computes a share of the E router logits.
//     Each logit is published as one 64-bit word that also carries the
//     call's tag, so readers need no barrier: they poll the words until
//     every tag is the current one.
//  2. Warp 0 of every CTA polls the E logits while the other warps prepare
//     x for the dots; every CTA then runs the same top-k and
//     renormalisation, so all CTAs know the k experts without a broadcast.
//  3. The k*I gate/up row pairs are split evenly over the CTAs and, inside a
//     CTA, over its warps.  Lane 0 of each warp requests all of the warp's
//     row pairs at once into private shared-memory slots, one 1-D bulk copy
//     per row and one mbarrier per pair; thread 0 requests the CTA's down
//     rows (its share of the H output rows, for all k experts, one bulk
//     copy per slot).  h = SiLU(g) * u is stored to the workspace.
//     (Requesting only a few rows ahead of the compute was measured slower:
//     the stream then falls short of the HBM bandwidth.)
//  4. Each CTA adds itself to a "rows done" counter (release); thread 0
//     waits for the call's full count (acquire), the CTA stages the k*I
//     values of h, and for each of its output rows computes
//     o_j = Wd[e_j][row] . h_j for j = 0..k-1 and y = sum_j w_j o_j in a
//     fixed order: deterministic, no atomics.
// The tag of a call comes from a counter in the workspace header to which
// every CTA adds 1 at its start, so it needs no reset between calls or graph
// replays.  Every wait is bounded by a global-timer deadline; on expiry the
// kernel records MOE_ERR_TIMEOUT, stops computing and waits (bounded) for
// its copies to land before returning.
//
// Arithmetic of the gate/up rows when H = 2048 (8 Q4_K blocks per row): lane
// L always covers the same 64 elements of x (sub-block pair L % 4 of block
// L / 4), so it keeps them in registers in an exact integer form: x / s, with
// s = max|x| / 127 over each 32-element run, is split into three signed
// base-254 digits (x ~= s (a + b/254 + c/254^2), each digit in [-127, 127];
// the digits leave 6.1e-8 of the run's max|x|, the fp32 scalings add a few
// ulps of x: below 2.5e-7 of the run's max|x| in all).  A 4-bit code times a
// digit word is then one dp4a (four exact 8-bit products summed in int32),
// and the fp32 scales of the block are applied once per sub-block; with
// I = 768 or 1024 h takes the same form for the down rows.  Other shapes dot
// fp32 vectors in shared memory.
#include <algorithm>

#include "async_copy.cuh"
#include "common.cuh"
#include "kernels.cuh"
#include "q4k_dot.cuh"

namespace moeq4k {
namespace fused {

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kMaxNbw = 8;         // ring slots per warp
constexpr int kHeadBytes = 6144;   // small shared arrays and barriers (see the kernel's first lines)
constexpr int kStageBatch = 8;     // 128-value chunks of h in flight per warp while staging
constexpr long long kPollPauseCycles = 128;  // pause after a poll round that found a stale word

// Optional phase timeline for profiling builds (-DMOEQ4K_TIMELINE): thread 0
// of each CTA stamps the global timer at phase boundaries into the
// workspace's per-slot activation region, which this path does not use.
#ifdef MOEQ4K_TIMELINE
#define TL_STAMP(p, i)                                                             \
    do {                                                                           \
        if (int(blockIdx.x) * 16 + (i) < (p).timeline_cap)                         \
            (p).timeline[blockIdx.x * 16 + (i)] = global_timer_ns();              \
    } while (0)
#else
#define TL_STAMP(p, i) ((void)0)
#endif

struct Params {
    const float *x, *Wr, *bias;
    const float *norm_w;          // pre-FFN RMSNorm weight [H], or null (x used as is)
    float eps;                    // the norm's epsilon
    OutEpilogue ep;               // residual add and output capture at the y store
    const int32_t *idx_in;
    const float *w_in;
    int32_t *idx_out;
    float *w_out;
    const uint8_t *gate, *up, *down;
    float *y;
    unsigned long long *sync;     // tagged router logits [E]
    float *hbuf;                  // h = SiLU(g) * u of the k slots [k, I]
    WsHeader *hdr;
    int H, E, k, I;
    int router_on;
    int nbw, slot_bytes, ring_off;  // per-warp ring: nbw slots, one per gate/up row pair
    int down_off;                   // the CTA's down rows, prefetched into [down_off, ...)
    int dig_off;                  // x digit planes (3 x H bytes), then H/32 run scales
    int withhold;                 // test hook: CTA 0 publishes nothing
    unsigned long long wait_ns;   // bound of every wait
    unsigned long long *timeline; // profiling builds only
    int timeline_cap;
};

__device__ __forceinline__ unsigned long long tagged(uint32_t tag, float v) {
    return (static_cast<unsigned long long>(tag) << 32) | __float_as_uint(v);
}
__device__ __forceinline__ uint32_t tag_of(unsigned long long w) { return uint32_t(w >> 32); }
__device__ __forceinline__ float value_of(unsigned long long w) {
    return __uint_as_float(uint32_t(w));
}

// Unsigned key with the order of the float: larger value, larger key.
__device__ __forceinline__ uint32_t ordered_key(float v) {
    const uint32_t b = __float_as_uint(v);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
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

// Sum each 32-float run of the padded vector into sum32, one warp per run
// (consecutive words, no bank conflicts; fixed reduction order).
__device__ __forceinline__ void run_sums32(const float *vec, float *sum32, int runs, int warp,
                                           int lane) {
    for (int r = warp; r < runs; r += kWarps) {
        const float s = warp_sum(vec[padded(32 * r + lane)]);
        if (lane == 0) sum32[r] = s;
    }
}

// Busy-wait on the SM clock (no memory traffic) for about `cycles`.
__device__ __forceinline__ void pause_cycles(long long cycles) {
    const long long until = clock64() + cycles;
    while (clock64() < until) {
    }
}

// One thread polls a counter until it reaches `target`; false when `deadline`
// passes.
__device__ __forceinline__ bool await_count(const unsigned long long *c, unsigned long long target,
                                            uint64_t deadline) {
    while (ld_relaxed_u64(c) < target) {
        if (global_timer_ns() > deadline) return false;
    }
    return true;
}

template <int NSB_H, int NSB_I>
__global__ void __launch_bounds__(kThreads, 1) decode_fused_kernel(const Params p) {
    // The integer form of x applies when every lane covers one sub-block pair.
    constexpr bool kDigits = (NSB_H == 8);
    extern __shared__ __align__(128) uint8_t smem[];
    uint32_t *tag_sh = reinterpret_cast<uint32_t *>(smem);
    int *sel_e = reinterpret_cast<int *>(smem + 16);
    float *sel_w = reinterpret_cast<float *>(sel_e + 32);
    int *flags = reinterpret_cast<int *>(sel_w + 32);  // [1] wait timed out, [2] tied ranks
    float *red = reinterpret_cast<float *>(flags + 4); // kWarps partial sums, then kMaxE logits,
                                                       // then kWarps partial sums of squares
    uint32_t *skey = reinterpret_cast<uint32_t *>(smem + 1536);  // kMaxE logit keys
    int *pcnt = reinterpret_cast<int *>(smem + 2560);            // kThreads partial ranks
    // one mbarrier per gate/up row pair of each warp (bytes of its two bulk
    // copies), one for the CTA's down rows
    uint64_t *rbar = reinterpret_cast<uint64_t *>(smem + 4608);  // [kWarps][kMaxNbw]
    uint64_t *dbar = rbar + kWarps * kMaxNbw;
    float *vec = reinterpret_cast<float *>(smem + kHeadBytes);
    const int H = p.H, E = p.E, k = p.k, I = p.I;
    const int vec_pad = max(padded_len(H), k * padded_len(I));
    float *vsum = vec + vec_pad;
    uint8_t *planes = smem + p.dig_off;
    float *xscale = reinterpret_cast<float *>(planes + 3 * H);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Let the next grid in the stream launch now (it waits in its own
    // pdl_wait() until this one has completed), warm L2 with this CTA's
    // router row (a prefetch changes nothing a predecessor could be writing),
    // then wait for the predecessor grid: x may be its output.
    pdl_trigger();
    if (threadIdx.x == 0 && p.router_on && int(blockIdx.x) < p.E)
        bulk_prefetch_l2(p.Wr + size_t(blockIdx.x) * p.H, uint32_t(p.H) * 4u);
    pdl_wait();
    const uint64_t deadline = global_timer_ns() + p.wait_ns;
    const unsigned nblk = gridDim.x;
    const int nsb_h = H / kQK, nsb_i = I / kQK;
    const int row_gu = nsb_h * kBlockBytes, row_dn = nsb_i * kBlockBytes;
    const size_t mat_gu = size_t(I) * row_gu, mat_dn = size_t(H) * row_dn;
    const int nbw = p.nbw;
    uint8_t *ring = smem + p.ring_off + size_t(warp) * nbw * p.slot_bytes;
    const bool publish = !(p.withhold && blockIdx.x == 0);

    // this call's tag: the add returns a value in [n * nblk, (n + 1) * nblk)
    // for the n-th call; the result is only needed once x is staged
    unsigned long long calls0 = 0;
    if (threadIdx.x == 0) {
        TL_STAMP(p, 0);
        calls0 = atomicAdd(&p.hdr->cta_calls, 1ull);
        flags[1] = 0;
        flags[2] = 0;
        for (int i = 0; i < kWarps * kMaxNbw + 1; ++i) mbar_init(rbar + i, 1);
        fence_mbar_init();
    }
    if (threadIdx.x < 32) sel_e[threadIdx.x] = -1;
    // ---------------- 1. router logits (a share per CTA).
    // The CTA's first logit is computed while x is staged: x and the router
    // row are requested together, so their latencies overlap.  With the
    // pre-FFN RMSNorm, the same pass stages x * gamma, sums x^2 and dots
    // x * gamma with the router row; the 1/rms scale (one number per token)
    // is applied to the logit and, in place, to the staged vector.
    {
        const int e = blockIdx.x;
        const bool logit = p.router_on && e < E;
        const bool norm = p.norm_w != nullptr;
        const float *wr = p.Wr + size_t(logit ? e : 0) * H;
        float a = 0.f, ss = 0.f;
        for (int i = threadIdx.x; i < (H >> 2); i += kThreads) {
            float4 x4 = __ldg(reinterpret_cast<const float4 *>(p.x) + i);
            if (norm) {
                ss = fmaf(x4.x, x4.x, ss);
                ss = fmaf(x4.y, x4.y, ss);
                ss = fmaf(x4.z, x4.z, ss);
                ss = fmaf(x4.w, x4.w, ss);
                const float4 g4 = __ldg(reinterpret_cast<const float4 *>(p.norm_w) + i);
                x4 = make_float4(x4.x * g4.x, x4.y * g4.y, x4.z * g4.z, x4.w * g4.w);
            }
            if (logit) {
                const float4 w4 = __ldg(reinterpret_cast<const float4 *>(wr) + i);
                a = fmaf(w4.x, x4.x, a);
                a = fmaf(w4.y, x4.y, a);
                a = fmaf(w4.z, x4.z, a);
                a = fmaf(w4.w, x4.w, a);
            }
            *reinterpret_cast<float4 *>(vec + padded(4 * i)) = x4;
        }
        float *red2 = red + kWarps + kMaxE;
        a = warp_sum(a);
        if (lane == 0) red[warp] = a;
        if (norm) {
            ss = warp_sum(ss);
            if (lane == 0) red2[warp] = ss;
        }
        if (threadIdx.x == 0) *tag_sh = uint32_t(calls0 / nblk) + 1u;
        __syncthreads();
        float inv = 1.f;
        if (norm) {  // every thread forms the same scale from the same sums in the same order
            float s2 = 0.f;
            for (int w = 0; w < kWarps; ++w) s2 += red2[w];
            inv = 1.0f / sqrtf(s2 / float(H) + p.eps);
        }
        if (logit && threadIdx.x == 0) {
            float sum = 0.f;
            for (int w = 0; w < kWarps; ++w) sum += red[w];
            if (norm) sum *= inv;
            sum += p.bias ? p.bias[e] : 0.f;
            if (publish) st_relaxed_u64(p.sync + e, tagged(*tag_sh, sum));
        }
        if (norm) {
            // each thread rescales the elements it staged
            for (int i = threadIdx.x; i < (H >> 2); i += kThreads) {
                float4 *v = reinterpret_cast<float4 *>(vec + padded(4 * i));
                const float4 t4 = *v;
                *v = make_float4(t4.x * inv, t4.y * inv, t4.z * inv, t4.w * inv);
            }
            __syncthreads();
        }
    }
    const uint32_t tag = *tag_sh;
    if (threadIdx.x == 0) TL_STAMP(p, 1);

    if (p.router_on && blockIdx.x + nblk < unsigned(E)) {
        __syncthreads();  // thread 0 is done with `red`
        for (int e = blockIdx.x + nblk; e < E; e += nblk) {
            const float *wr = p.Wr + size_t(e) * H;
            float a = 0.f;
            for (int i = threadIdx.x; i < (H >> 2); i += kThreads) {
                const float4 w4 = __ldg(reinterpret_cast<const float4 *>(wr) + i);
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
                s += p.bias ? p.bias[e] : 0.f;
                if (publish) st_relaxed_u64(p.sync + e, tagged(tag, s));
            }
            __syncthreads();
        }
    }
    if (threadIdx.x == 0) TL_STAMP(p, 2);

    // ---------------- 2. warp 0 polls the E logits into shared memory, as
    // floats and as order-preserving keys, while the other warps prepare x
    // for the gate/up rows (run sums, and for digit kernels the digits).
    // Lane l holds words l, l+32, ...; every round reloads all of the lane's
    // still-stale words together, so a round costs one L2 round trip.
    const int Ep = p.router_on ? ((E + 31) & ~31) : 0;
    float *lsm = red + kWarps;  // E logits, clear of the partial sums thread 0 may still read
    if (p.router_on && warp == 0) {
        constexpr int kPer = kMaxE / 32;
        bool got[kPer];
#pragma unroll
        for (int i = 0; i < kPer; ++i) got[i] = lane + 32 * i >= E;
        bool timed_out = false;
        while (true) {
            unsigned long long wv[kPer];
#pragma unroll
            for (int i = 0; i < kPer; ++i)
                if (!got[i]) wv[i] = ld_relaxed_u64(p.sync + lane + 32 * i);
            bool all = true;
#pragma unroll
            for (int i = 0; i < kPer; ++i) {
                if (got[i]) continue;
                if (tag_of(wv[i]) != tag) {
                    all = false;
                    continue;
                }
                got[i] = true;
                const int e = lane + 32 * i;
                float v = value_of(wv[i]);
                v = (v == v) ? v + 0.0f : -INFINITY;  // a NaN never ranks first; -0 ties +0
                lsm[e] = v;
                skey[e] = ordered_key(v);
            }
            if (__all_sync(0xffffffffu, all)) break;
            if (global_timer_ns() > deadline) {
                timed_out = true;
                break;
            }
            pause_cycles(kPollPauseCycles);
        }
        for (int e = E + lane; e < Ep; e += 32) skey[e] = 0;  // below every logit's key
        if (timed_out && lane == 0) flags[1] = 1;
    } else {
        // x in 128-element chunks, lane l holding elements 4l..4l+3 of a chunk
        // (8 lanes per 32-element run): run sums, and for digit kernels the
        // digits (one packed word per plane and lane) and run scales
        const int w0 = p.router_on ? 1 : 0, nw = kWarps - w0;
        for (int c = warp - w0; c < (H >> 7); c += nw) {
            const int e0 = 128 * c + 4 * lane;
            const float4 v = *reinterpret_cast<const float4 *>(vec + padded(e0));
            if (kDigits) {
                uint32_t wa, wb, wc;
                float sum;
                const float sc = run_digits4(v, lane, wa, wb, wc, sum);
                const int off = plane_offset(e0, H >> 6);
                *reinterpret_cast<uint32_t *>(planes + off) = wa;
                *reinterpret_cast<uint32_t *>(planes + H + off) = wb;
                *reinterpret_cast<uint32_t *>(planes + 2 * H + off) = wc;
                if ((lane & 7) == 0) {
                    xscale[e0 >> 5] = sc;
                    vsum[e0 >> 5] = sum;
                }
            } else {
                const float sum = run_sum4(v);
                if ((lane & 7) == 0) vsum[e0 >> 5] = sum;
            }
        }
    }
    __syncthreads();
    if (flags[1]) {
        if (threadIdx.x == 0) {
            record_status(p.hdr, MOE_ERR_TIMEOUT, 1);
            red_relaxed_add_u64(&p.hdr->rows_done, 1ull);  // keep one count per CTA and call
        }
        return;  // no copies issued yet, no output written
    }
    if (threadIdx.x == 0) TL_STAMP(p, 8);

    // Top-k by rank in the order (value descending, index ascending): the
    // logit of rank j < k is slot j; every CTA finds the same.  Thread t
    // counts, for logit t % Ep, the keys in part t / Ep of the list that are
    // greater (G parts; a warp shares its part, so every load is a broadcast
    // of four keys).  Equal keys get equal counts; when two logits claim the
    // same rank below k, the counts are redone with ties ranked by index.
    // The softmax weights are computed later, off this path.
    if (p.router_on) {
        int G = 1;
        while (2 * G * Ep <= kThreads && G < 8) G *= 2;
        const int per = Ep / G;  // a multiple of 4
        const bool counter = int(threadIdx.x) < Ep * G;
        const int e = threadIdx.x % Ep, b0 = (threadIdx.x / Ep) * per;
        if (counter) {
            const uint32_t ke = skey[e];
            int cnt = 0;
            for (int o = b0; o < b0 + per; o += 4) {
                const uint4 k4 = *reinterpret_cast<const uint4 *>(skey + o);
                cnt += int(k4.x > ke) + int(k4.y > ke) + int(k4.z > ke) + int(k4.w > ke);
            }
            pcnt[threadIdx.x] = cnt;
        }
        if (threadIdx.x == 0) TL_STAMP(p, 11);
        __syncthreads();
        if (threadIdx.x == 0) TL_STAMP(p, 12);
        if (int(threadIdx.x) < E) {
            int r = 0;
            for (int g = 0; g < G; ++g) r += pcnt[g * Ep + threadIdx.x];
            if (r < k && atomicCAS(sel_e + r, -1, int(threadIdx.x)) != -1) flags[2] = 1;
        }
        __syncthreads();
        if (flags[2]) {
            if (counter) {
                const uint32_t ke = skey[e];
                int cnt = 0;
                for (int o = b0; o < b0 + per; o += 4) {
                    const uint4 k4 = *reinterpret_cast<const uint4 *>(skey + o);
                    cnt += int(k4.x > ke) + int(k4.y > ke) + int(k4.z > ke) + int(k4.w > ke);
                    cnt += int((k4.x == ke) & (o < e)) + int((k4.y == ke) & (o + 1 < e)) +
                           int((k4.z == ke) & (o + 2 < e)) + int((k4.w == ke) & (o + 3 < e));
                }
                pcnt[threadIdx.x] = cnt;
            }
            __syncthreads();
            if (int(threadIdx.x) < E) {
                int r = 0;
                for (int g = 0; g < G; ++g) r += pcnt[g * Ep + threadIdx.x];
                if (r < k) sel_e[r] = threadIdx.x;
            }
            __syncthreads();
        }
        if (threadIdx.x == 0) TL_STAMP(p, 13);
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

    // Lane 0 of each warp issues its i-th gate/up row pair as two bulk copies
    // (the gate row, then the up row: one contiguous segment each) into ring
    // slot i, counted on the row's mbarrier; a row of an invalid expert is
    // marked complete with no bytes.
    auto issue_gu = [&](int i) {
        const int u = u0 + warp + kWarps * i, j = u / I, r = u % I;
        const int e = sel_e[j];
        uint8_t *dst = ring + i * p.slot_bytes;
        uint64_t *bar = rbar + warp * kMaxNbw + i;
        if (e >= 0 && e < E) {
            mbar_arrive_expect_tx(bar, uint32_t(2 * row_gu));
            bulk_g2s(dst, p.gate + e * mat_gu + size_t(r) * row_gu, uint32_t(row_gu), bar);
            bulk_g2s(dst + row_gu, p.up + e * mat_gu + size_t(r) * row_gu, uint32_t(row_gu), bar);
        } else {
            mbar_arrive(bar);
        }
    };
    // the CTA's R output rows of each of the k experts: one contiguous range
    // per slot, one bulk copy each, all counted on the down mbarrier
    uint8_t *dbuf = smem + p.down_off;
    const uint32_t dbytes = uint32_t(R) * uint32_t(row_dn);
    auto issue_down = [&]() {
        uint32_t total = 0;
        for (int j = 0; j < k; ++j)
            if (sel_e[j] >= 0 && sel_e[j] < E) total += dbytes;
        mbar_arrive_expect_tx(dbar, total);
        if (dbytes == 0) return;
        for (int j = 0; j < k; ++j) {
            const int e = sel_e[j];
            if (e >= 0 && e < E)
                bulk_g2s(dbuf + size_t(j) * dbytes, p.down + e * mat_dn + size_t(r0) * row_dn, dbytes,
                         dbar);
        }
    };

    // Every row of the warp has its own slot (the host only launches shapes
    // where n_mine <= nbw): all gate/up rows are requested at once, then the
    // down rows; a bulk copy's bytes arrive in one piece, and each row has
    // its own barrier, so rows are consumed as they land.  No copy targets
    // shared memory that ordinary loads or stores used earlier in the
    // kernel: kernels that did (slots reused for later rows, scratch arrays
    // in the slots) raised illegal-instruction faults on GB300.
    if (lane == 0)
        for (int i = 0; i < n_mine; ++i) issue_gu(i);
    if (threadIdx.x == 0) issue_down();

    // the renormalised router weights of the k slots (softmax over the top k),
    // needed only by the down rows
    if (p.router_on && warp == 0) {
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

    XDigits X;
    if (kDigits) load_digits(X, planes, H, H >> 6, lane, xscale, vsum);

    for (int i = 0; i < n_mine; ++i) {
        if (!mbar_wait(rbar + warp * kMaxNbw + i, 0, deadline) && lane == 0) {
            flags[1] = 1;
            record_status(p.hdr, MOE_ERR_TIMEOUT, 5);
        }
        __syncwarp();
        if (threadIdx.x == 0 && i == 0) TL_STAMP(p, 9);
        const int u = u0 + warp + kWarps * i, j = u / I, r = u % I;
        const int e = sel_e[j];
        if (e >= 0 && e < E) {
            const uint8_t *src = ring + i * p.slot_bytes;
            float g, uu;
            if (kDigits) {
                const uint8_t *blk = src + (lane >> 2) * kBlockBytes;
                g = pair_dot_digits(blk, lane & 3, X);
                uu = pair_dot_digits(blk + row_gu, lane & 3, X);
                warp_sum2(g, uu, lane);
            } else {
                g = warp_sum(row_dot_pairs<NSB_H>(src, nsb_h, vec, vsum, lane));
                uu = warp_sum(row_dot_pairs<NSB_H>(src + row_gu, nsb_h, vec, vsum, lane));
            }
            if (lane == 0) p.hbuf[size_t(j) * I + r] = silu_mul(g, uu);
        }
        __syncwarp();
    }
    if (threadIdx.x == 0) TL_STAMP(p, 4);

    // ---------------- 4. h of all k slots -> down rows + combine
    __syncthreads();  // x in `vec` is dead once every warp is past its rows
    // This CTA's h values are out: count it in the header (release: the
    // CTA barrier above orders every warp's h stores before it), then thread
    // 0 waits until every CTA of the call has (acquire; one polled word per
    // CTA keeps the polling cheap).  h is then read once.
    if (threadIdx.x == 0) {
        if (publish) {
            __threadfence();
            red_release_add_u64(&p.hdr->rows_done, 1ull);
        }
        if (!await_count(&p.hdr->rows_done, (unsigned long long)tag * nblk, deadline)) flags[1] = 1;
    }
    __syncthreads();
    if (threadIdx.x == 0) TL_STAMP(p, 6);
    const int ip = padded_len(I);
    // digit kernels keep h as three digit planes of k*I bytes plus one scale
    // per 32-element run, in place of the fp32 vector
    uint8_t *hplanes = reinterpret_cast<uint8_t *>(vec);
    float *hscale = reinterpret_cast<float *>(hplanes + 3 * k * I);
    if (flags[1] == 0) {
        // h in 128-element chunks (a chunk never spans two slots: I is a
        // multiple of 256); warp w stages chunks w, w+16, ..., lane l holding
        // elements 4l..4l+3, kStageBatch chunks in flight per warp.  Slots of
        // invalid experts read as 0.
        const int nchunks = (k * I) >> 7;
        const float4 *h4 = reinterpret_cast<const float4 *>(p.hbuf);
        for (int c0 = warp; c0 < nchunks; c0 += kStageBatch * kWarps) {
            float4 v[kStageBatch];
#pragma unroll
            for (int t = 0; t < kStageBatch; ++t) {
                const int c = c0 + t * kWarps, e0 = 128 * c + 4 * lane;
                v[t] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (c < nchunks) {
                    const int e = sel_e[e0 / I];
                    if (e >= 0 && e < E) v[t] = __ldcg(h4 + (e0 >> 2));
                }
            }
            if (threadIdx.x == 0 && c0 == 0) TL_STAMP(p, 14);
#pragma unroll
            for (int t = 0; t < kStageBatch; ++t) {
                const int c = c0 + t * kWarps, e0 = 128 * c + 4 * lane;
                if (c >= nchunks) break;  // warp-uniform
                if (kDigits) {
                    uint32_t wa, wb, wc;
                    float sum;
                    const float sc = run_digits4(v[t], lane, wa, wb, wc, sum);
                    const int off = plane_offset(e0, (k * I) >> 6);
                    *reinterpret_cast<uint32_t *>(hplanes + off) = wa;
                    *reinterpret_cast<uint32_t *>(hplanes + k * I + off) = wb;
                    *reinterpret_cast<uint32_t *>(hplanes + 2 * k * I + off) = wc;
                    if ((lane & 7) == 0) {
                        hscale[e0 >> 5] = sc;
                        vsum[e0 >> 5] = sum;
                    }
                } else {
                    const int j = e0 / I;
                    *reinterpret_cast<float4 *>(vec + j * ip + padded(e0 - j * I)) = v[t];
                    const float sum = run_sum4(v[t]);
                    if ((lane & 7) == 0) vsum[e0 >> 5] = sum;
                }
            }
        }
    }
    if (threadIdx.x == 0) TL_STAMP(p, 15);
    __syncthreads();
    if (threadIdx.x == 0) TL_STAMP(p, 5);
    if (flags[1]) {
        if (threadIdx.x == 0) record_status(p.hdr, MOE_ERR_TIMEOUT, 4);
    } else {

        if (threadIdx.x == 0 && !mbar_wait(dbar, 0, deadline)) flags[1] = 1;
        __syncthreads();  // the down rows have landed
        if (threadIdx.x == 0) TL_STAMP(p, 10);
        const size_t jstride = size_t(R) * row_dn;
        if (kDigits) {
            // Thread -> unit u = (slot j, block sb, pair c) of the down rows;
            // its 64 elements of h_j stay in registers while it walks rows
            // q, q + Q, ... of the CTA's share.  The weighted partial dots go
            // to P[row][u] (in the gate/up slots, free now), then one warp per
            // row sums them in a fixed order.
            constexpr int kPer = (NSB_I > 0 ? NSB_I : 1) * 4;  // units per slot
            const int Ud = k * kPer;                           // <= 512
            const int Q = kThreads / Ud;
            float *P = reinterpret_cast<float *>(smem + p.ring_off);
            const int u = threadIdx.x % Ud, q = threadIdx.x / Ud;
            if (q < Q) {
                const int j = u / kPer, rem = u - j * kPer, sb = rem >> 2, c = rem & 3;
                const int e = sel_e[j];
                const bool valid = e >= 0 && e < E;
                const float wj = sel_w[j];
                XDigits Xh;
                load_digits(Xh, hplanes, k * I, (k * I) >> 6, (j * I + kQK * sb + 64 * c) >> 6,
                            hscale, vsum);
                const uint8_t *base = dbuf + j * jstride + sb * kBlockBytes;
                for (int rr = q; rr < R; rr += Q) {
                    const float part = valid ? wj * pair_dot_digits(base + rr * row_dn, c, Xh) : 0.f;
                    P[rr * Ud + u] = part;
                }
            }
            __syncthreads();
            for (int rr = warp; rr < R; rr += kWarps) {
                float acc = 0.f;
                for (int uu = lane; uu < Ud; uu += 32) acc += P[rr * Ud + uu];
                acc = warp_sum(acc);
                if (lane == 0) p.y[r0 + rr] = epilogue_value(p.ep, 0, H, r0 + rr, acc);
            }
        } else {
            const int n_rows = R > warp ? (R - warp + kWarps - 1) / kWarps : 0;  // rows warp+16i
            for (int i = 0; i < n_rows; ++i) {
                const int rr = warp + kWarps * i;  // row inside the CTA's share
                const uint8_t *src = dbuf + size_t(rr) * row_dn;
                // k experts x nsb_i blocks x 4 sub-block pairs, spread over the
                // 32 lanes in a fixed order; each pair's partial dot is
                // weighted by its slot's router weight, then one warp reduction
                // gives y (deterministic)
                float yacc = 0.f;
                const int per_j = (NSB_I > 0 ? NSB_I : nsb_i) * 4;  // (block, pair) units per slot
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
                if (lane == 0) p.y[r0 + rr] = epilogue_value(p.ep, 0, H, r0 + rr, yacc);
            }
        }
    }
    // every copy must land before the CTA's shared memory goes away (on a
    // timed-out path some barriers were not waited for): a second bounded wait
    {
        const uint64_t limit = global_timer_ns() + p.wait_ns;
        if (lane == 0)
            for (int i = 0; i < n_mine; ++i) mbar_wait(rbar + warp * kMaxNbw + i, 0, limit);
        if (threadIdx.x == 0) mbar_wait(dbar, 0, limit);
    }
    if (threadIdx.x == 0) TL_STAMP(p, 7);
}

}  // namespace fused

namespace {

struct FusedConfig {
    int nbw = 0, slot_bytes = 0, ring_off = 0, down_off = 0, dig_off = 0, smem = 0;
};

// The kernels instantiated for 8 blocks per gate/up row and 3 or 4 per down
// row keep x as digits.
bool uses_digits(int H, int I) { return H / kQK == 8 && (I / kQK == 3 || I / kQK == 4); }

bool fused_config(int H, int E, int k, int I, int nblk, int max_smem, FusedConfig &c) {
    using namespace fused;
    if (E > kMaxE || k > kMaxK || nblk < 1) return false;
    const int row_gu = (H / kQK) * kBlockBytes, row_dn = (I / kQK) * kBlockBytes;
    const int vec_pad = std::max(padded_len(H), k * padded_len(I));
    const int vec_sum = std::max(H, k * I) / 16;
    const int vec_end = int(align256(size_t(kHeadBytes) + sizeof(float) * size_t(vec_pad + vec_sum)));
    // x as three digit planes plus one scale per 32-element run
    const int dig_bytes =
        uses_digits(H, I) ? int(align256(size_t(3) * H + sizeof(float) * (H / 32))) : 0;
    const int dig_end = vec_end + dig_bytes;
    const int rmax = (H + nblk - 1) / nblk;
    const int down_bytes = int(align256(size_t(k) * rmax * row_dn));
    // the CTA's down rows resident, rings hold gate/up row pairs
    const int slot = (2 * row_gu + 127) / 128 * 128;
    const int nbw = std::min(kMaxNbw, (max_smem - dig_end - down_bytes) / (kWarps * slot));
    // Only shapes where the CTA's down rows stay resident and every warp's
    // gate/up rows have a ring slot each take this kernel: all weight bytes
    // are requested at once.  Variants that reused ring slots (streaming
    // down rows through the rings, or gate/up rows beyond the ring's size)
    // raised illegal-instruction faults on GB300 and are not built; those
    // shapes (Qwen3-235B-A22B among them) run the multi-kernel path.
    const int units_max = (k * I + nblk - 1) / nblk;
    const int rows_per_warp = (units_max + kWarps - 1) / kWarps;
    if (nbw < 1 || nbw < rows_per_warp) return false;
    // digit kernels keep the down rows' partial dots (rmax x units) in the slots
    if (uses_digits(H, I) &&
        size_t(rmax) * k * (I / kQK) * 4 * sizeof(float) > size_t(kWarps) * rows_per_warp * slot)
        return false;
    c.dig_off = vec_end;
    c.down_off = dig_end;
    c.ring_off = dig_end + down_bytes;
    c.nbw = rows_per_warp;
    c.slot_bytes = slot;
    c.smem = c.ring_off + kWarps * c.nbw * slot;
    return c.smem <= max_smem;
}

template <int A, int B>
void *kernel_ptr() {
    return reinterpret_cast<void *>(&fused::decode_fused_kernel<A, B>);
}

void *pick_kernel(int H, int I) {
    const int a = H / kQK, b = I / kQK;
    if (a == 8 && b == 3) return kernel_ptr<8, 3>();
    if (a == 8 && b == 4) return kernel_ptr<8, 4>();
    if (a == 1 && b == 1) return kernel_ptr<1, 1>();
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
    void *ks[] = {kernel_ptr<8, 3>(), kernel_ptr<8, 4>(), kernel_ptr<1, 1>(), kernel_ptr<0, 0>()};
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

cudaError_t launch_decode_fused(int dev, const float *x, const float *norm_w, float eps,
                                const OutEpilogue &ep, const float *Wr, const float *bias,
                                const int32_t *idx_in, const float *w_in, int32_t *idx_out,
                                float *w_out, const uint8_t *gate, const uint8_t *up,
                                const uint8_t *down, int H, int E, int k, int I, float *y,
                                unsigned long long *sync, float *hbuf, WsHeader *hdr, int withhold,
                                unsigned long long wait_ns, unsigned long long *timeline,
                                int timeline_cap, cudaStream_t s) {
    FusedConfig c;
    if (!fused_config(H, E, k, I, g_fused_blocks[dev], g_fused_max_smem[dev], c))
        return cudaErrorInvalidValue;
    fused::Params p;
    p.x = x;
    p.norm_w = norm_w;
    p.eps = eps;
    p.ep = ep;
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
    p.sync = sync;
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
    p.down_off = c.down_off;
    p.dig_off = c.dig_off;
    p.withhold = withhold;
    p.wait_ns = wait_ns;
    p.timeline = timeline;
    p.timeline_cap = timeline ? timeline_cap : 0;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(g_fused_blocks[dev]);
    cfg.blockDim = dim3(fused::kThreads);
    cfg.dynamicSmemBytes = c.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    void *args[] = {&p};
    return cudaLaunchKernelExC(&cfg, pick_kernel(H, I), args);
}

}  // namespace moeq4k
