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
//     router logits.
//     Each logit is published as one 64-bit word that also carries the
//     call's tag, so readers need no barrier: they poll the words until
//     every tag is the current one.
//  2. Every CTA reads the E logits and runs the same top-k and
//     renormalisation, so all CTAs know the k experts without a broadcast.
//  3. The k*I gate/up row pairs are split evenly over the CTAs and, inside a
//     CTA, over its warps.  Each warp requests all of its rows at once into
//     private shared-memory slots with 16-byte cp.async copies (every lane
//     issues, so hundreds of requests per SM are in flight; one commit group
//     per row, waited with cp.async.wait_group), then all threads request
//     the CTA's down rows (its share of the H output rows, for all k
//     experts).  Each value of h = SiLU(g) * u is published as a tagged word
//     like the logits.  (Requesting only a few rows ahead of the compute was
//     measured slower: the stream then falls short of the HBM bandwidth.)
//  4. Each CTA polls the k*I tagged h words into shared memory, then for
//     each of its output rows computes o_j = Wd[e_j][row] . h_j for
//     j = 0..k-1 and y = sum_j w_j o_j in slot order: deterministic, no
//     atomics.
// The tag of a call comes from a counter in the workspace header to which
// every CTA adds 1 at its start, so it needs no reset between calls or graph
// replays.  Every wait is bounded by a global-timer deadline; on expiry the
// kernel records MOE_ERR_TIMEOUT, stops computing and lets its copies land
// before returning.  (Copy completion needs no bound: loads always finish.)
//
// Arithmetic of the gate/up rows when H = 2048 (8 Q4_K blocks per row): lane
// L always covers the same 64 elements of x (sub-block pair L % 4 of block
// L / 4), so it keeps them in registers in an exact integer form: x / s, with
// s = max|x| / 127 over each 32-element run, is split into three signed
// base-254 digits (x ~= s (a + b/254 + c/254^2), each digit in [-127, 127];
// the digits leave 6.1e-8 of the run's max|x|, the fp32 scalings add a few
// ulps of x: below 2.5e-7 of the run's max|x| in all).  A 4-bit code times a
// digit word is then one dp4a (four exact 8-bit products summed in int32),
// and the fp32 scales of the block are applied once per sub-block.  Other
// shapes, and all down rows, dot fp32 vectors in shared memory.
#include <algorithm>

#include "async_copy.cuh"
#include "common.cuh"
#include "kernels.cuh"

namespace moeq4k {
namespace fused {

constexpr int kWarps = 16;
constexpr int kThreads = kWarps * 32;
constexpr int kMaxNbw = 8;         // ring slots per warp
constexpr int kHeadBytes = 5120;   // small shared arrays (see the kernel's first lines)
constexpr int kStageBatch = 8;     // 128-value chunks of h in flight per warp while staging
constexpr long long kBackoffCycles = 600;  // wait after a poll that found a stale word

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

// Padded shared-memory vector: 4 floats of padding after every 64, so the
// 8 lanes of a quarter-warp reading 16-float runs that are 64 floats apart
// hit distinct banks.
__device__ __forceinline__ int padded(int i) { return i + ((i >> 6) << 2); }
__host__ __device__ inline int padded_len(int n) { return n + (n >> 4); }

// 1 + q/128 as fp32 from byte i of v, where v's bytes are 0x80 | q.
__device__ __forceinline__ float one_plus_q(uint32_t v, int i) {
    return __uint_as_float(__byte_perm(v, 0x3F000000u, 0x7044u | (uint32_t(i) << 8)));
}

__device__ __forceinline__ float u6_to_float(uint32_t v) {
    return __uint_as_float(0x4B000000u | v) - 8388608.0f;
}

// Scale and min of sub-blocks 2c and 2c+1 of a block head, as dmul*d*sc and
// dmin*m.
__device__ __forceinline__ void pair_scales(const uint4 &head, int c, float dmul, float &A0,
                                            float &B0, float &A1, float &B1) {
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
    const float dm = dd.x * dmul;
    A0 = dm * u6_to_float(sc0);
    A1 = dm * u6_to_float(sc1);
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
    pair_scales(head, c, 128.0f, A0, B0, A1, B1);
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

// Sum each 32-float run of the padded vector into sum32, one warp per run
// (consecutive words, no bank conflicts; fixed reduction order).
__device__ __forceinline__ void run_sums32(const float *vec, float *sum32, int runs, int warp,
                                           int lane) {
    for (int r = warp; r < runs; r += kWarps) {
        const float s = warp_sum(vec[padded(32 * r + lane)]);
        if (lane == 0) sum32[r] = s;
    }
}

// ---------------------------------------------------------------------------
// Integer form of x for the gate/up rows (H = 2048).
// ---------------------------------------------------------------------------

// d = c + sum_i a.byte[i] * b.byte[i], a's bytes unsigned, b's signed.
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ bool finite_f(float v) { return fabsf(v) <= 3.402823466e38f; }

// Unsigned key with the order of the float: larger value, larger key.
__device__ __forceinline__ uint32_t ordered_key(float v) {
    const uint32_t b = __float_as_uint(v);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Round to nearest (ties to even) of |t| < 2^22 by adding 1.5 * 2^23: the
// integer sits in the low mantissa bits.  Returns it, and the rounded value
// in `r`.  The _rn intrinsics keep the adds out of any fused multiply-add.
__device__ __forceinline__ int round_shift(float t, float &r) {
    const float tm = __fadd_rn(t, 12582912.0f);
    r = __fadd_rn(tm, -12582912.0f);
    return __float_as_int(tm) - 0x4B400000;
}

// Three base-254 digits of t (|t| <= 127): t ~= a + b/254 + c/254^2, each in
// [-127, 127].  Each remainder t - rint(t) is exact in fp32; only the
// scalings by 254 round, at fp32 precision.
__device__ __forceinline__ void digits3(float t, int &a, int &b, int &c) {
    float ra, rb, rc;
    a = round_shift(t, ra);
    const float r1 = __fmul_rn(__fsub_rn(t, ra), 254.0f);
    b = round_shift(r1, rb);
    const float r2 = __fmul_rn(__fsub_rn(r1, rb), 254.0f);
    c = round_shift(r2, rc);
}

// Low bytes of four ints as one word (a0 in the lowest byte).
__device__ __forceinline__ uint32_t pack4(int a0, int a1, int a2, int a3) {
    return __byte_perm(__byte_perm(a0, a1, 0x0040), __byte_perm(a2, a3, 0x0040), 0x5410);
}

// A warp holds 128 consecutive elements, lane l the four at 4l (so lanes
// 8q..8q+7 hold the q-th 32-element run).  Sum of the lane's run, in a fixed
// order.
__device__ __forceinline__ float run_sum4(const float4 v) {
    float s = (v.x + v.y) + (v.z + v.w);
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    return s;
}

// The same layout: writes the lane's digits of x / s (s = max|x| / 127 over
// its run) as one packed word per plane and the run's sum; returns s / 254.
// Only the scaling by 127/max rounds besides digits3's.  A run with a
// non-finite element gets a NaN scale, so the non-finite value propagates.
__device__ __forceinline__ float run_digits4(const float4 v, int lane, uint32_t &wa, uint32_t &wb,
                                             uint32_t &wc, float &sum) {
    float mx = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    sum = run_sum4(v);
    const uint32_t bad = __ballot_sync(
        0xffffffffu, !(finite_f(v.x) && finite_f(v.y) && finite_f(v.z) && finite_f(v.w)));
    const bool finite = ((bad >> (lane & 24)) & 0xFFu) == 0;
    const float inv = (finite && mx > 0.f) ? 127.0f / mx : 0.f;
    int a0, b0, c0, a1, b1, c1, a2, b2, c2, a3, b3, c3;
    digits3(v.x * inv, a0, b0, c0);
    digits3(v.y * inv, a1, b1, c1);
    digits3(v.z * inv, a2, b2, c2);
    digits3(v.w * inv, a3, b3, c3);
    wa = pack4(a0, a1, a2, a3);
    wb = pack4(b0, b1, b2, b3);
    wc = pack4(c0, c1, c2, c3);
    return finite ? mx * (1.0f / (127.0f * 254.0f)) : __uint_as_float(0x7FC00000u);
}

// Digit planes hold 64-element units (unit u = elements 64u .. 64u+63):
// element e sits at byte plane_offset(e, nunits) of its plane, so that the
// 16-byte chunk q of consecutive units is contiguous (a warp reading its
// units' chunk q touches consecutive banks).
__device__ __forceinline__ int plane_offset(int e, int nunits) {
    const int u = e >> 6, w = e & 63;
    return ((w >> 4) * nunits + u) * 16 + (w & 15);
}

// One thread's 64-element unit of a vector (sub-block pair c of block s) as
// digit words (4 consecutive elements each; words 0-7 are sub-block 2c,
// 8-15 sub-block 2c+1), their scales and fp32 sums.
struct XDigits {
    uint32_t a[16], b[16], c[16];
    float s0, s1;      // run scale / 254; s1 also / 16 (high nibbles are read unshifted)
    float sum0, sum1;  // sum of x over each run
};

// Planes a, b, c are `plane_bytes` apart; `u` is the unit, of `nunits`.
__device__ __forceinline__ void load_digits(XDigits &X, const uint8_t *planes, int plane_bytes,
                                            int nunits, int u, const float *scales,
                                            const float *sum32) {
    const int e0 = 64 * u;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint8_t *chunk = planes + (q * nunits + u) * 16;
        const uint4 va = *reinterpret_cast<const uint4 *>(chunk);
        const uint4 vb = *reinterpret_cast<const uint4 *>(chunk + plane_bytes);
        const uint4 vc = *reinterpret_cast<const uint4 *>(chunk + 2 * plane_bytes);
        X.a[4 * q] = va.x, X.a[4 * q + 1] = va.y, X.a[4 * q + 2] = va.z, X.a[4 * q + 3] = va.w;
        X.b[4 * q] = vb.x, X.b[4 * q + 1] = vb.y, X.b[4 * q + 2] = vb.z, X.b[4 * q + 3] = vb.w;
        X.c[4 * q] = vc.x, X.c[4 * q + 1] = vc.y, X.c[4 * q + 2] = vc.z, X.c[4 * q + 3] = vc.w;
    }
    X.s0 = scales[e0 >> 5];
    X.s1 = scales[(e0 >> 5) + 1] * 0.0625f;
    X.sum0 = sum32[e0 >> 5];
    X.sum1 = sum32[(e0 >> 5) + 1];
}

// Dot of sub-blocks 2c and 2c+1 of one block with the lane's x digits:
// sum(q x) over a run is s/254 * ((254 A + B) + C/254) with A, B, C the
// exact integer sums of the codes times each digit.
__device__ __forceinline__ float pair_dot_digits(const uint8_t *blk, int c, const XDigits &X) {
    const uint4 head = *reinterpret_cast<const uint4 *>(blk);
    const uint4 qa = *reinterpret_cast<const uint4 *>(blk + 16 + 32 * c);
    const uint4 qb = *reinterpret_cast<const uint4 *>(blk + 32 + 32 * c);
    const uint32_t w[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
    int a0 = 0, b0 = 0, c0 = 0, a1 = 0, b1 = 0, c1 = 0;
#pragma unroll
    for (int m = 0; m < 8; ++m) {
        const uint32_t lo = w[m] & 0x0F0F0F0Fu;  // codes of elements 4m..4m+3
        const uint32_t hi = w[m] & 0xF0F0F0F0u;  // 16 x codes of elements 32+4m..32+4m+3
        a0 = dp4a_us(lo, X.a[m], a0);
        b0 = dp4a_us(lo, X.b[m], b0);
        c0 = dp4a_us(lo, X.c[m], c0);
        a1 = dp4a_us(hi, X.a[8 + m], a1);
        b1 = dp4a_us(hi, X.b[8 + m], b1);
        c1 = dp4a_us(hi, X.c[8 + m], c1);
    }
    // |254 a + b| < 2^28 (high nibbles) and < 2^24 (low): no overflow
    const float qx0 = X.s0 * fmaf(float(c0), 1.0f / 254.0f, float(254 * a0 + b0));
    const float qx1 = X.s1 * fmaf(float(c1), 1.0f / 254.0f, float(254 * a1 + b1));
    float A0, B0, A1, B1;
    pair_scales(head, c, 1.0f, A0, B0, A1, B1);
    float acc = A0 * qx0;
    acc = fmaf(-B0, X.sum0, acc);
    acc = fmaf(A1, qx1, acc);
    acc = fmaf(-B1, X.sum1, acc);
    return acc;
}

// Warp sums of g and u in a fixed order; every lane of 0..15 gets the sum of
// g, every lane gets the sum of u.
__device__ __forceinline__ void warp_sum2(float &g, float &u, int lane) {
    const bool upper = (lane & 16) != 0;
    float keep = upper ? u : g;
    keep += __shfl_xor_sync(0xffffffffu, upper ? g : u, 16);
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) keep += __shfl_xor_sync(0xffffffffu, keep, o);
    g = keep;
    u = __shfl_sync(0xffffffffu, keep, 16);
}

// Busy-wait on the SM clock (no memory traffic) for about `cycles`.
__device__ __forceinline__ void pause_cycles(long long cycles) {
    const long long until = clock64() + cycles;
    while (clock64() < until) {
    }
}

// Poll one tagged word until it carries `tag`; false when `deadline` passes.
// A miss waits kBackoffCycles before the next load: every CTA polls the same
// few lines, and back-to-back reloads were measured to delay the stores they
// wait for by microseconds.
__device__ __forceinline__ bool await_word(const unsigned long long *p, uint32_t tag,
                                           uint64_t deadline, unsigned long long &w) {
    w = ld_relaxed_u64(p);
    while (tag_of(w) != tag) {
        if (global_timer_ns() > deadline) return false;
        pause_cycles(kBackoffCycles);
        w = ld_relaxed_u64(p);
    }
    return true;
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
    float *red = reinterpret_cast<float *>(flags + 4); // kWarps partial sums, then kMaxE logits
    uint32_t *skey = reinterpret_cast<uint32_t *>(smem + 1536);  // kMaxE logit keys
    int *pcnt = reinterpret_cast<int *>(smem + 2560);            // kThreads partial ranks
    float *vec = reinterpret_cast<float *>(smem + kHeadBytes);
    const int H = p.H, E = p.E, k = p.k, I = p.I;
    const int vec_pad = max(padded_len(H), k * padded_len(I));
    float *vsum = vec + vec_pad;
    uint8_t *planes = smem + p.dig_off;
    float *xscale = reinterpret_cast<float *>(planes + 3 * H);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
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
    }
    if (threadIdx.x < 32) sel_e[threadIdx.x] = -1;
    // ---------------- 1. router logits (a share per CTA).
    // The CTA's first logit is computed while x is staged: x and the router
    // row are requested together, so their latencies overlap.
    {
        const int e = blockIdx.x;
        const bool logit = p.router_on && e < E;
        const float *wr = p.Wr + size_t(logit ? e : 0) * H;
        float a = 0.f;
        for (int i = threadIdx.x; i < (H >> 2); i += kThreads) {
            const float4 x4 = __ldg(reinterpret_cast<const float4 *>(p.x) + i);
            if (logit) {
                const float4 w4 = __ldg(reinterpret_cast<const float4 *>(wr) + i);
                a = fmaf(w4.x, x4.x, a);
                a = fmaf(w4.y, x4.y, a);
                a = fmaf(w4.z, x4.z, a);
                a = fmaf(w4.w, x4.w, a);
            }
            *reinterpret_cast<float4 *>(vec + padded(4 * i)) = x4;
        }
        a = warp_sum(a);
        if (lane == 0) red[warp] = a;
        if (threadIdx.x == 0) *tag_sh = uint32_t(calls0 / nblk) + 1u;
        __syncthreads();
        if (logit && threadIdx.x == 0) {
            float sum = 0.f;
            for (int w = 0; w < kWarps; ++w) sum += red[w];
            sum += p.bias ? p.bias[e] : 0.f;
            if (publish) st_relaxed_u64(p.sync + e, tagged(*tag_sh, sum));
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

    // ---------------- 2. the first Ep threads (E rounded up to a warp) poll
    // the E logits into shared memory, as floats and as order-preserving
    // keys, while the other warps prepare x for the gate/up rows (run sums,
    // and for digit kernels the digits).
    const int Ep = p.router_on ? ((E + 31) & ~31) : 0;
    float *lsm = red + kWarps;  // E logits, clear of the partial sums thread 0 may still read
    if (int(threadIdx.x) < Ep) {
        uint32_t key = 0;  // below every logit's key
        if (int(threadIdx.x) < E) {
            unsigned long long wv;
            if (!await_word(p.sync + threadIdx.x, tag, deadline, wv)) flags[1] = 1;
            float v = value_of(wv);
            v = (v == v) ? v + 0.0f : -INFINITY;  // a NaN never ranks first; -0 ties +0
            lsm[threadIdx.x] = v;
            key = ordered_key(v);
        }
        skey[threadIdx.x] = key;
    } else {
        // x in 128-element chunks, lane l holding elements 4l..4l+3 of a chunk
        // (8 lanes per 32-element run): run sums, and for digit kernels the
        // digits (one packed word per plane and lane) and run scales
        const int w0 = Ep >> 5, nw = kWarps - w0;
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
    const int n16_gu = row_gu >> 4, n16_dn = row_dn >> 4;

    // issue the copies of this warp's i-th gate/up row pair into ring slot i
    auto issue_gu = [&](int i) {
        const int u = u0 + warp + kWarps * i, j = u / I, r = u % I;
        const int e = sel_e[j];
        uint8_t *dst = ring + i * p.slot_bytes;
        if (e >= 0 && e < E) {
            const uint8_t *g = p.gate + e * mat_gu + size_t(r) * row_gu;
            const uint8_t *uu = p.up + e * mat_gu + size_t(r) * row_gu;
            for (int c = lane; c < 2 * n16_gu; c += 32) {
                const uint8_t *src = c < n16_gu ? g + 16 * c : uu + 16 * (c - n16_gu);
                cp_async_16(dst + 16 * c, src);
            }
        }
        cp_async_commit();
    };
    // this thread's share of the CTA's R output rows of all k experts (k
    // contiguous ranges), one commit group
    uint8_t *dbuf = smem + p.down_off;
    auto issue_down = [&]() {
        const int per_j = R * n16_dn;
        for (int c = threadIdx.x; c < k * per_j; c += kThreads) {
            const int j = c / per_j, w16 = c % per_j;
            const int e = sel_e[j];
            if (e >= 0 && e < E)
                cp_async_16(dbuf + 16 * c, p.down + e * mat_dn + size_t(r0) * row_dn + 16 * w16);
        }
        cp_async_commit();
    };

    // Every row of the warp has its own slot (the host only launches shapes
    // where n_mine <= nbw): all gate/up rows are requested at once, then the
    // down rows.  Commit groups: row 0, ..., row n_mine-1, the down rows.
    // No cp.async targets shared memory that ordinary loads or stores used
    // earlier in the kernel: kernels that did (slots reused for later rows,
    // scratch arrays in the slots) raised illegal-instruction faults on
    // GB300.
    for (int i = 0; i < n_mine; ++i) issue_gu(i);
    issue_down();

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
        cp_async_wait_pending(n_mine - i);  // the later rows and the down rows may pend
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

        cp_async_wait_all();  // this thread's share of the down rows
        __syncthreads();      // everyone's share
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
                if (lane == 0) p.y[r0 + rr] = acc;
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
                if (lane == 0) p.y[r0 + rr] = yacc;
            }
        }
    }
    // every copy this thread issued must land before the CTA's shared memory goes away
    cp_async_wait_all();
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

cudaError_t launch_decode_fused(int dev, const float *x, const float *Wr, const float *bias,
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
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void *args[] = {&p};
    return cudaLaunchKernelExC(&cfg, pick_kernel(H, I), args);
}

}  // namespace moeq4k
