// Dot products of Q4_K sub-block pairs with an fp32 vector, shared by the
// single-token kernels.  A lane's unit is sub-block pair c (sub-blocks 2c
// and 2c+1: the low and high nibbles of code bytes qs[32c .. 32c+31]) of one
// 256-weight block; its 16-byte block head carries d, dmin and the 6-bit
// scales and mins.  Two forms of the vector:
//   fp32     a padded shared-memory copy plus 32-element sums; the codes
//            enter as 1 + q/128 (one byte permute and one FMA per weight);
//   digits   three signed base-254 digits per element with a scale per
//            32-element run (x ~= s (a + b/254 + c/254^2)), so four codes
//            times four elements is one dp4a per digit; the digits leave
//            6.1e-8 of the run's max|x|, the fp32 scalings a few ulps.
// A GGUF Q4_K weight is w = d * sc * q - dmin * m.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

#include "common.cuh"

namespace moeq4k {

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
__device__ __forceinline__ float pair_dot(const uint4 &head, const uint4 &qa, const uint4 &qb, int c,
                                          const float *xs, const float *s2) {
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

// The same with the block in (shared or global) memory at `blk`.
__device__ __forceinline__ float pair_dot(const uint8_t *blk, int c, const float *xs,
                                          const float *s2) {
    const uint4 head = *reinterpret_cast<const uint4 *>(blk);
    const uint4 qa = *reinterpret_cast<const uint4 *>(blk + 16 + 32 * c);
    const uint4 qb = *reinterpret_cast<const uint4 *>(blk + 32 + 32 * c);
    return pair_dot(head, qa, qb, c, xs, s2);
}

// ---------------------------------------------------------------------------
// Integer form of a vector: per 32-element run, x / s (s = max|x| / 127)
// as three signed base-254 digits, so that a 4-bit code times four
// elements is one dp4a per digit.
// ---------------------------------------------------------------------------

// d = c + sum_i a.byte[i] * b.byte[i], a's bytes unsigned, b's signed.
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ bool finite_f(float v) { return fabsf(v) <= 3.402823466e38f; }

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
__device__ __forceinline__ float pair_dot_digits(const uint4 &head, const uint4 &qa, const uint4 &qb,
                                                 int c, const XDigits &X) {
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

// The same with the block in (shared or global) memory at `blk`.
__device__ __forceinline__ float pair_dot_digits(const uint8_t *blk, int c, const XDigits &X) {
    const uint4 head = *reinterpret_cast<const uint4 *>(blk);
    const uint4 qa = *reinterpret_cast<const uint4 *>(blk + 16 + 32 * c);
    const uint4 qb = *reinterpret_cast<const uint4 *>(blk + 32 + 32 * c);
    return pair_dot_digits(head, qa, qb, c, X);
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

}  // namespace moeq4k
