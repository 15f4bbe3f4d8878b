// Router logits of large batches on the tensor cores, top-k fused.
//
// forward_qwen3_moe_cuda_traced.rs (aprender-serve 0.34.0), doc of
// forward_qwen3_moe_cuda_traced_with_plan: the router stage is the k
// post-softmax, renormalised top-k weights of a token; the logits are the
// fp32 product l = x Wr^T (+ bias).
//
// The tensor cores have no fp32 operand type; tf32 keeps 11 of fp32's 24
// significand bits.  Each operand value v is split as v = hi(v) + lo(v),
// hi(v) = v with its low 13 significand bits cleared (exactly a tf32
// value), lo(v) = v - hi(v) (exact in fp32), and
//     x . w ~= hi(x) . hi(w) + lo(x) . hi(w) + hi(x) . lo(w),
// which drops lo(x) . lo(w) (below 2^-22 of |x w|) and the tf32 rounding of
// the lo parts (below 2^-21): a relative error near 2^-20 per product, so a
// logit's error stays near 1e-6 of the sum of |x_h w_h|, far below the gaps
// the selection depends on.  Three MMAs per K step, fp32 accumulation in
// tensor memory.
//
// A cluster of four CTAs per tile of 128 tokens, CTA r taking the K quarter
// r.  Per 32-K stage: TMA brings the x and Wr tiles (128 rows x 128 bytes,
// 128-byte swizzle) into a five-slot ring; eight split warps split the two
// tiles in place (hi back into the tile, lo into one of two lo buffers: the
// split is elementwise, so the swizzled layout carries over) and arrive on
// the slot's barrier; a ninth warp, one elected lane issuing, waits for that
// barrier and issues twelve MMAs (M = 128 tokens, N = 128 experts, K = 8
// each) into the stage's own accumulator, then commits.  Stage st's
// accumulator is added into fp32 registers by the split warps during stage
// st + 2 (three accumulators), so the tensor pipe runs up to two stages
// behind the split, and no CTA-wide barrier sits in the loop.  The four
// partial tiles then meet in the owner's shared memory: each split warp
// pushes its rows of another CTA's 32 tokens there with 16-byte
// asynchronous stores that complete on the owner's barrier, and CTA r adds
// the quarters of its tokens in rank order with the bias and ranks each
// token with one warp, from registers.  Fixed MMA and reduction order:
// deterministic.  Every wait is bounded by a global-timer deadline; a
// timed-out wait records MOE_ERR_TIMEOUT and the cluster writes no routing.
#include <cooperative_groups.h>
#include <cuda.h>

#include "async_copy.cuh"
#include "common.cuh"
#include "kernels.cuh"
#include "tcgen05.cuh"

namespace moeq4k {
namespace rtc {

constexpr int kTM = 128;                  // tokens per cluster tile (MMA M)
constexpr int kEN = 128;                  // experts (MMA N), E <= 128
constexpr int kSplit = 4;                 // K quarters = CTAs per cluster
constexpr int kBK = 32;                   // K per stage: one 128-byte fp32 row
constexpr int kStages = 5;                // copy ring: the x and Wr tiles of a stage
constexpr int kTile = kTM * kBK * 4;      // 16 KB
constexpr int kStage = 2 * kTile;         // x, Wr (hi written back in place)
constexpr int kLo = 2 * kTile;            // lo(x), lo(Wr) of a stage; two buffers
constexpr int kHead = 1024;               // barriers and flags
constexpr int kSmem = 1024 + kHead + kStages * kStage + 2 * kLo;  // + slack to align to 1024
constexpr int kSplitWarps = 8;           // split / accumulate warps
constexpr int kThreads = 32 * (kSplitWarps + 1);  // + the MMA warp
constexpr int kPS = kEN + 4;              // row of the partial tile (floats)
constexpr int kTok = kTM / kSplit;        // tokens ranked by each CTA
static_assert(kSplit * kTok * kPS * 4 <= kStages * kStage, "the received quarters reuse the copy ring");
static_assert(kSmem <= 232448, "shared memory of one CTA");

struct Params {
    CUtensorMap mx, mw;   // x [T][H] and Wr [E][H], fp32, boxes of 32 K x 128 rows
    const float *bias;
    int T, H, E, k;
    int32_t *idx;
    float *w;
    WsHeader *hdr;
    unsigned long long wait_ns;
};

__device__ __forceinline__ void tma_2d(void *dst, const CUtensorMap *map, int x, int y,
                                       uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}

// hi(v) (low 13 significand bits cleared) and lo(v) = v - hi(v), four at once.
__device__ __forceinline__ void split4(const float4 v, float4 &hi, float4 &lo) {
    hi.x = __uint_as_float(__float_as_uint(v.x) & 0xFFFFE000u);
    hi.y = __uint_as_float(__float_as_uint(v.y) & 0xFFFFE000u);
    hi.z = __uint_as_float(__float_as_uint(v.z) & 0xFFFFE000u);
    hi.w = __uint_as_float(__float_as_uint(v.w) & 0xFFFFE000u);
    lo = make_float4(v.x - hi.x, v.y - hi.y, v.z - hi.z, v.w - hi.w);
}

__global__ void __cluster_dims__(1, kSplit, 1) __launch_bounds__(kThreads, 1)
    router_tc_kernel(const __grid_constant__ Params p) {
    pdl_enter();
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);  // [kStages] a stage's tiles landed
    uint64_t *done = full + kStages;                      // [kStages] the MMAs reading the slot are complete
    uint64_t *splitb = done + kStages;                    // [kStages] the eight split warps are done with it
    uint64_t *accfree = splitb + kStages;                 // [3] an accumulator has been added to registers
    uint64_t *fin = accfree + 3;                          // every MMA complete
    uint32_t *tmem_ptr = reinterpret_cast<uint32_t *>(fin + 1);
    volatile int *failed = reinterpret_cast<volatile int *>(tmem_ptr + 2);
    uint64_t *pgot = reinterpret_cast<uint64_t *>(tmem_ptr + 4);  // the four quarters of my tokens
    uint32_t *flags_in = reinterpret_cast<uint32_t *>(pgot + 1);   // [kSplit] each sender's flag
    uint8_t *ring = smem + kHead;                   // copy ring
    uint8_t *lobuf = ring + kStages * kStage;       // two lo buffers
    namespace cg = cooperative_groups;
    cg::cluster_group cl = cg::this_cluster();
    const int r = int(cl.block_rank());
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int t0 = blockIdx.x * kTM;
    const int kq = p.H / kSplit, kbeg = r * kq, nst = kq / kBK;
    const uint64_t deadline = global_timer_ns() + p.wait_ns;

    if (tid == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(full + i, 1);            // the copying thread's arrival + the tiles' bytes
            mbar_init(done + i, 1);            // the stage's MMAs (commit)
            mbar_init(splitb + i, kSplitWarps);  // one arrival per split warp
        }
        for (int i = 0; i < 3; ++i) mbar_init(accfree + i, kSplitWarps);
        mbar_init(fin, 1);
        mbar_init(pgot, 1);
        *failed = 0;
        fence_mbar_init();
    }
    // three accumulators of 128 fp32 columns, D[128 tokens][128 experts]
    // (512 columns allocated): stage st accumulates into buffer st % 3 from
    // zero, and the split warps add stage st - 2 into fp32 registers while
    // the MMAs of stages st - 1 and st run
    constexpr uint32_t kCols = 4 * kEN;
    if (warp == 0) tc::tmem_alloc(tmem_ptr, kCols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t taddr = *tmem_ptr;

    auto issue = [&](int st) {  // thread 0: stage st's two tiles into slot st % kStages
        const int slot = st % kStages;
        uint8_t *dst = ring + slot * kStage;
        mbar_arrive_expect_tx(full + slot, 2 * kTile);
        tma_2d(dst, &p.mx, kbeg + st * kBK, t0, full + slot);
        tma_2d(dst + kTile, &p.mw, kbeg + st * kBK, 0, full + slot);
    };
    if (tid == 0)
        for (int st = 0; st < kStages && st < nst; ++st) issue(st);
    int issued = kStages < nst ? kStages : nst;

    // split warp w: accumulator lanes and columns of quadrant w % 4, half w / 4
    const uint32_t lane_off = (uint32_t((warp & 3) * 32) << 16) + uint32_t((warp >> 2) * 64);
    float racc[64];
#pragma unroll
    for (int j = 0; j < 64; ++j) racc[j] = 0.f;
    auto add_stage = [&](int st) {  // stage st's accumulator into racc (its MMAs are complete)
        const uint32_t lb = taddr + uint32_t(st % 3) * kEN + lane_off;
#pragma unroll
        for (int c0 = 0; c0 < 64; c0 += 8) {
            float v[8];
            tc::tmem_ld8(lb + c0, v);
#pragma unroll
            for (int j = 0; j < 8; ++j) racc[c0 + j] += v[j];
        }
    };
    // stage st - 2's MMAs complete: its copy slot is refilled (thread 0), its
    // lo buffer (stage st's) is free, and its accumulator is added and released
    auto retire = [&](int st2) {
        const int ps = st2 % kStages;
        if (!mbar_wait(done + ps, uint32_t(st2 / kStages) & 1u, deadline)) *failed = 1;
        if (tid == 0 && st2 + kStages < nst && *failed == 0) {
            issue(st2 + kStages);
            ++issued;
        }
        tc::fence_after_sync();
        add_stage(st2);
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(accfree + st2 % 3);
    };

    if (warp < kSplitWarps) {
        // ---- split warps: every thread splits its share of each stage's tiles
        // and adds finished accumulators; no CTA-wide barrier in the loop
        for (int st = 0; st < nst; ++st) {
            const int slot = st % kStages;
            uint8_t *base = ring + slot * kStage;
            uint8_t *lo = lobuf + (st & 1) * kLo;
            if (st >= 2) retire(st - 2);
            if (!mbar_wait(full + slot, uint32_t(st / kStages) & 1u, deadline)) *failed = 1;
            // hi back into the x and Wr tiles, lo into the stage's lo buffer
            float4 *t = reinterpret_cast<float4 *>(base);
            float4 *tl = reinterpret_cast<float4 *>(lo);
#pragma unroll 4
            for (int i = tid; i < 2 * kTile / 16; i += kSplitWarps * 32) {
                float4 hi, lv;
                split4(t[i], hi, lv);
                t[i] = hi;
                tl[i] = lv;
            }
            fence_proxy_async_smem();  // generic stores before the MMA's async-proxy reads
            __syncwarp();
            if (lane == 0) mbar_arrive(splitb + slot);
        }
        if (nst > 1) retire(nst - 2);
        if (nst > 0) retire(nst - 1);
    } else {
        // ---- MMA warp: stage st's twelve MMAs once the eight split warps are
        // done with its slot and stage st - 3's accumulator buffer is free; the
        // whole warp walks the loop, one elected lane issues
        uint32_t is = 0;
        asm volatile("{\n\t.reg .pred P;\n\telect.sync _|P, 0xffffffff;\n\tselp.u32 %0, 1, 0, P;\n\t}"
                     : "=r"(is));
        const bool leader = is != 0u;
        const uint32_t idesc = tc::idesc_tf32_f32(kTM, kEN);
        for (int st = 0; st < nst; ++st) {
            const int slot = st % kStages;
            bool ok = mbar_wait(splitb + slot, uint32_t(st / kStages) & 1u, deadline);
            if (st >= 3) ok = mbar_wait(accfree + st % 3, uint32_t(st / 3 - 1) & 1u, deadline) && ok;
            if (!__all_sync(0xffffffffu, ok)) {
                *failed = 1;
                break;  // no more MMAs: the split warps' waits then run out as well
            }
            tc::fence_after_sync();
            if (leader) {
                uint8_t *base = ring + slot * kStage;
                uint8_t *lo = lobuf + (st & 1) * kLo;
                const uint32_t a = smem_addr(base), al = smem_addr(lo);
                const uint64_t dx = tc::smem_desc_sw128(a), dw = tc::smem_desc_sw128(a + kTile);
                const uint64_t dxl = tc::smem_desc_sw128(al), dwl = tc::smem_desc_sw128(al + kTile);
                const uint32_t dacc = taddr + uint32_t(st % 3) * kEN;
#pragma unroll
                for (int kk = 0; kk < kBK / 8; ++kk) {  // K = 8 per MMA: 32 bytes (2 in the address field)
                    const uint64_t o = uint64_t(2 * kk);
                    tc::mma_tf32(dacc, dx + o, dw + o, idesc, kk > 0);
                    tc::mma_tf32(dacc, dxl + o, dw + o, idesc, true);
                    tc::mma_tf32(dacc, dx + o, dwl + o, idesc, true);
                }
                tc::commit_arrive(done + slot);
            }
            __syncwarp();
        }
        if (leader) tc::commit_arrive(fin);
        __syncwarp();
        if (!mbar_wait(fin, 0, deadline)) *failed = 1;
    }
    // copies still in flight after a time-out must land before the ring is reused
    __syncthreads();
    if (tid == 0) {
        const uint64_t limit = global_timer_ns() + p.wait_ns;
        for (int i = 0; i < kStages && i < issued; ++i) {
            const int st = issued - 1 - i;
            mbar_wait(full + st % kStages, uint32_t(st / kStages) & 1u, limit);
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 0) tc::tmem_dealloc(taddr, kCols);

    // The four K quarters of CTA r's 32 tokens land in its ring (free once
    // every CTA of the cluster is past its loop): split warp w sends its 64
    // partial columns of token row 32 (w % 4) + lane, owned by CTA w % 4, as
    // 16-byte asynchronous stores completing on the owner's barrier, and
    // every CTA sends each owner its flag the same way.
    float *recv = reinterpret_cast<float *>(ring);  // [kSplit][kTok][kPS]
    constexpr uint32_t kRecvBytes = uint32_t(kSplit) * kTok * kEN * 4u + uint32_t(kSplit) * 4u;
    if (tid == 0) mbar_arrive_expect_tx(pgot, kRecvBytes);
    cl.sync();  // every CTA's ring is free and its barrier armed
    if (warp < kSplitWarps) {
        const int owner = warp & 3;
        float *dst = recv + (size_t(r) * kTok + lane) * kPS + (warp >> 2) * 64;
#pragma unroll
        for (int j = 0; j < 16; ++j)
            st_async_v4f(dst + 4 * j, racc[4 * j], racc[4 * j + 1], racc[4 * j + 2], racc[4 * j + 3],
                               pgot, owner);
    }
    if (tid == 0)
#pragma unroll
        for (int q = 0; q < kSplit; ++q) st_async_u32(flags_in + r, uint32_t(*failed), pgot, q);
    if (warp >= kSplitWarps) return;
    const bool got = mbar_wait_cluster(pgot, 0u, deadline + p.wait_ns);
    bool any_failed = !got;
#pragma unroll
    for (int q = 0; q < kSplit; ++q) any_failed |= flags_in[q] != 0u;
    if (any_failed) {
        if (tid == 0) record_status(p.hdr, MOE_ERR_TIMEOUT, 30 + r);
        return;
    }
    // CTA r sums the quarters of its tokens in rank order: warp v takes tokens
    // v, v + 8, ..., lane L experts L + 32 s
    constexpr int kTW = kTok / kSplitWarps;      // tokens per split warp
    constexpr int kEL = kEN / 32;                // experts per lane
    float part[kTW][kEL][kSplit];
#pragma unroll
    for (int i = 0; i < kTW; ++i)
#pragma unroll
        for (int s = 0; s < kEL; ++s)
#pragma unroll
            for (int q = 0; q < kSplit; ++q)
                part[i][s][q] = recv[(size_t(q) * kTok + warp + kSplitWarps * i) * kPS + lane + 32 * s];
    // the warp's kTW tokens ranked together (interleaved rounds)
    float lg[kTW][kEL];
    int32_t *oi[kTW];
    float *ow[kTW];
    bool oo[kTW];
#pragma unroll
    for (int i = 0; i < kTW; ++i) {
        const int t = t0 + r * kTok + warp + kSplitWarps * i;
        oo[i] = t < p.T;
        oi[i] = p.idx + size_t(oo[i] ? t : 0) * p.k;
        ow[i] = p.w + size_t(oo[i] ? t : 0) * p.k;
#pragma unroll
        for (int s = 0; s < kEL; ++s) {
            const int e = lane + 32 * s;
            float v = part[i][s][0];
#pragma unroll
            for (int q = 1; q < kSplit; ++q) v += part[i][s][q];
            lg[i][s] = v + (p.bias && e < p.E ? p.bias[e] : 0.f);
        }
    }
    warp_topk_multi<kEL, kTW>(lg, p.E, p.k, oi, ow, oo);
}

}  // namespace rtc

bool router_tc_supported(int T, int H, int E) {
    return T >= 256 && E <= rtc::kEN && H % (rtc::kSplit * rtc::kBK) == 0;
}

cudaError_t init_router_tc() {
    return cudaFuncSetAttribute(rtc::router_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                rtc::kSmem);
}

cudaError_t launch_router_tc(const float *x, const float *Wr, const float *bias, int T, int H, int E,
                             int k, int32_t *idx, float *w, WsHeader *hdr,
                             unsigned long long wait_ns, cudaStream_t s) {
    using namespace rtc;
    Params p = {};
    if (!encode_fp32_sw128_map(&p.mx, x, T, H, kTM) || !encode_fp32_sw128_map(&p.mw, Wr, E, H, kEN))
        return cudaErrorInvalidValue;
    p.bias = bias;
    p.T = T;
    p.H = H;
    p.E = E;
    p.k = k;
    p.idx = idx;
    p.w = w;
    p.hdr = hdr;
    p.wait_ns = wait_ns;
    launch_pdl(router_tc_kernel, dim3((T + kTM - 1) / kTM, kSplit), dim3(kThreads), size_t(kSmem), s, p);
    return cudaGetLastError();
}

}  // namespace moeq4k
