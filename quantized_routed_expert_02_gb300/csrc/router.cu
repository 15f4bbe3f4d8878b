// Router: fp32 logits, softmax over all experts, top-k, renormalisation.
//
// forward_qwen3_moe_cuda_traced.rs (aprender-serve 0.34.0), doc of
// forward_qwen3_moe_cuda_traced_with_plan: the router stage is the k
// post-softmax, renormalised top-k weights of a token.  Softmax is monotone,
// so the top-k of p is the top-k of the logits; after renormalisation the
// full-softmax denominator cancels and w_j = exp(l_j - l_max) / sum over the
// selected slots of exp(l - l_max).
#include <cooperative_groups.h>

#include <algorithm>

#include "async_copy.cuh"
#include "common.cuh"
#include "kernels.cuh"

namespace moeq4k {

// ---------------------------------------------------------------------------
// 3..255 tokens: a cluster of kCS CTAs per tile of TT tokens; CTA r takes
// expert group r (EG = ceil(E / kCS) consecutive rows of Wr).
//  - Copies: per K chunk of kKC floats, one TMA box of the group's Wr rows
//    (requested before the wait on the preceding launch) and one of the
//    tile's x rows, into a ring of shared-memory slots, every slot requested
//    at once (rows past E or T arrive as zeros).
//  - Dots: the eight warps split each chunk's 64 float4 columns, warp v
//    taking columns 8v..8v+7; lane = (column, expert subset): lane L dots
//    column 8v + (L & 7) of rows L/8, L/8 + 4, ... of the group with the
//    column of every token.  Each shared-memory byte is read about once.
//  - Sums: a reduce-scatter over the eight column lanes (fixed butterfly),
//    then the eight warps' partials added in warp order, plus the bias.
//  - Exchange: warp t of every group CTA sends its logits of token t, and
//    its failure flag, into the shared memory of CTA t of the cluster with
//    st.async, completing as transaction bytes on CTA t's barrier; CTA t
//    waits for its E + 8 words.
//  - Ranking: the logits become order-preserving keys (logit_key: NaN below
//    every number, as in warp_topk); a thread pair per expert (one thread
//    above 128 experts) counts the experts that beat it in the order (key
//    descending, index ascending); ranks below k name the selection in
//    order, and one warp renormalises.
// One launch, no logits in global memory, a fixed summation order.  Every
// wait is bounded; a timed-out wait records MOE_ERR_TIMEOUT and the cluster
// writes no routing for the tile.
// ---------------------------------------------------------------------------
namespace rcl {
constexpr int kCS = 8;                // CTAs per cluster: expert groups
constexpr int kKC = 256;              // K per chunk (floats): one box row of 1 KB
constexpr int kCols = kKC / 4;        // float4 columns per chunk
constexpr int kMaxSlots = 16;         // ring slots
constexpr int kMaxEG = kMaxE / kCS;   // rows of Wr per group (32)
constexpr int kMaxTT = 8;             // tokens per tile
constexpr int kFlagOff = 8 * (kMaxSlots + 1);             // after full[], got: failed, flags_in[kCS]
constexpr int kInboxOff = 256;                            // the ranked token's logits
constexpr int kRedOff = kInboxOff + kMaxE * 4;            // [8 warps][kMaxEG * kMaxTT]
constexpr int kSelOff = kRedOff + 8 * kMaxEG * kMaxTT * 4;  // the selection, in rank order
constexpr int kHead = (kSelOff + 2 * kMaxK * 4 + 1023) / 1024 * 1024;
constexpr int kRingSolo = 200 * 1024;  // ring bytes when the clusters fit one CTA per SM
constexpr int kRingPair = 100 * 1024;  // ... and when two CTAs share an SM
constexpr int kSmemMax = 1024 + kHead + kRingSolo;  // + slack to align the base to 1024
static_assert(kFlagOff + 4 * (1 + kCS) <= kInboxOff, "barriers and flags");
static_assert(kSmemMax <= 232448, "shared memory of one CTA");

struct Params {
    CUtensorMap mx, mw;  // x [T][H], Wr [E][H] fp32; boxes kKC x TT rows, kKC x EG rows
    const float *bias;
    int T, H, E, k, nslots;
    int32_t *idx;
    float *w;
    WsHeader *hdr;
    unsigned long long wait_ns;
};

__device__ __forceinline__ void tma_box(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}

// Split cluster barrier, executed by every thread of the cluster: the
// arrive is relaxed (what other CTAs need to see before the wait returns is
// the mbarrier initialisation, which fence.mbarrier_init publishes at
// cluster scope); the wait returns once every thread has arrived.
__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Sum each of the V values of a lane over the eight lanes that share
// lane / 8 (lane bits 0-2), by a reduce-scatter in a fixed order.  After it,
// lane L holds the sums of the values V/8 * (L & 7) + i, i < V/8, in a[i]
// (V >= 8); for V = 4, a[0] holds value (L & 7) / 2.
template <int V, int N>  // one step: N values per lane -> N / 2 (or a plain butterfly at N = 1)
__device__ __forceinline__ void fold_step(float (&a)[V], int lane, int o) {
    if constexpr (N > 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < N / 2; ++i) {
            const float send = up ? a[i] : a[i + N / 2];
            const float recv = __shfl_xor_sync(0xffffffffu, send, o);
            a[i] = (up ? a[i + N / 2] : a[i]) + recv;
        }
    } else {
        a[0] += __shfl_xor_sync(0xffffffffu, a[0], o);
    }
}
template <int V>
__device__ __forceinline__ void fold8(float (&a)[V], int lane) {
    static_assert(V >= 4 && (V & (V - 1)) == 0, "a power of two, at least 4");
    fold_step<V, V>(a, lane, 4);
    fold_step<V, V / 2>(a, lane, 2);
    fold_step<V, (V / 4 > 1 ? V / 4 : 1)>(a, lane, 1);
}
}  // namespace rcl

template <int TT, int NEL>
__global__ void __cluster_dims__(rcl::kCS, 1, 1) __launch_bounds__(256)
    router_cluster_kernel(const __grid_constant__ rcl::Params p) {
    using namespace rcl;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(sm);  // [nslots] a chunk's boxes landed
    uint64_t *got = full + kMaxSlots;                   // the eight groups' logits of my token
    int *failed = reinterpret_cast<int *>(sm + kFlagOff);  // a wait of this CTA timed out
    int *flags_in = failed + 1;  // [kCS] group g's flag for my token (1: its waits timed out)
    float *inbox = reinterpret_cast<float *>(sm + kInboxOff);
    float *red = reinterpret_cast<float *>(sm + kRedOff);
    float *sel_v = reinterpret_cast<float *>(sm + kSelOff);
    int *sel_i = reinterpret_cast<int *>(sel_v + kMaxK);
    float *ring = reinterpret_cast<float *>(sm + kHead);
    namespace cg = cooperative_groups;
    const int r = int(cg::this_cluster().block_rank());
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int EG = (p.E + kCS - 1) / kCS;
    const int e0 = r * EG;
    const int ne = max(0, min(EG, p.E - e0));  // rows of this CTA's group
    const int t0 = blockIdx.y * TT;
    const int nt = min(TT, p.T - t0);          // tokens of this tile
    const int rows = EG + TT;                  // rows per ring slot: the Wr box, then the x box
    const int nch = p.H / kKC;
    const int nslots = p.nslots;
    const uint32_t wbytes = ne > 0 ? uint32_t(EG) * kKC * 4u : 0u;
    const uint32_t chunk_bytes = wbytes + uint32_t(TT) * kKC * 4u;
    const uint64_t deadline = global_timer_ns() + p.wait_ns;
    auto slot_of = [&](int c) { return ring + size_t(c % nslots) * rows * kKC; };

    const int npre = min(nslots, nch);
    if (tid == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.mx)) : "memory");
        for (int i = 0; i < nslots; ++i) mbar_init(full + i, 1);
        // my token's logits: E words from the groups and one flag word from each
        mbar_init(got, 1);
        *failed = 0;
        fence_mbar_init();
        if (r < nt) mbar_arrive_expect_tx(got, uint32_t(p.E + kCS) * 4u);
        for (int c = 0; c < npre; ++c) {
            mbar_arrive_expect_tx(full + c, chunk_bytes);
            if (ne > 0) tma_box(slot_of(c), &p.mw, c * kKC, e0, full + c);
        }
    }
    __syncthreads();   // every slot's byte count is set before any x box can land
    cluster_arrive();  // this CTA's barriers exist; waited for before the exchange
    pdl_enter();      // x, idx and w belong to the stream's order from here
    if (tid == 32)
        for (int c = 0; c < npre; ++c) tma_box(slot_of(c) + EG * kKC, &p.mx, c * kKC, t0, full + c);
    int issued = npre;  // chunks requested (thread 0's count)

    float acc[NEL * TT];
#pragma unroll
    for (int i = 0; i < NEL * TT; ++i) acc[i] = 0.f;
    const int q = 8 * warp + (lane & 7);  // this lane's float4 column of a chunk
    const int g = lane >> 3;              // ... and expert subset: rows g, g + 4, ...
    for (int c = 0; c < nch; ++c) {
        const int slot = c % nslots;
        // after a time-out every later wait returns at once (the deadline has passed)
        if (!mbar_wait(full + slot, uint32_t(c / nslots) & 1u, deadline)) atomicExch(failed, 1);
        const float4 *wb = reinterpret_cast<const float4 *>(ring + size_t(slot) * rows * kKC);
        const float4 *xb = wb + EG * kCols;
        float4 xv[TT];
#pragma unroll
        for (int t = 0; t < TT; ++t) xv[t] = xb[t * kCols + q];
#pragma unroll
        for (int m = 0; m < NEL; ++m) {
            const int el = g + 4 * m;
            if (el < ne) {
                const float4 a = wb[el * kCols + q];
#pragma unroll
                for (int t = 0; t < TT; ++t) {
                    float s = acc[m * TT + t];
                    s = fmaf(a.x, xv[t].x, s);
                    s = fmaf(a.y, xv[t].y, s);
                    s = fmaf(a.z, xv[t].z, s);
                    s = fmaf(a.w, xv[t].w, s);
                    acc[m * TT + t] = s;
                }
            }
        }
        if (nch > nslots) {  // the ring wraps: refill this slot once every warp is done with it
            __syncthreads();
            if (tid == 0 && c + nslots < nch && *reinterpret_cast<volatile int *>(failed) == 0) {
                const int cn = c + nslots;
                mbar_arrive_expect_tx(full + slot, chunk_bytes);
                if (ne > 0) tma_box(slot_of(cn), &p.mw, cn * kKC, e0, full + slot);
                tma_box(slot_of(cn) + EG * kKC, &p.mx, cn * kKC, t0, full + slot);
                ++issued;
            }
        }
    }
    // fold the column lanes; lane L now holds values V/8 * (L & 7) + i (value
    // m * TT + t is row g + 4m, token t), or value (L & 7) / 2 when V = 4
    constexpr int V = NEL * TT;
    fold8<V>(acc, lane);
    {
        float *rw = red + warp * (kMaxEG * kMaxTT);  // [EG * TT] of this warp, row-major (row, token)
        if constexpr (V >= 8) {
#pragma unroll
            for (int i = 0; i < V / 8; ++i) {
                const int v = (V / 8) * (lane & 7) + i, m = v / TT, t = v - m * TT;
                const int el = g + 4 * m;
                if (el < EG) rw[el * TT + t] = acc[i];
            }
        } else if ((lane & 1) == 0) {
            const int v = (lane & 7) >> 1, m = v / TT, t = v - m * TT;
            const int el = g + 4 * m;
            if (el < EG) rw[el * TT + t] = acc[0];
        }
    }
    __syncthreads();
    const bool bad = *reinterpret_cast<volatile int *>(failed) != 0;
    if (bad && tid == 0) {
        // copies still in flight land before the CTA's shared memory is released:
        // the latest phase of every slot
        const uint64_t limit = global_timer_ns() + p.wait_ns;
        for (int i = 0; i < nslots && i < issued; ++i) {
            const int cc = issued - 1 - i;
            mbar_wait(full + cc % nslots, uint32_t(cc / nslots) & 1u, limit);
        }
    }
    cluster_wait();  // every CTA's barriers are initialised
    namespace cgx = cooperative_groups;
    cgx::cluster_group cl = cgx::this_cluster();
    // warp t sends token t's logits of this group, and this group's flag, to CTA t
    if (warp < nt) {
        const int t = warp;
        for (int el = lane; el < ne; el += 32) {
            float sum = 0.f;
#pragma unroll
            for (int v = 0; v < 8; ++v) sum += red[v * (kMaxEG * kMaxTT) + el * TT + t];
            sum += p.bias ? p.bias[e0 + el] : 0.f;
            st_async_u32(inbox + e0 + el, __float_as_uint(sum), got, t);
        }
        if (lane == 0) st_async_u32(flags_in + r, bad ? 1u : 0u, got, t);
    }
    if (r >= nt) return;  // no token of this tile is ranked here; nothing is sent to this CTA
    // CTA r ranks token t0 + r once the eight groups' logits are in
    if (!mbar_wait_cluster(got, 0u, deadline + p.wait_ns)) {
        if (tid == 0) record_status(p.hdr, MOE_ERR_TIMEOUT, 41);
        return;
    }
    bool any_failed = false;
#pragma unroll
    for (int g2 = 0; g2 < kCS; ++g2) any_failed |= flags_in[g2] != 0;
    if (any_failed) {
        if (tid == 0) record_status(p.hdr, MOE_ERR_TIMEOUT, 40);
        return;
    }
    const int E = p.E, k = p.k;
    const int E4 = (E + 3) & ~3;
    // the logits as order-preserving keys (logit_key: -0 as +0, NaN below
    // every number, as warp_topk ranks them); pads past E lose every comparison
    uint32_t *keys = reinterpret_cast<uint32_t *>(inbox);
    if (tid < E4) keys[tid] = tid < E ? logit_key(inbox[tid]) : 0u;
    __syncthreads();
    {
        // rank of expert e in the order (key descending, index ascending): the
        // experts that beat it, counted by two threads (halves of the list) for
        // E <= 128, else by one
        const bool pair = E <= 128;
        const int e = pair ? tid >> 1 : tid;
        const int nq = E4 / 4, half = pair ? (nq + 1) / 2 : nq;
        const int q0 = pair && (tid & 1) ? half : 0, q1 = pair && !(tid & 1) ? half : nq;
        const uint32_t v = e < E ? keys[e] : 0u;
        int rank = 0;
        const uint4 *in4 = reinterpret_cast<const uint4 *>(keys);
#pragma unroll 4
        for (int j4 = q0; j4 < q1; ++j4) {
            const uint4 u = in4[j4];
            const int j = 4 * j4;
            rank += (u.x > v || (u.x == v && j < e)) ? 1 : 0;
            rank += (u.y > v || (u.y == v && j + 1 < e)) ? 1 : 0;
            rank += (u.z > v || (u.z == v && j + 2 < e)) ? 1 : 0;
            rank += (u.w > v || (u.w == v && j + 3 < e)) ? 1 : 0;
        }
        if (pair) rank += __shfl_xor_sync(0xffffffffu, rank, 1);
        if (e < E && rank < k && (!pair || (tid & 1) == 0)) {
            sel_v[rank] = logit_of_key(v);
            sel_i[rank] = e;
        }
    }
    __syncthreads();
    if (warp == 0) {
        const int t = t0 + r;
        const float vmax = sel_v[0];
        const float ex = lane < k ? expf(sel_v[lane] - vmax) : 0.f;
        const float z = warp_sum(ex);
        if (lane < k) {
            p.idx[size_t(t) * k + lane] = sel_i[lane];
            p.w[size_t(t) * k + lane] = ex / z;
        }
    }
}

// ---------------------------------------------------------------------------
// One or two tokens: one CTA per expert row, each thread a strided share of
// the row (float4 steps), reduced in a fixed order (warp shuffles, then the
// eight warp sums in order), so every row of Wr is read by 256 threads at
// once.  The last CTA to store its logits ranks them (top-k + renormalise):
// one launch for the whole router.
// ---------------------------------------------------------------------------
template <int kTT>
__global__ void __launch_bounds__(256) router_row_kernel(const float *__restrict__ x,
                                                         const float *__restrict__ Wr,
                                                         const float *__restrict__ bias, int T,
                                                         int H, int E, int k,
                                                         float *__restrict__ logits,
                                                         int32_t *__restrict__ idx,
                                                         float *__restrict__ w, WsHeader *hdr) {
    pdl_enter();
    __shared__ float part[kTT][8];
    __shared__ float lg[kTT][kMaxE];
    __shared__ int last;
    const int e = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float4 *wr = reinterpret_cast<const float4 *>(Wr + size_t(e) * H);
    float acc[kTT];
#pragma unroll
    for (int i = 0; i < kTT; ++i) acc[i] = 0.f;
    for (int c = threadIdx.x; c < H / 4; c += blockDim.x) {
        const float4 a = __ldg(wr + c);
#pragma unroll
        for (int i = 0; i < kTT; ++i) {
            if (i < T) {
                const float4 b = __ldg(reinterpret_cast<const float4 *>(x + size_t(i) * H) + c);
                acc[i] = fmaf(a.x, b.x, acc[i]);
                acc[i] = fmaf(a.y, b.y, acc[i]);
                acc[i] = fmaf(a.z, b.z, acc[i]);
                acc[i] = fmaf(a.w, b.w, acc[i]);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < kTT; ++i) {
        const float s = warp_sum(acc[i]);
        if (lane == 0) part[i][warp] = s;
    }
    __syncthreads();
    if (threadIdx.x < kTT && int(threadIdx.x) < T) {
        const int i = threadIdx.x;
        float s = 0.f;
        for (int ww = 0; ww < 8; ++ww) s += part[i][ww];
        logits[size_t(i) * E + e] = s + (bias ? bias[e] : 0.f);
        __threadfence();  // the logit is visible GPU-wide before this CTA is counted
    }
    __syncthreads();
    // The count starts every call at 0 (moe_workspace_init, then the ranking
    // CTA of each call sets it back), so exactly the last CTA to count itself
    // sees gridDim.x - 1 and every other logit is stored by then.  A count at
    // or past gridDim.x means the header was never initialised (or was
    // overwritten): that is recorded, and no CTA ranks logits it cannot
    // trust; the count stays off until the workspace is re-initialised.
    if (threadIdx.x == 0) {
        const unsigned long long prev = atomicAdd(&hdr->router_rows, 1ull);
        last = prev == gridDim.x - 1;
        if (prev >= gridDim.x)
            record_status(hdr, MOE_ERR_INTERNAL, 500000000 + int(prev % 1000000ull));
    }
    __syncthreads();
    if (!last) return;
    __threadfence();
    for (int i = threadIdx.x; i < T * E; i += blockDim.x) lg[i / E][i % E] = __ldcg(logits + i);
    __syncthreads();
    if (warp < T) warp_topk(&lg[warp][0], E, k, idx + size_t(warp) * k, w + size_t(warp) * k);
    if (threadIdx.x == 0) atomicExch(&hdr->router_rows, 0ull);  // every CTA has counted itself
}

// ---------------------------------------------------------------------------
// Large batches: logits of 32 tokens x all E experts per CTA as a shared-
// memory-tiled fp32 GEMM (each thread a 4 x 4 register tile, K in chunks of
// 32, double-buffered), then the top-k of each token by one warp from the
// CTA's logits in shared memory.
// ---------------------------------------------------------------------------
constexpr int kRT = 32;   // tokens per CTA
constexpr int kRE = 128;  // experts per pass
constexpr int kRK = 32;   // K per chunk
constexpr int kRouterBigSmem = int(sizeof(float)) * (2 * kRK * kRT + 2 * kRK * kRE + kRT * (kMaxE + 1));

__global__ void __launch_bounds__(256) router_big_kernel(const float *__restrict__ x,
                                                         const float *__restrict__ Wr,
                                                         const float *__restrict__ bias, int T,
                                                         int H, int E, int k,
                                                         int32_t *__restrict__ idx,
                                                         float *__restrict__ w) {
    pdl_enter();
    // dynamic shared memory: xs[2][kRK][kRT], ws[2][kRK][kRE] (k-major), lg[kRT][kMaxE + 1]
    extern __shared__ __align__(16) float rsm[];
    float (*xs)[kRK][kRT] = reinterpret_cast<float (*)[kRK][kRT]>(rsm);
    float (*ws)[kRK][kRE] = reinterpret_cast<float (*)[kRK][kRE]>(rsm + 2 * kRK * kRT);
    float (*lg)[kMaxE + 1] = reinterpret_cast<float (*)[kMaxE + 1]>(rsm + 2 * kRK * kRT + 2 * kRK * kRE);
    const int tid = threadIdx.x, ty = tid >> 5, tx = tid & 31;
    const int t0 = blockIdx.x * kRT;
    const int nchunk = H / kRK;
    for (int e0 = 0; e0 < E; e0 += kRE) {
        float acc[4][4] = {};
        auto load = [&](int c, int buf) {
            // x: 32 tokens x 32 k = 256 float4, one per thread
            {
                const int t = tid >> 3, q = tid & 7;
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (t0 + t < T) v = __ldg(reinterpret_cast<const float4 *>(x + size_t(t0 + t) * H + c * kRK) + q);
                xs[buf][4 * q + 0][t] = v.x;
                xs[buf][4 * q + 1][t] = v.y;
                xs[buf][4 * q + 2][t] = v.z;
                xs[buf][4 * q + 3][t] = v.w;
            }
            // Wr: 128 experts x 32 k = 1024 float4, four per thread
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int f = tid + 256 * r, e = f >> 3, q = f & 7;
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (e0 + e < E) v = __ldg(reinterpret_cast<const float4 *>(Wr + size_t(e0 + e) * H + c * kRK) + q);
                ws[buf][4 * q + 0][e] = v.x;
                ws[buf][4 * q + 1][e] = v.y;
                ws[buf][4 * q + 2][e] = v.z;
                ws[buf][4 * q + 3][e] = v.w;
            }
        };
        load(0, 0);
        __syncthreads();
        for (int c = 0; c < nchunk; ++c) {
            const int buf = c & 1;
            if (c + 1 < nchunk) load(c + 1, buf ^ 1);
            // two-level sum: a fresh partial per 32-wide chunk keeps the fp32
            // rounding of the 2048-term dot products small
            float part[4][4] = {};
#pragma unroll 8
            for (int kk = 0; kk < kRK; ++kk) {
                const float4 a = *reinterpret_cast<const float4 *>(&xs[buf][kk][ty * 4]);
                const float4 b = *reinterpret_cast<const float4 *>(&ws[buf][kk][tx * 4]);
                const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) part[i][j] = fmaf(av[i], bv[j], part[i][j]);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] += part[i][j];
            __syncthreads();
        }
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int e = e0 + tx * 4 + j;
                if (e < E) lg[ty * 4 + i][e] = acc[i][j] + (bias ? bias[e] : 0.f);
            }
        __syncthreads();
    }
    // top-k: warp ty takes tokens ty, ty+8, ty+16, ty+24
    for (int i = ty; i < kRT; i += 8) {
        const int t = t0 + i;
        if (t < T) warp_topk(&lg[i][0], E, k, idx + size_t(t) * k, w + size_t(t) * k);
    }
}

cudaError_t init_router() {
    cudaError_t err = cudaFuncSetAttribute(router_big_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           kRouterBigSmem);
    if (err != cudaSuccess) return err;
    for (void *fn : {(void *)router_cluster_kernel<1, 4>, (void *)router_cluster_kernel<2, 4>,
                     (void *)router_cluster_kernel<4, 4>, (void *)router_cluster_kernel<8, 4>,
                     (void *)router_cluster_kernel<1, 8>, (void *)router_cluster_kernel<2, 8>,
                     (void *)router_cluster_kernel<4, 8>, (void *)router_cluster_kernel<8, 8>}) {
        err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, rcl::kSmemMax);
        if (err != cudaSuccess) return err;
    }
    return cudaSuccess;
}

// Tokens per cluster tile for 3..255 tokens: the largest of 8, 4, 2 that
// still gives at least 8 tiles (64 CTAs), else 1.  More tokens per tile
// means fewer reads of every group's Wr rows; on one SM the bytes arrive at
// a few tens of GB/s, so the tile stays small enough to spread over 64 SMs
// or more (measured at 64 tokens: 8 tiles of 8 beat 16 tiles of 4 by 3 %
// of the layer call, at 32 A22B tokens by 1.5 %).
static int router_tile_tokens(int T) {
    for (int tt = 8; tt > 1; tt >>= 1)
        if ((T + tt - 1) / tt >= 8) return tt;
    return 1;
}

template <int NEL>
static void launch_cluster(int tt, dim3 grid, size_t smem, cudaStream_t s, const rcl::Params &p) {
    const dim3 blk(256);
    switch (tt) {
        case 8: launch_pdl(router_cluster_kernel<8, NEL>, grid, blk, smem, s, p); break;
        case 4: launch_pdl(router_cluster_kernel<4, NEL>, grid, blk, smem, s, p); break;
        case 2: launch_pdl(router_cluster_kernel<2, NEL>, grid, blk, smem, s, p); break;
        default: launch_pdl(router_cluster_kernel<1, NEL>, grid, blk, smem, s, p); break;
    }
}

cudaError_t launch_router(const float *x, const float *Wr, const float *bias, int T, int H, int E,
                          int k, int32_t *idx, float *w, float *logits, WsHeader *hdr, int num_sms,
                          unsigned long long wait_ns, cudaStream_t s) {
    dim3 blk(256);
    // T >= 256, E <= 128: tensor cores (three-pass TF32, router_tc.cu)
    if (router_tc_supported(T, H, E))
        return launch_router_tc(x, Wr, bias, T, H, E, k, idx, w, hdr, wait_ns, s);
    if (T >= 256) {
        launch_pdl(router_big_kernel, dim3((T + kRT - 1) / kRT), dim3(blk), size_t(kRouterBigSmem), s, x, Wr, bias, T, H, E, k, idx, w);
        return cudaGetLastError();
    }
    if (T <= 2) {
        launch_pdl(router_row_kernel<2>, dim3(E), dim3(blk), size_t(0), s, x, Wr, bias, T, H, E, k, logits, idx, w, hdr);
        return cudaGetLastError();
    }
    using namespace rcl;
    const int tt = router_tile_tokens(T);
    const int tiles = (T + tt - 1) / tt;
    const int EG = (E + kCS - 1) / kCS;
    const int slot_bytes = (EG + tt) * kKC * 4;
    const int budget = tiles * kCS <= num_sms ? kRingSolo : kRingPair;
    const int nslots = std::min({H / kKC, kMaxSlots, budget / slot_bytes});
    if (nslots < 1) return cudaErrorInvalidValue;
    Params p = {};
    if (!encode_fp32_box_map(&p.mx, x, T, H, kKC, tt) || !encode_fp32_box_map(&p.mw, Wr, E, H, kKC, EG))
        return cudaErrorInvalidValue;
    p.bias = bias;
    p.T = T;
    p.H = H;
    p.E = E;
    p.k = k;
    p.nslots = nslots;
    p.idx = idx;
    p.w = w;
    p.hdr = hdr;
    p.wait_ns = wait_ns;
    const size_t smem = size_t(1024 + kHead) + size_t(nslots) * slot_bytes;
    const dim3 grid(kCS, tiles);
    if (EG <= 16)
        launch_cluster<4>(tt, grid, smem, s, p);
    else
        launch_cluster<8>(tt, grid, smem, s, p);
    return cudaGetLastError();
}

}  // namespace moeq4k
