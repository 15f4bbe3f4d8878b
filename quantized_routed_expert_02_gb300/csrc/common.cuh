// Shared device helpers and the workspace layout of the moeq4k library.
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "moeq4k.h"

namespace moeq4k {

constexpr int kQK = 256;          // weights per Q4_K block
constexpr int kBlockBytes = 144;  // bytes per Q4_K block
constexpr int kMaxE = 256;
constexpr int kMaxK = 32;
constexpr int kMaxHI = 8192;

// ---------------------------------------------------------------------------
// Workspace layout (all regions 256-byte aligned).  moe_workspace_init zeroes
// the whole workspace.  The header and the tag region must keep their
// contents between calls; everything else is scratch rewritten by every call.
// ---------------------------------------------------------------------------
struct WsHeader {
    uint32_t status;                 // first device-side moe_status recorded (sticky)
    int32_t detail;                  // value that caused it
    // Single-token kernel: every CTA adds 1 per call, so during the n-th call
    // since initialisation (n = 0, 1, ...) a CTA's add returns a value in
    // [n * nblk, (n + 1) * nblk); the call tags what it publishes with n + 1.
    unsigned long long cta_calls;
    // Single-token kernel: every CTA adds 1 (release) once its values of h
    // are stored, so the count reaches tag * nblk when the call's h is
    // complete.
    unsigned long long rows_done;
    uint32_t pad1[2];
    int32_t tc_chunks;               // grouped GEMMs: expert chunks of the gate/up GEMM
    int32_t tc_chunks_dn;            //   and of the down GEMM (capacity <= 128 slots)
    // One- and two-token router: every CTA (one per expert) adds 1 once its
    // logits are stored; the CTA whose add returns E - 1 ranks them and sets
    // the count back to 0 for the next call (a count >= E at an add means an
    // uninitialised header and is recorded as MOE_ERR_INTERNAL).
    unsigned long long router_rows;
    uint32_t pad[52];
};

// One expert's chunk of at most 256 routed slots (prefill GEMM column tile).
struct TcChunk {
    int32_t e, tok_off, tok_cnt, pad;
};
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");

// Chunks of <= cap slots for each active expert, in active order, written by
// one warp (lanes take active experts in turns of 32; a warp scan gives each
// expert's first chunk); their number goes to *count.  `offs`: the experts'
// first sorted slots (E + 1 entries), `active`: the na active experts.
__device__ inline void warp_plan_chunks(const int32_t *offs, const int32_t *active, int na, int cap,
                                        TcChunk *chunks, int32_t *count) {
    const int lane = threadIdx.x & 31;
    int nc = 0;
    for (int base = 0; base < na; base += 32) {
        const int a = base + lane;
        const int e = a < na ? active[a] : 0;
        const int n = a < na ? offs[e + 1] - offs[e] : 0;
        const int mine = (n + cap - 1) / cap;
        int incl = mine;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += u;
        }
        for (int c = 0; c < mine; ++c) {
            TcChunk ch;
            ch.e = e;
            ch.tok_off = c * cap;
            ch.tok_cnt = min(cap, n - c * cap);
            ch.pad = 0;
            chunks[nc + incl - mine + c] = ch;
        }
        nc += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) *count = nc;
}

// A chunk plan the permutation launch may write on the way (cap 0: none).
struct ChunkPlan {
    int cap = 0;
    TcChunk *chunks = nullptr;
    int32_t *count = nullptr;
};

// Routed slots up to which the permutation runs as one CTA in one launch.
constexpr int kSmallPermSlots = 4096;

// Tag region of the single-token kernel, right after the header: the router
// logits, each a word (call tag << 32 | fp32 bits).  Place and size are the
// same for every shape, so the region never holds anything but tags (or the
// zeros of moe_workspace_init), and tags only grow between initialisations:
// a word left by an earlier call can never carry the current call's tag.
constexpr size_t kSyncWords = kMaxE;

// Slots per block of the permutation kernels.
constexpr int kPermSlots = 256;

struct WsLayout {
    size_t sync, blockcnt, slotpos, counts, offs, active, nactive, perm, h, o, logits, x16, h16, chunks, chunks_dn, ready,
        xn, xstage, ystage, total;
};

__host__ __device__ inline size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

inline WsLayout ws_layout(int T, int H, int E, int k, int I, bool host_staging) {
    WsLayout L;
    size_t off = sizeof(WsHeader);
    size_t pairs = size_t(T) * k;
    L.sync = off;    off = align256(off + sizeof(unsigned long long) * kSyncWords);
    L.counts = off;  off = align256(off + sizeof(int32_t) * E);
    L.offs = off;    off = align256(off + sizeof(int32_t) * (E + 1));
    L.active = off;  off = align256(off + sizeof(int32_t) * E);
    L.nactive = off; off = align256(off + sizeof(int32_t) * 4);
    // permutation: per-block expert counts (then their per-expert prefix) and
    // each slot's position in the sorted order
    L.blockcnt = off; off = align256(off + sizeof(int32_t) * ((pairs + kPermSlots - 1) / kPermSlots) * E);
    L.slotpos = off; off = align256(off + sizeof(int32_t) * pairs);
    L.logits = off;  off = align256(off + sizeof(float) * size_t(T) * E);
    L.perm = off;    off = align256(off + sizeof(int32_t) * pairs);
    L.h = off;       off = align256(off + sizeof(float) * pairs * I);
    L.o = off;       off = align256(off + sizeof(float) * pairs * H);
    L.x16 = off;     off = align256(off + 2 * pairs * H);                // fp16 activations, sorted rows
    L.h16 = off;     off = align256(off + 2 * pairs * I);                // fp16 SwiGLU output
    L.chunks = off;  off = align256(off + sizeof(TcChunk) * (pairs / 32 + E + 1));  // chunks of >= 32 slots
    L.chunks_dn = off; off = align256(off + sizeof(TcChunk) * (pairs / 32 + E + 1));
    L.ready = off;   off = align256(off + sizeof(uint32_t) * kMaxE);      // gate/up rows done per expert
    L.xn = off;      off = align256(off + sizeof(float) * size_t(T) * H);  // normed FFN input
    L.xstage = off;
    L.ystage = off;
    if (host_staging) {
        L.xstage = off; off = align256(off + sizeof(float) * size_t(T) * H);
        L.ystage = off; off = align256(off + sizeof(float) * size_t(T) * H);
    }
    L.total = off;
    return L;
}

// What the final store of an output value does besides storing it (the
// steps on the far side of the layer): add the residual stream
// (hidden += ffn_output) and copy one token's pre-residual output row to a
// capture buffer (the [H] FFN-output stage of a traced forward).
struct OutEpilogue {
    const float *residual = nullptr;  // [T,H] added to every output value, or null
    float *capture = nullptr;         // [H] receives token cap_t's pre-residual row, or null
    int cap_t = -1;
};

// The value to store at y[t*H + r] for the FFN output v.
__device__ __forceinline__ float epilogue_value(const OutEpilogue &ep, int t, int H, int r, float v) {
    if (ep.capture != nullptr && t == ep.cap_t) ep.capture[r] = v;
    return ep.residual != nullptr ? ep.residual[size_t(t) * H + r] + v : v;
}

// Programmatic dependent launch.  Every kernel of the library is launched
// with programmatic stream serialisation (launch_pdl below) and begins with
// pdl_enter(): it waits until the grids it depends on have completed and their
// writes are visible, then lets the next grid in the stream be launched, so
// that grid's launch and set-up overlap this one's tail instead of following
// its end.  Work that reads nothing a predecessor may write (an L2 prefetch
// of weights) may run between pdl_trigger() and pdl_wait().
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_enter() {
    pdl_wait();
    pdl_trigger();
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

// Record the first device-side error (later ones are dropped).
__device__ inline void record_status(WsHeader *hdr, moe_status s, int32_t detail) {
    if (atomicCAS(&hdr->status, 0u, uint32_t(s)) == 0u) {
        hdr->detail = detail;
    }
}

// ---------------------------------------------------------------------------
// Q4_K block pieces.  The 16-byte block head holds d, dmin and scales[12]:
//   head.x = d | dmin << 16, head.y = scales[0..3], head.z = scales[4..7],
//   head.w = scales[8..11] (little-endian bytes).
// Sub-block j < 4:  sc = scales[j] & 63,  m = scales[j+4] & 63
// Sub-block j >= 4: sc = (scales[j+4] & 15) | (scales[j-4] >> 6) << 4
//                   m  = (scales[j+4] >> 4) | (scales[j]   >> 6) << 4
// ---------------------------------------------------------------------------
__device__ __forceinline__ void q4k_scale_min(const uint4 &head, int j, float &sc, float &m) {
    uint32_t s, mm;
    if (j < 4) {
        s = (head.y >> (8 * j)) & 63u;
        mm = (head.z >> (8 * j)) & 63u;
    } else {
        int jj = j - 4;
        s = ((head.w >> (8 * jj)) & 15u) | (((head.y >> (8 * jj + 6)) & 3u) << 4);
        mm = ((head.w >> (8 * jj + 4)) & 15u) | (((head.z >> (8 * jj + 6)) & 3u) << 4);
    }
    sc = float(s);
    m = float(mm);
}

__device__ __forceinline__ float2 q4k_d_dmin(const uint4 &head) {
    __half2 hd = *reinterpret_cast<const __half2 *>(&head.x);
    return __half22float2(hd);
}

// Code byte i (0..3) of a 32-bit word as an exact fp32 value: the byte lands
// in the low mantissa bits of 2^23, then 2^23 is subtracted.
__device__ __forceinline__ float nib_to_float(uint32_t nibbles4, int i) {
    uint32_t bits = __byte_perm(nibbles4, 0x4B000000u, 0x7540u | uint32_t(i));
    return __uint_as_float(bits) - 8388608.0f;
}

// Dot products of one 16-byte code chunk (qs bytes b = 0..15 of a 32-byte
// group c) with the matching activations: `lo` = sum_b q_lo[b] * xlo[b]
// (sub-block 2c), `hi` = sum_b q_hi[b] * xhi[b] (sub-block 2c+1).
__device__ __forceinline__ void chunk_dot(const uint4 &q, const float *xlo, const float *xhi,
                                          float &lo, float &hi) {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
    float a = 0.f, b = 0.f;
#pragma unroll
    for (int wi = 0; wi < 4; ++wi) {
        uint32_t l4 = w[wi] & 0x0F0F0F0Fu;
        uint32_t h4 = (w[wi] >> 4) & 0x0F0F0F0Fu;
        float4 xl = *reinterpret_cast<const float4 *>(xlo + 4 * wi);
        float4 xh = *reinterpret_cast<const float4 *>(xhi + 4 * wi);
        a = fmaf(nib_to_float(l4, 0), xl.x, a);
        a = fmaf(nib_to_float(l4, 1), xl.y, a);
        a = fmaf(nib_to_float(l4, 2), xl.z, a);
        a = fmaf(nib_to_float(l4, 3), xl.w, a);
        b = fmaf(nib_to_float(h4, 0), xh.x, b);
        b = fmaf(nib_to_float(h4, 1), xh.y, b);
        b = fmaf(nib_to_float(h4, 2), xh.z, b);
        b = fmaf(nib_to_float(h4, 3), xh.w, b);
    }
    lo = a;
    hi = b;
}

// Read-only 16-byte load of weight bytes.  An intrinsic, not inline asm: the
// compiler must never move a load above the bounds check that guards it.
__device__ __forceinline__ uint4 ldg_nc_v4(const void *p) {
    return __ldg(reinterpret_cast<const uint4 *>(p));
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float silu_mul(float g, float u) {
    return g / (1.0f + expf(-g)) * u;
}

// ---------------------------------------------------------------------------
// Top-k + renormalise by one warp (the routers end here).  The order is
// (logit descending, expert index ascending).  Each lane holds the logits
// of experts lane, lane + 32, ... as order-preserving integer keys, sorted
// once by that order; each of the k rounds takes the largest key over the
// warp and then the smallest expert index among the lanes showing it (two
// warp reductions), and the winning lane drops its head.
// ---------------------------------------------------------------------------
// Key of a logit: larger logits give larger keys, -0 the key of +0 (they
// compare equal), NaN the key 0 (below -inf: a NaN is taken only after
// every number).  logit_of_key inverts it (NaN -> a NaN).
__device__ __forceinline__ uint32_t logit_key(float v) {
    if (v != v) return 0u;
    uint32_t u = __float_as_uint(v);
    if (u == 0x80000000u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float logit_of_key(uint32_t key) {
    return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

// (key, index) a comes first: larger key, or equal key and smaller index
__device__ __forceinline__ bool topk_first(uint32_t ka, uint32_t ia, uint32_t kb, uint32_t ib) {
    return ka > kb || (ka == kb && ia < ib);
}

// Top-k of NT tokens' E <= 32 * kPer logits each (bias already added) by one
// warp, lane L holding the logits of experts L + 32 s of token u in v[u][s];
// the tokens' rounds run interleaved (independent chains).  For token u with
// out[u] set, writes idx[u][0..k) in selection order and the renormalised
// weights w_j = exp(l_j - l_max) / sum over the selection of exp(l - l_max).
template <int kPer, int NT>
__device__ __forceinline__ void warp_topk_multi(const float (&v)[NT][kPer], int E, int k,
                                                int32_t *const (&idx)[NT], float *const (&w)[NT],
                                                const bool (&out)[NT]) {
    const int lane = threadIdx.x & 31;
    uint32_t key[NT][kPer], id[NT][kPer];
#pragma unroll
    for (int u = 0; u < NT; ++u)
#pragma unroll
        for (int s = 0; s < kPer; ++s) {
            const int e = lane + 32 * s;
            key[u][s] = e < E ? logit_key(v[u][s]) : 0u;
            id[u][s] = e < E ? uint32_t(e) : 0xffffffffu;  // past E: after every expert
        }
    // sort each token's candidates in this lane (insertion, unrolled)
#pragma unroll
    for (int u = 0; u < NT; ++u)
#pragma unroll
        for (int s = 1; s < kPer; ++s)
#pragma unroll
            for (int j = s; j > 0; --j)
                if (topk_first(key[u][j], id[u][j], key[u][j - 1], id[u][j - 1])) {
                    const uint32_t tk = key[u][j], ti = id[u][j];
                    key[u][j] = key[u][j - 1];
                    id[u][j] = id[u][j - 1];
                    key[u][j - 1] = tk;
                    id[u][j - 1] = ti;
                }
    uint32_t sel_key[NT], sel_i[NT], kmax[NT];
#pragma unroll
    for (int u = 0; u < NT; ++u) sel_key[u] = sel_i[u] = kmax[u] = 0u;
    for (int j = 0; j < k; ++j) {
#pragma unroll
        for (int u = 0; u < NT; ++u) {
            const uint32_t m = __reduce_max_sync(0xffffffffu, key[u][0]);
            const uint32_t win = __reduce_min_sync(0xffffffffu, key[u][0] == m ? id[u][0] : 0xffffffffu);
            if (id[u][0] == win) {  // the winner drops its head
#pragma unroll
                for (int s = 0; s + 1 < kPer; ++s) {
                    key[u][s] = key[u][s + 1];
                    id[u][s] = id[u][s + 1];
                }
                key[u][kPer - 1] = 0u;
                id[u][kPer - 1] = 0xffffffffu;
            }
            if (j == 0) kmax[u] = m;
            if (lane == j) {
                sel_key[u] = m;
                sel_i[u] = win;
            }
        }
    }
#pragma unroll
    for (int u = 0; u < NT; ++u) {
        const float vmax = logit_of_key(kmax[u]);
        const float ex = (lane < k) ? expf(logit_of_key(sel_key[u]) - vmax) : 0.f;
        const float z = warp_sum(ex);
        if (out[u] && lane < k) {
            idx[u][lane] = int32_t(sel_i[u]);
            w[u][lane] = ex / z;
        }
    }
}

// One token (kPer logits per lane in v).
template <int kPer>
__device__ __forceinline__ void warp_topk_regs(const float (&v)[kPer], int E, int k, int32_t *idx,
                                               float *w) {
    float vv[1][kPer];
#pragma unroll
    for (int s = 0; s < kPer; ++s) vv[0][s] = v[s];
    int32_t *const ii[1] = {idx};
    float *const ww[1] = {w};
    const bool oo[1] = {true};
    warp_topk_multi<kPer, 1>(vv, E, k, ii, ww, oo);
}

// The same, reading the logits from `lg` (E <= kMaxE).
__device__ __forceinline__ void warp_topk(const float *lg, int E, int k, int32_t *idx, float *w) {
    constexpr int kPer = kMaxE / 32;
    const int lane = threadIdx.x & 31;
    float v[kPer];
#pragma unroll
    for (int s = 0; s < kPer; ++s) v[s] = lane + 32 * s < E ? lg[lane + 32 * s] : 0.f;
    warp_topk_regs<kPer>(v, E, k, idx, w);
}

}  // namespace moeq4k
