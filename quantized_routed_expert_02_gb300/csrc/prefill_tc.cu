// Prefill: the expert FFN of a large batch as two grouped GEMMs on the
// tcgen05 tensor cores, with the Q4_K weights dequantised to fp16 in shared
// memory on the way in.
//
// forward_qwen3_moe.rs (aprender-serve 0.35.0), step 2g of forward_qwen3_moe
// runs every position through the layer on its own; tokens are independent,
// so the slots routed to one expert form the columns of one GEMM per expert:
//   gate/up:  G = X_e Wg[e]^T, U = X_e Wu[e]^T  (128 weight rows of each per
//             tile, up to 256 tokens, K = H), epilogue h = SiLU(G) * U (fp16);
//   down:     O = H_e Wd[e]^T (K = I), epilogue o[p, row] in fp32, followed
//             by the slot-ordered combine kernel.
// The activations are first gathered into expert-sorted rows (fp16), and h
// is written in that order too, so every activation tile is one contiguous
// block of rows.
//
// One persistent CTA per SM; work items (expert chunk of <= cap slots x 128
// rows each of gate and up, or 256 rows of down) are taken round-robin
// (item = CTA + i * grid), row tile fastest, so every role walks the same
// sequence without an exchange and one running stage count per ring carries
// the pipeline across item boundaries.  cap = the batch's token count
// rounded up to 32, at most 256 for gate/up and 128 for down.  20 warps; the
// three issuing roles run on whole warps (every lane computes the same
// operands, one elected lane issues):
//   warp 1      raw Q4_K bytes by TMA: one whole block (144 contiguous bytes)
//               of each of the tile's rows per raw stage, 2 x 128 rows;
//   warps 4-19  dequantise each raw stage into four 64-K stages of fp16
//               K-major tiles with the 128-byte swizzle (generic stores, then
//               a proxy fence) in two groups of eight warps, group g taking
//               the stages c % 2 == g (two stages written at once), thread =
//               (row, operand): all 32 code bytes of its row per stage;
//               each group runs its share of the previous item's epilogue
//               after its last stage below the tile ring's depth;
//   warp 2      the chunk's activation rows of each stage by TMA (boxes of 32
//               rows, 128-byte swizzle) into a ring of chunk-sized slots;
//   warp 0      issues tcgen05.mma with the tokens as the M operand:
//               D[tokens][256 weight rows] (+)= A[128 tokens][16 K] x
//               B[256 rows][16 K]^T, the activation tile as M = 128 (a second
//               half for chunks of more than 128 slots; M = 64 when no chunk
//               exceeds 64 slots) and the stage's gate and up (or two down)
//               tiles as one N = 256 operand: four (eight) MMAs per 64-K
//               stage whatever the token count;
//               accumulators fp32 in tensor memory, double-buffered for
//               chunks of <= 128 slots so an item's epilogue overlaps the
//               next item's MMAs.
// The down launch does not wait for the gate/up grid as a whole: every
// gate/up epilogue warp counts its finished h rows per expert (release), and
// the down launch's activation warp loads an expert's rows once its count is
// complete (acquire), so down CTAs start on the SMs that finished gate/up
// CTAs leave.
// The epilogue reads one token per TMEM lane and writes whole 16-byte runs
// of that token's row: h = SiLU(g) * u in fp16 (gate/up), or the per-slot
// fp32 outputs (down).  Every wait is bounded by a global-timer deadline and
// records MOE_ERR_TIMEOUT when it runs out.
#include <cuda.h>
#include <cuda_fp16.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.cuh"
#include "tcgen05.cuh"

namespace moeq4k {
namespace ptc {

constexpr int kThreads = 640;  // 4 role warps + 16 dequantise/epilogue warps
constexpr int kBM = 128;   // weight rows per tile
constexpr int kBN = 256;   // tokens per tile (max): two M = 128 halves
constexpr int kBK = 64;    // K per stage
constexpr int kTileA = kBM * kBK * 2;
constexpr int kBoxRows = 32;                   // activation rows per TMA box
constexpr int kBoxB = kBoxRows * kBK * 2;
constexpr int kStageSlot = 2 * kTileA;         // stage ring slot: the two weight tiles
constexpr int kHead = 2048;  // barriers, item info, token list
constexpr int kDeq = 512;      // warps 4-19
constexpr int kMaxSlots = 16;  // per ring
constexpr int kSub = kQK / kBK;                  // MMA stages per Q4_K block (4)
constexpr int kRawMat = kBM * kBlockBytes;       // one matrix's raw bytes of a raw stage:
                                                 // one whole block (144 B) of each row

struct Params {
    CUtensorMap raw0, raw1;     // raw Q4_K bytes of the two A operands as [E*rows][row bytes]
                                //   uint8: boxes of one block (144 B) x 128 rows
    CUtensorMap mapB;           // activations [T*k sorted rows][K] fp16, 128-byte swizzle
    int mode;                   // 0: gate/up + SwiGLU -> h16; 1: down -> o
    int K;                      // reduction length
    int row_tiles;              // weight rows per expert / item_rows
    int item_rows;              // weight rows per item: 128 (gate/up: 128 of each) or 256
    int y_off1;                 // row offset of the second A operand: 0 (up) or 128 (down)

    const int32_t *offs, *perm;
    const TcChunk *chunks;
    const int32_t *nchunks;     // number of chunks (written by the plan kernel)
    WsHeader *hdr;              // work counters, chunk count, status
    __half *h16;                // mode 0 output [T*k sorted rows][I]
    float *o;                   // mode 1 output [T*k][H]
    int I, H;
    int rows_per_expert;        // I (mode 0) or H (mode 1)
    int nr, r_off;              // raw ring: slots, byte offset (slot = nmat * kRawMat bytes)
    int mh;                     // M halves: 1 (chunks of <= 128 slots, two accumulator
                                //   buffers) or 2 (<= 256 slots, one buffer of two halves)
    int mrows;                  // MMA M: 64 when every chunk has <= 64 slots, else 128
                                //   (M = 64 puts D's rows 16q..16q+15 on TMEM lanes
                                //   32q..32q+15 of lane quadrant q)
    int ns, s_off;              // stage ring: slots, byte offset (slot = kStageSlot bytes)
    int nb, b_off, b_slot;      // activation ring: slots, byte offset, bytes per slot (the
                                //   chunk capacity x 128 B; mrows x 128 - b_slot bytes of
                                //   padding follow the last slot, since the MMA reads mrows
                                //   rows from a slot's start)
    unsigned long long wait_ns;
    unsigned long long *timeline;  // profiling builds only: per-stage role stamps of CTA 0
    // Per-expert count of finished gate/up epilogue pieces (one per
    // epilogue warp and item).  Gate/up adds to it; the down launch, which
    // does not wait for the gate/up grid as a whole, loads an expert's h rows
    // once the count reaches ceil(slots / ready_cap) * ready_tiles * 16.
    unsigned int *ready;
    int ready_cap, ready_tiles;
    int withhold;  // test hook: CTA 0 of the gate/up launch counts none of its pieces
};

// Optional per-stage timeline for profiling builds (-DMOEQ4K_TIMELINE): the
// listed thread of CTA 0 stamps the global timer for event `ev` of global
// stage (or item) `g` < 256.
#ifdef MOEQ4K_TIMELINE
#define GT_STAMP(p, ev, g)                                                        \
    do {                                                                          \
        if (blockIdx.x == 0 && (p).timeline != nullptr && (g) < 256u)             \
            (p).timeline[(ev) * 256 + (g)] = global_timer_ns();                  \
    } while (0)
#else
#define GT_STAMP(p, ev, g) ((void)0)
#endif

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, uint64_t deadline,
                                         WsHeader *hdr, int site) {
    if (mbar_wait_sleep(bar, parity, deadline)) return true;
    record_status(hdr, MOE_ERR_TIMEOUT, site);
    return false;
}

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }
__device__ __forceinline__ __half2 bits_h2(uint32_t u) { return *reinterpret_cast<__half2 *>(&u); }

// K order inside the fp16 operand tiles: within each aligned group of four,
// positions 1 and 2 are swapped (the dequantiser below produces that order
// two codes per instruction; the activation operands are written in the same
// order, so every dot product is unchanged).
__host__ __device__ inline int kperm(int k) { return (k & ~3) | ((k & 1) << 1) | ((k >> 1) & 1); }

// d*sc and -dmin*m of sub-blocks 2c and 2c+1 from a 16-byte block head, as
// fp16 pairs A = (d*sc0, d*sc1), NB = (-dmin*m0, -dmin*m1).  The 6-bit
// fields land in the low mantissa bits of the fp16 value 1024 (exact), 1024
// is subtracted exactly, and one fp16 multiply per pair rounds each product
// once.  Fields: sub-block j < 4: sc = scales[j] & 63, m = scales[j+4] & 63;
// j >= 4: sc = scales[j+4] & 15 | (scales[j-4] >> 6) << 4,
//         m = scales[j+4] >> 4 | (scales[j] >> 6) << 4 (head.y = scales[0..3],
// head.z = scales[4..7], head.w = scales[8..11]).
__device__ __forceinline__ void stage_scales_h2(const uint4 &h, int c, __half2 &A, __half2 &NB) {
    // bytes 2(c%2) and 2(c%2)+1 of a head word to bits 0-7 and 16-23
    const uint32_t sel = 0x4140u + 0x202u * uint32_t(c & 1);
    uint32_t sc, mm;
    if (c < 2) {
        sc = __byte_perm(h.y, 0u, sel);
        mm = __byte_perm(h.z, 0u, sel);
    } else {
        const uint32_t wp = __byte_perm(h.w, 0u, sel);
        const uint32_t yp = __byte_perm(h.y, 0u, sel);
        const uint32_t zp = __byte_perm(h.z, 0u, sel);
        sc = (wp & 0x000F000Fu) | ((yp >> 2) & 0x00300030u);
        mm = ((wp >> 4) & 0x000F000Fu) | ((zp >> 2) & 0x00300030u);
    }
    const __half2 k1024 = bits_h2(0x64006400u);
    const __half2 scv = __hsub2(bits_h2((sc & 0x003F003Fu) | 0x64006400u), k1024);
    const __half2 mneg = __hsub2(k1024, bits_h2((mm & 0x003F003Fu) | 0x64006400u));
    A = __hmul2(bits_h2(__byte_perm(h.x, 0u, 0x1010u)), scv);    // (d, d) * (sc0, sc1)
    NB = __hmul2(bits_h2(__byte_perm(h.x, 0u, 0x3232u)), mneg);  // (dmin, dmin) * (-m0, -m1)
}

// (v & 0x000F000F) | 0x64006400: the codes in bits 0-3 and 16-19 as the fp16
// values 1024 + q (exact).
__device__ __forceinline__ uint32_t code_pair(uint32_t v) { return (v & 0x000F000Fu) | 0x64006400u; }

// q*a + nb for one pair: the subtraction of 1024 is exact, the fused
// multiply-add rounds once.
__device__ __forceinline__ uint32_t weight_pair(uint32_t p, __half2 a, __half2 nb) {
    return h2_bits(__hfma2(__hsub2(bits_h2(p), bits_h2(0x64006400u)), a, nb));
}

// The 8 weights of one 16-byte tile chunk from code words va, vb (bytes
// 4i..4i+7 of the stage's codes): nibble SH (0 low, 4 high) of bytes 0..3
// of va then of vb, in the kperm order 0, 2, 1, 3, 4, 6, 5, 7.
template <int SH>
__device__ __forceinline__ uint4 chunk8(uint32_t va, uint32_t vb, __half2 a, __half2 nb) {
    uint4 r;
    r.x = weight_pair(code_pair(va >> SH), a, nb);
    r.y = weight_pair(code_pair(va >> (SH + 8)), a, nb);
    r.z = weight_pair(code_pair(vb >> SH), a, nb);
    r.w = weight_pair(code_pair(vb >> (SH + 8)), a, nb);
    return r;
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ void sts128(uint32_t addr, const uint4 &v) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

// A bounded wait by every lane of a warp, with one outcome for the warp (a
// lane that saw the phase complete just as another hit the deadline still
// takes the abort path with it), so the warp never splits at a __syncwarp.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, uint64_t deadline,
                                          WsHeader *hdr, int site) {
    return __all_sync(0xffffffffu, wait_bar(bar, parity, deadline, hdr, site));
}

// A bounded warp-wide wait that probes the phase without a suspend hint and
// sleeps 64 ns between probes: a waiting warp then issues a handful of
// instructions per wait instead of a loop of suspended probes that return
// early, leaving issue slots to the warps that work (measured: 2 % faster
// at batched decode when the dequantising warps wait this way).
__device__ __forceinline__ bool nap_wait(uint64_t *bar, uint32_t parity, uint64_t deadline,
                                         WsHeader *hdr, int site) {
    bool done = mbar_try_wait(bar, parity);
    while (!done) {
        if (global_timer_ns() > deadline) {
            record_status(hdr, MOE_ERR_TIMEOUT, site);
            break;
        }
        __nanosleep(64);
        done = mbar_try_wait(bar, parity);
    }
    return __all_sync(0xffffffffu, done);
}

// One lane of a fully active warp, chosen once by elect.sync.  The issuing
// roles run on whole warps so the operands of their tcgen05 / TMA
// instructions are computed by every lane alike (warp-uniform), and only the
// elected lane issues; a role's MMAs and the commits that track them come
// from that same lane.
__device__ __forceinline__ bool elect_one() {
    uint32_t is = 0;
    asm volatile(
        "{\n\t.reg .pred P;\n\telect.sync _|P, 0xffffffff;\n\tselp.u32 %0, 1, 0, P;\n\t}"
        : "=r"(is));
    return is != 0u;
}

// Position in a ring of n slots: the slot and the parity of its current
// phase (how many times the ring wrapped, mod 2), advanced without division.
struct RingPos {
    uint32_t slot = 0, phase = 0;
    __device__ __forceinline__ void next(uint32_t n) {
        if (++slot == n) {
            slot = 0;
            phase ^= 1u;
        }
    }
};

// One work item: expert chunk `ch` (its sorted slots) x weight-row tile `rt`.
struct Item {
    TcChunk ch;
    int rt, nmma, row0;  // MMA width (slots rounded up to 16), first sorted activation row
};

// Items run row-tile fastest: the row tiles of one chunk (which share its
// activation rows) and the chunks of one expert (which share its weight rows)
// are consecutive items, so they run at the same time on neighbouring CTAs
// and the second and later reads of those bytes are L2 hits.
__device__ __forceinline__ Item item_of(const Params &p, int it, int nch) {
    (void)nch;
    Item I;
    I.ch = p.chunks[it / p.row_tiles];
    I.rt = it % p.row_tiles;
    I.nmma = (I.ch.tok_cnt + 15) & ~15;
    I.row0 = p.offs[I.ch.e] + I.ch.tok_off;
    return I;
}

// The epilogue of item `E` (the li_e-th of this CTA) from accumulator
// buffer li_e % nbuf, run by the sixteen dequantising warps (warp (q, part):
// TMEM lane quadrant q, column quarter `part`).  The accumulator is
// D[token][weight row]: TMEM lane = the chunk's token (slot) n, column =
// weight row c of the item's 256 (gate rows 0-127 then up rows 0-127, or 256
// down rows).  Warp (q, part) reads lanes 32q.. (tokens 32q..32q+31) and a
// quarter of the rows; each thread then writes whole 16-byte runs of its
// token's row.  Not inlined: the stage loop that calls it is unrolled.
__device__ __noinline__ bool item_epilogue(const Params &p, const Item &E, uint32_t li_e,
                                           uint32_t nbuf, uint32_t taddr, uint64_t *accfull,
                                           uint64_t *accempty, uint64_t deadline, int q, int part,
                                           int lane) {
            const uint32_t buf = li_e % nbuf, use = li_e / nbuf;
            if (!warp_wait(accfull + buf, use & 1u, deadline, p.hdr, 14)) return false;
            tc::fence_after_sync();
            const int ntok = E.ch.tok_cnt;
            const int tq = p.mrows / 4;  // tokens per TMEM lane quadrant
            for (int h = 0; h < p.mh; ++h) {
            // warp-uniform: quadrants past the chunk's tokens have no output
            if (128 * h + tq * q < ntok) {
                const int n = 128 * h + tq * q + lane;
                const bool valid = lane < tq && n < ntok;
                const uint32_t lanebase = taddr + (buf + uint32_t(h)) * 256u + (uint32_t(q * 32) << 16);
                if (p.mode == 0) {
                    // h = SiLU(g) * u for rows 32*part .. +31 of the item's 128,
                    // stored in the kperm order of the down GEMM's K
                    __half *hrow = p.h16 + size_t(E.row0 + n) * p.I + E.rt * kBM;
                    for (int c0 = 32 * part; c0 < 32 * part + 32; c0 += 8) {
                        float g[8], u[8];
                        tc::tmem_ld8(lanebase + c0, g);
                        tc::tmem_ld8(lanebase + 128 + c0, u);
                        float h[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            // SiLU(g) * u with the fast exponential and divide: the
                            // result is rounded to fp16
                            const float e = __expf(fminf(-g[j], 80.0f));
                            h[j] = __fdividef(g[j], 1.0f + e) * u[j];
                        }
                        uint4 o;  // positions c0 + (0, 2, 1, 3, 4, 6, 5, 7) hold h[0..7]
                        o.x = h2_bits(__floats2half2_rn(h[0], h[2]));
                        o.y = h2_bits(__floats2half2_rn(h[1], h[3]));
                        o.z = h2_bits(__floats2half2_rn(h[4], h[6]));
                        o.w = h2_bits(__floats2half2_rn(h[5], h[7]));
                        if (valid) *reinterpret_cast<uint4 *>(hrow + c0) = o;
                    }
                } else {
                    // per-slot outputs: rows 64*part .. +63 of the item's 256
                    float *orow = p.o + size_t(valid ? p.perm[E.row0 + n] : 0) * p.H +
                                  E.rt * p.item_rows;
                    for (int c0 = 64 * part; c0 < 64 * part + 64; c0 += 8) {
                        float v[8];
                        tc::tmem_ld8(lanebase + c0, v);
                        if (valid) tc::st_global_v8(orow + c0, v);  // 32-byte aligned
                    }
                }
            }
            }
            // every lane's tensor-memory loads have completed (each load waits for
            // its values): the next item's MMAs may overwrite the accumulator
            // while this warp's h rows are still being made visible below
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(accempty + buf);
            if (p.mode == 0 && p.ready != nullptr && !(p.withhold && blockIdx.x == 0)) {
                // this warp's h rows of the item are stored: visible GPU-wide
                // before the count that the down launch acquires
                __threadfence();
                __syncwarp();
                if (lane == 0) red_release_add_u32(p.ready + E.ch.e, 1u);
            }
            __syncwarp();
            return true;
        }

__global__ void __launch_bounds__(kThreads, 1) grouped_gemm_kernel(const __grid_constant__ Params p) {
    // The down launch with per-expert readiness does not wait for the gate/up
    // grid: its CTAs start on the SMs that gate/up CTAs leave, stream and
    // dequantise down weights at once, and load an expert's h rows when its
    // count is complete.  What else it reads (chunk plans, offsets,
    // permutation) was written by launches that completed before the gate/up
    // launch began.
    // (Measured: 86.5 -> 71.2 us at 64 Zipf tokens, 503 -> 498 us at 32 A22B
    // tokens, 591 -> 575 us at 4096 tokens against waiting for the grid.)
    const bool overlap = p.mode == 1 && p.ready != nullptr;
    if (overlap)
        pdl_trigger();
    else
        pdl_enter();
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t *rfull = reinterpret_cast<uint64_t *>(smem);
    uint64_t *rempty = rfull + kMaxSlots;
    // stage ring: the two weight tiles of an MMA stage (2 x 16 KB per slot);
    // activation ring: the chunk's activation rows of an MMA stage
    uint64_t *sfull = rempty + kMaxSlots;   // weight tiles written
    uint64_t *sempty = sfull + kMaxSlots;   // the stage slot's MMAs are complete
    uint64_t *bfull = sempty + kMaxSlots;   // the activation copy's bytes (TMA only)
    uint64_t *bempty = bfull + kMaxSlots;   // the activation slot's MMAs are complete
    uint64_t *accfull = bempty + kMaxSlots;  // [2] an item's accumulators are complete
    uint64_t *accempty = accfull + 2;        // [2] the epilogue has read them
    uint64_t *drain = accempty + 2;
    uint32_t *tmem_ptr = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_ptr + 4);
    uint8_t *rring = smem + p.r_off;
    uint8_t *sring = smem + p.s_off;
    uint8_t *bring = smem + p.b_off;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int NR = p.nr, NS = p.ns, NB = p.nb;
    constexpr int nmat = 2;  // two A operands per item: gate and up, or two 128-row halves
    const int S = p.K / kBK;  // MMA stages per item
    const int SR = S / kSub;  // raw stages per item
    const uint64_t deadline = global_timer_ns() + p.wait_ns;
    const uint32_t tcols = 512u;  // two 256-column accumulators (buffers, or M halves)
    const uint32_t nbuf = p.mh == 2 ? 1u : 2u;  // accumulator buffers (item li uses li % nbuf)

    if (tid == 0) {
        for (int i = 0; i < NR; ++i) {
            mbar_init(rfull + i, 1);           // the TMA thread's arrival + its bytes
            mbar_init(rempty + i, kDeq / 32);  // one arrival per dequant warp
        }
        for (int i = 0; i < NS; ++i) {
            mbar_init(sfull + i, kDeq / 64);   // one arrival per warp of the stage's group
            mbar_init(sempty + i, 1);          // MMA completion
        }
        for (int i = 0; i < NB; ++i) {
            mbar_init(bfull + i, 1);           // the TMA thread's arrival + its bytes
            mbar_init(bempty + i, 1);          // MMA completion
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(accfull + i, 1);             // MMA completion of the item's last stage
            mbar_init(accempty + i, kDeq / 32);    // every epilogue warp has read them
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    // the activation ring (and the padding after it) starts as zeros: the MMA
    // reads 128 rows from a slot's start, and rows no copy has written must
    // hold finite values
    for (int i = tid; i < (NB * p.b_slot + max(0, p.mrows * kBK * 2 - p.b_slot)) / 16; i += kThreads)
        reinterpret_cast<uint4 *>(bring)[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();  // before any TMA write into the ring
    if (warp == 0) tc::tmem_alloc(tmem_ptr, tcols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t taddr = *tmem_ptr;
    const int nch = *p.nchunks;
    const int total = nch * p.row_tiles;
    // Items are taken round-robin (item = blockIdx.x + i * gridDim.x), so every
    // role walks the same sequence with no exchange, and one running stage
    // count per ring carries the pipeline across item boundaries.
    uint32_t issued = 0;  // warps 1 and 2: copy phases started (for the abort drain)

    if (warp >= 4) {
        // ---- dequantise weight rows into the A tiles; after the first stages
        // of the next item, run the previous item's epilogue
        // two groups of eight warps (warps 4-11: hh = 0, 12-19: hh = 1); group
        // hh dequantises the stages c of each raw block with c % 2 == hh, so
        // two stages are being written at once; thread -> (row r of A operand
        // m): all 32 code bytes of its row per stage, tile chunks 0-7
        const int dq = tid - 128;
        const int r = dq & 127;
        const int m = (dq >> 7) & 1;  // A operand: gate / up, or the first / second 128 rows
        const int hh = dq >> 8;
        const uint32_t rbase = smem_addr(rring) + uint32_t(m * kRawMat) + uint32_t(kBlockBytes) * r;
        const uint32_t til0 = smem_addr(sring) + uint32_t(m * kTileA);
        // the row's eight tile chunks: 0-3 from the low nibbles of code words
        // 0-7, 4-7 from the high nibbles
        uint32_t soff[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) soff[j] = tc::sw128_offset(r, 8 * j);
        const int q = warp & 3, part = (warp - 4) >> 2;  // TMEM lane quadrant, column quarter

        uint32_t g = 0, gr = 0, li = 0;
        RingPos rp, ap;  // raw ring, stage ring
        Item prev;
        bool have_prev = false;
        bool ok = true;
        for (int it = blockIdx.x; ok && it < total; it += gridDim.x, ++li) {
            const Item cur = item_of(p, it, nch);
            if (tid == 128) GT_STAMP(p, 8, li);
            const int epi_at = min(S, NS) - 1;  // stage after which the previous epilogue runs
            for (int sr = 0; ok && sr < SR; ++sr, ++gr, rp.next(NR)) {
                const uint32_t rs = rp.slot;
                if (!nap_wait(rfull + rs, rp.phase, deadline, p.hdr, 16)) {
                    ok = false;
                    break;
                }
                const uint32_t rsl = rbase + rs * uint32_t(nmat * kRawMat);
                const uint4 head = lds128(rsl);
#pragma unroll
                for (int c = 0; c < kSub; ++c) {
                    // group hh (warps 4-11: 0, 12-19: 1) dequantises the sub-stages
                    // with c % 2 == hh, all 32 code bytes of its row each
                    const int s = sr * kSub + c;
                    const uint32_t as = ap.slot, aph = ap.phase;
                    ap.next(NS);
                    const uint32_t gcur = g++;
                    if ((c & 1) != hh) continue;
                    if (tid == 128) GT_STAMP(p, 1, gcur);  // profiling builds: group 0's stages
                    const uint4 q0 = lds128(rsl + 16u + 32u * c), q1 = lds128(rsl + 16u + 32u * c + 16u);
                    if (c + 2 >= kSub) {
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(rempty + rs);
                    }
                    if (gcur >= uint32_t(NS) && !nap_wait(sempty + as, aph ^ 1u, deadline, p.hdr, 11)) {
                        ok = false;
                        break;
                    }
                    if (tid == 128) GT_STAMP(p, 2, gcur);
                    __half2 A, NB;
                    stage_scales_h2(head, c, A, NB);
                    const __half2 a0 = __low2half2(A), a1 = __high2half2(A);
                    const __half2 n0 = __low2half2(NB), n1 = __high2half2(NB);
                    const uint32_t tile = til0 + as * uint32_t(kStageSlot);
                    sts128(tile + soff[0], chunk8<0>(q0.x, q0.y, a0, n0));
                    sts128(tile + soff[1], chunk8<0>(q0.z, q0.w, a0, n0));
                    sts128(tile + soff[2], chunk8<0>(q1.x, q1.y, a0, n0));
                    sts128(tile + soff[3], chunk8<0>(q1.z, q1.w, a0, n0));
                    sts128(tile + soff[4], chunk8<4>(q0.x, q0.y, a1, n1));
                    sts128(tile + soff[5], chunk8<4>(q0.z, q0.w, a1, n1));
                    sts128(tile + soff[6], chunk8<4>(q1.x, q1.y, a1, n1));
                    sts128(tile + soff[7], chunk8<4>(q1.z, q1.w, a1, n1));
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(sfull + as);
                    if (tid == 128) GT_STAMP(p, 3, gcur);
                    // this group's share of the previous item's epilogue, after its last
                    // stage below the ring depth: every wait before it depends only on the
                    // previous item's MMAs, and the next item's first MMA needs it
                    if (have_prev && s + 2 >= epi_at + 1) {
                        if (!item_epilogue(p, prev, li - 1, nbuf, taddr, accfull, accempty, deadline,
                                           q, part, lane))
                            ok = false;
                        have_prev = false;
                    }
                }
            }
            prev = cur;
            have_prev = true;
        }
        if (ok && have_prev) {
            if (tid == 128) GT_STAMP(p, 9, li - 1);
            ok = item_epilogue(p, prev, li - 1, nbuf, taddr, accfull, accempty, deadline, q, part,
                               lane);
            if (tid == 128) GT_STAMP(p, 10, li - 1);
        }
        if (!ok) *abort_flag = 1;
    } else if (warp == 0) {
        // ---- MMA issue: accumulators of item li in buffer li % nbuf.  The
        // whole warp walks the loop (waits by all lanes with one outcome);
        // the elected lane issues the MMAs and their commits.
        const bool leader = elect_one();
        uint32_t g = 0, li = 0;
        RingPos sp, bp;  // stage ring, activation ring
        const uint32_t ring0 = smem_addr(sring), act0 = smem_addr(bring);
        bool ok = true;
#ifdef MOEQ4K_TIMELINE
        long long cyc[6] = {0, 0, 0, 0, 0, 0};  // afull wait, bfull wait, MMA issue, commits, loop, stages
        long long c0 = clock64(), c1;
#define MMA_CYC(i) (c1 = clock64(), cyc[i] += c1 - c0, c0 = c1)
#else
#define MMA_CYC(i) ((void)0)
#endif
        for (int it = blockIdx.x; ok && it < total; it += gridDim.x, ++li) {
            const Item cur = item_of(p, it, nch);
            const uint32_t buf = li % nbuf, use = li / nbuf;
            if (use >= 1 && !warp_wait(accempty + buf, (use - 1) & 1u, deadline, p.hdr, 19)) {
                ok = false;
                break;
            }
            tc::fence_after_sync();
            // D[M tokens][256 weight rows] (+)= A[M tokens][16 K] x B[256 rows][16 K]^T:
            // the activation tile is the M operand, the stage's two 128-row weight
            // tiles (contiguous 8-row swizzle groups) are one N = 256 operand
            const uint32_t idesc = tc::idesc_f16_f32(p.mrows, 2 * kBM);
            const uint32_t d = taddr + buf * 256u;  // half h at d + 256 h (p.mh == 2: buf = 0)
            // the second 128-token half only for chunks that reach into it
            const bool two_halves = __all_sync(0xffffffffu, p.mh == 2 && cur.nmma > kBM);
            for (int s = 0; s < S; ++s, ++g, sp.next(NS), bp.next(NB)) {
                const uint32_t ss = sp.slot, bs = bp.slot;
                MMA_CYC(4);
                if (!warp_wait(sfull + ss, sp.phase, deadline, p.hdr, 13)) {
                    ok = false;
                    break;
                }
                MMA_CYC(0);
                if (!warp_wait(bfull + bs, bp.phase, deadline, p.hdr, 18)) {
                    ok = false;
                    break;
                }
                MMA_CYC(1);
                tc::fence_after_sync();
                // descriptors of the stage's first 16-wide K slice; each next slice
                // starts 32 bytes on (2 in the descriptor's address field)
                const uint32_t wts = ring0 + ss * uint32_t(kStageSlot);
                const uint64_t dw = tc::smem_desc_sw128(wts);
                const uint64_t da = tc::smem_desc_sw128(act0 + bs * uint32_t(p.b_slot));
                if (leader) {
                    if (two_halves) {
#pragma unroll
                        for (int kk = 0; kk < kBK / 16; ++kk) {
                            // rows 128.. of the activation tile start 16 KB on (1024 in
                            // the descriptor's address field) and accumulate 256 columns on
                            tc::mma_f16(d, da + uint64_t(2 * kk), dw + uint64_t(2 * kk), idesc,
                                        s > 0 || kk > 0);
                            tc::mma_f16(d + 256u, da + uint64_t(2 * kk + 1024), dw + uint64_t(2 * kk),
                                        idesc, s > 0 || kk > 0);
                        }
                    } else {
#pragma unroll
                        for (int kk = 0; kk < kBK / 16; ++kk)
                            tc::mma_f16(d, da + uint64_t(2 * kk), dw + uint64_t(2 * kk), idesc,
                                        s > 0 || kk > 0);
                    }
                    MMA_CYC(2);
                    tc::commit_arrive(sempty + ss);
                    tc::commit_arrive(bempty + bs);
                    MMA_CYC(3);
                }
                __syncwarp();
#ifdef MOEQ4K_TIMELINE
                ++cyc[5];
#endif
            }
            if (ok && leader) tc::commit_arrive(accfull + buf);
            __syncwarp();
        }
        if (!ok) *abort_flag = 1;
#ifdef MOEQ4K_TIMELINE
        if (blockIdx.x == 0 && p.timeline != nullptr && leader)
            for (int i = 0; i < 6; ++i) p.timeline[11 * 256 + 128 + i] = (unsigned long long)cyc[i];
#endif
#undef MMA_CYC
        // every issued MMA must be complete before the tensor memory is released
        if (leader) tc::commit_arrive(drain);
        __syncwarp();
        warp_wait(drain, 0, global_timer_ns() + p.wait_ns, p.hdr, 15);
    } else if (warp == 2) {
        // ---- activation tile of each stage by TMA: the chunk's sorted rows
        // (rounded up to 32) x 64 K, in boxes of 32 rows; the whole warp walks
        // the loop, the elected lane issues
        const bool leader = elect_one();
        uint32_t g = 0;
        RingPos bp;
        bool ok = true;
        int ready_e = -1;  // the expert whose h rows were last seen complete
        for (int it = blockIdx.x; ok && it < total; it += gridDim.x) {
            const Item cur = item_of(p, it, nch);
            if (overlap && cur.ch.e != ready_e) {
                const int e = cur.ch.e;
                const int cnt = p.offs[e + 1] - p.offs[e];
                const unsigned need = unsigned((cnt + p.ready_cap - 1) / p.ready_cap) *
                                      unsigned(p.ready_tiles) * unsigned(kDeq / 32);
                bool seen = ld_acquire_u32(p.ready + e) >= need;
                while (!seen && global_timer_ns() <= deadline) {
                    __nanosleep(256);
                    seen = ld_acquire_u32(p.ready + e) >= need;
                }
                if (!__all_sync(0xffffffffu, seen)) {
                    record_status(p.hdr, MOE_ERR_TIMEOUT, 18);
                    ok = false;
                    break;
                }
                // the h rows were written through the generic proxy; the TMA
                // reads them through the async proxy
                asm volatile("fence.proxy.async.global;" ::: "memory");
                ready_e = e;
            }
            // the boxes of 32 rows holding the chunk's rows; the M operand's
            // other rows keep what the slot held before (zeros, or earlier
            // activations: finite values) and give accumulator rows the
            // epilogue never reads
            const int nbox = (cur.nmma + kBoxRows - 1) / kBoxRows;
            for (int s = 0; s < S; ++s, ++g, bp.next(NB)) {
                const uint32_t bs = bp.slot;
                if (__any_sync(0xffffffffu, *abort_flag != 0) ||
                    (g >= uint32_t(NB) && !warp_wait(bempty + bs, bp.phase ^ 1u, deadline, p.hdr, 12))) {
                    ok = false;
                    break;
                }
                ++issued;
                if (leader) {
                    GT_STAMP(p, 7, g);
                    mbar_arrive_expect_tx(bfull + bs, nbox * kBoxB);
                    for (int i = 0; i < nbox; ++i)
                        tma_load_2d(bring + size_t(bs) * p.b_slot + i * kBoxB, &p.mapB, s * kBK,
                                    cur.row0 + i * kBoxRows, bfull + bs);
                }
                __syncwarp();
            }
        }
        if (!ok) *abort_flag = 1;
    } else if (warp == 1) {
        // ---- raw bytes by TMA, one whole block (144 B) of each of the
        // tile's rows per raw stage: one contiguous segment per row; the whole
        // warp walks the loop, the elected lane issues
        const bool leader = elect_one();
        uint32_t gr = 0;
        RingPos rp;
        bool ok = true;
        for (int it = blockIdx.x; ok && it < total; it += gridDim.x) {
            const Item cur = item_of(p, it, nch);
            const int y = cur.ch.e * p.rows_per_expert + cur.rt * p.item_rows;
            for (int sr = 0; sr < SR; ++sr, ++gr, rp.next(NR)) {
                const uint32_t rs = rp.slot;
                if (__any_sync(0xffffffffu, *abort_flag != 0) ||
                    (gr >= uint32_t(NR) && !warp_wait(rempty + rs, rp.phase ^ 1u, deadline, p.hdr, 17))) {
                    ok = false;
                    break;
                }
                ++issued;
                if (leader) {
                    uint8_t *dst = rring + size_t(rs) * nmat * kRawMat;
                    GT_STAMP(p, 0, gr * kSub);
                    mbar_arrive_expect_tx(rfull + rs, nmat * kRawMat);
                    tma_load_2d(dst, &p.raw0, sr * kBlockBytes, y, rfull + rs);
                    tma_load_2d(dst + kRawMat, &p.raw1, sr * kBlockBytes, y + p.y_off1, rfull + rs);
                }
                __syncwarp();
            }
        }
        if (!ok) *abort_flag = 1;
    }
    __syncthreads();
    // After a timed-out wait the consumers may have left copies unawaited:
    // each copying thread waits (bounded) for the last phase it started on
    // every slot of its ring, so no copy still targets this CTA's shared
    // memory when it exits.  (Without a time-out every phase was consumed.)
    if (*abort_flag && (warp == 1 || warp == 2) && lane == 0) {
        uint64_t *bars = warp == 1 ? rfull : bfull;
        const uint32_t n = warp == 1 ? uint32_t(NR) : uint32_t(NB);
        const uint64_t limit = global_timer_ns() + p.wait_ns;
        for (uint32_t i = 0; i < n && i < issued; ++i) {
            const uint32_t gg = issued - 1 - i;
            wait_bar(bars + gg % n, (gg / n) & 1, limit, p.hdr, 19);
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 0) tc::tmem_dealloc(taddr, tcols);
}

// Activations in expert-sorted order: row slotpos[t*k + j] of xs = x[t] as
// fp16 for every slot j of token t, each group of four elements in kperm
// order.  Thread per (token, 4 elements): x is read once, written k times.
__global__ void gather_half_kernel(const float *__restrict__ x, const int32_t *__restrict__ slotpos,
                                   int T, int k, int H, __half *__restrict__ xs,
                                   unsigned int *__restrict__ ready, int E) {
    pdl_enter();
    // the per-expert gate/up counts start every call at zero (the previous
    // call's down launch, which read them, has completed)
    if (blockIdx.x == 0)
        for (int e = threadIdx.x; e < E; e += blockDim.x) ready[e] = 0u;
    const int per_row = H / 4;
    const size_t total = size_t(T) * per_row;
    for (size_t i = blockIdx.x * size_t(blockDim.x) + threadIdx.x; i < total;
         i += size_t(gridDim.x) * blockDim.x) {
        const int t = int(i / per_row), c = int(i % per_row);
        const float4 v = reinterpret_cast<const float4 *>(x + size_t(t) * H)[c];
        // kperm order within each group of four: x0, x2, x1, x3
        __half2 a = __floats2half2_rn(v.x, v.z), b = __floats2half2_rn(v.y, v.w);
        uint2 o;
        o.x = *reinterpret_cast<uint32_t *>(&a);
        o.y = *reinterpret_cast<uint32_t *>(&b);
        for (int j = 0; j < k; ++j) {
            const int pos = slotpos[t * k + j];
            if (pos < 0) continue;  // invalid expert index: no sorted row
            reinterpret_cast<uint2 *>(xs + size_t(pos) * H)[c] = o;
        }
    }
}

}  // namespace ptc

namespace {
int g_tc_smem_optin[64];

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

// Raw bytes of one matrix family as a 2-D uint8 tensor: E*rows rows of
// nsb*144 bytes; box = one block (144 B, a multiple of 16) x 128 rows.
// Every x coordinate used (a block start, 144*b) is a multiple of 16 bytes.
bool encode_raw_map(CUtensorMap *map, const void *base, int E, int rows, int nsb) {
    const cuuint64_t dims[2] = {cuuint64_t(nsb) * kBlockBytes, cuuint64_t(E) * rows};
    const cuuint64_t strides[1] = {cuuint64_t(nsb) * kBlockBytes};
    const cuuint32_t box[2] = {cuuint32_t(kBlockBytes), cuuint32_t(ptc::kBM)};
    const cuuint32_t estr[2] = {1, 1};
    return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
// Sorted activation rows as a 2-D fp16 tensor [rows][K]; box = 32 rows x 64
// K, stored with the 128-byte swizzle the MMA descriptors expect (the
// swizzle pattern repeats every 8 rows, so boxes stack at 4 KB steps).
bool encode_act_map(CUtensorMap *map, const void *base, int rows, int K) {
    const cuuint64_t dims[2] = {cuuint64_t(K), cuuint64_t(rows)};
    const cuuint64_t strides[1] = {cuuint64_t(K) * 2};
    const cuuint32_t box[2] = {cuuint32_t(ptc::kBK), cuuint32_t(ptc::kBoxRows)};
    const cuuint32_t estr[2] = {1, 1};
    return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void *>(base), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
}  // namespace

bool encode_fp32_sw128_map(CUtensorMap *map, const float *base, int rows, int cols, int box_rows) {
    if (g_encode == nullptr) return false;
    const cuuint64_t dims[2] = {cuuint64_t(cols), cuuint64_t(rows)};
    const cuuint64_t strides[1] = {cuuint64_t(cols) * sizeof(float)};
    const cuuint32_t box[2] = {32, cuuint32_t(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(base), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A row-major fp32 matrix [rows][cols] as a 2-D tensor with boxes of
// box_cols x box_rows and no swizzle (the box lands as box_rows rows of
// box_cols floats); rows past the end arrive as zeros.
bool encode_fp32_box_map(CUtensorMap *map, const float *base, int rows, int cols, int box_cols,
                         int box_rows) {
    if (g_encode == nullptr) return false;
    const cuuint64_t dims[2] = {cuuint64_t(cols), cuuint64_t(rows)};
    const cuuint64_t strides[1] = {cuuint64_t(cols) * sizeof(float)};
    const cuuint32_t box[2] = {cuuint32_t(box_cols), cuuint32_t(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(base), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t init_prefill_tc(int dev) {
    int optin = 0;
    cudaError_t err = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (err != cudaSuccess) return err;
    g_tc_smem_optin[dev] = optin;
    if (g_encode == nullptr) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
        if (err != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr)
            return err != cudaSuccess ? err : cudaErrorNotSupported;
        g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    return cudaFuncSetAttribute(ptc::grouped_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                optin);
}

// Batches of at least kMinTcSlots routed slots take the tensor-core GEMMs:
// their cost is one dequantisation per weight per expert chunk, whatever the
// number of tokens, while the CUDA-core path's grows with the tokens.
constexpr int kMinTcSlots = 256;

bool prefill_tc_supported(int T, int H, int E, int k, int I) {
    return T * k >= kMinTcSlots && I % ptc::kBM == 0 && H % (2 * ptc::kBM) == 0;
}

// Chunk capacity: no more than the batch's tokens (rounded to 32), so small
// batches get deep rings; up to 256 slots (two M halves, one accumulator
// buffer) for gate/up, up to 128 for down, whose large fp32 epilogue then
// overlaps the next item's MMAs (two accumulator buffers).  A larger expert
// list (a caller's routing with repeated experts) is split into more chunks.
void prefill_tc_caps(int T, int *cap_gu, int *cap_dn) {
    const int tcap = (T + ptc::kBoxRows - 1) / ptc::kBoxRows * ptc::kBoxRows;
    *cap_gu = std::min(ptc::kBN, tcap);
    *cap_dn = std::min(ptc::kBM, tcap);
}

cudaError_t launch_prefill_tc(int dev, const float *x, const uint8_t *gate, const uint8_t *up,
                              const uint8_t *down, int T, int H, int E, int k, int I,
                              const int32_t *offs, const int32_t *perm, const int32_t *slotpos,
                              const int32_t *active, const int32_t *nactive, __half *x16,
                              __half *h16, float *obuf, TcChunk *chunks, TcChunk *chunks_dn,
                              unsigned int *ready, WsHeader *hdr,
                              int num_sms, unsigned long long wait_ns, int withhold,
                              unsigned long long *timeline, cudaStream_t s) {
    using namespace ptc;
    launch_pdl(gather_half_kernel, dim3(num_sms * 8), dim3(256), size_t(0), s, x, slotpos, T, k, H, x16,
               ready, E);
    int cap_gu = 0, cap_dn = 0;  // the plans for these capacities came with the permutation
    prefill_tc_caps(T, &cap_gu, &cap_dn);
    const int rows = T * k;

    Params p = {};
    int cap = cap_gu;
    p.mh = cap > kBM ? 2 : 1;
    p.mrows = cap <= 64 ? 64 : kBM;
    p.offs = offs;
    p.perm = perm;
    p.chunks = chunks;
    p.nchunks = &hdr->tc_chunks;
    p.hdr = hdr;
    p.h16 = h16;
    p.o = obuf;
    p.I = I;
    p.H = H;
    p.wait_ns = wait_ns;
    p.timeline = timeline;  // gate/up GEMM; the down GEMM stamps the next 12 x 256 words
    p.ready = ready;
    p.ready_cap = cap_gu;
    p.ready_tiles = I / kBM;
    p.withhold = withhold;
    const int optin = g_tc_smem_optin[dev];

    // Shared memory: header, raw ring, weight-tile ring (1024-aligned), then
    // the activation ring, sized by rings() below.
    auto rings = [&](int nmat) -> size_t {
        (void)nmat;
        // The stage ring (weight tiles) covers the round trip tile ready ->
        // MMA issued -> complete -> slot free; the raw ring (one block of every
        // row per slot) covers the HBM latency of the weights; the activation
        // ring (slots of the chunk capacity's rows, padded so the MMA's
        // M-row read of the last slot stays inside the ring) covers the
        // copies of the activation rows.  Preference, for chunks of at most
        // 64 slots: at least 4 activation slots, then the deepest stage ring
        // (4..2), raw ring (3..2) and activation ring (8..2); larger chunks
        // (and, failing that, small ones) take at least 2 activation slots.
        p.r_off = kHead;
        p.b_slot = cap * kBK * 2;
        const int pad = std::max(0, p.mrows * kBK * 2 - p.b_slot);
        for (int nb_min = cap <= 64 ? 4 : 2; nb_min >= 2; nb_min -= 2)
            for (int ns = 4; ns >= 2; --ns)
                for (int nr = 3; nr >= 2; --nr)
                    for (int nb = 8; nb >= nb_min; --nb) {
                        const int s_off = (kHead + nr * 2 * kRawMat + 1023) & ~1023;
                        const int b_off = s_off + ns * kStageSlot;
                        const size_t smem = size_t(b_off) + size_t(nb) * p.b_slot + pad;
                        if (smem <= size_t(optin)) {
                            p.nr = nr, p.ns = ns, p.nb = nb, p.s_off = s_off, p.b_off = b_off;
                            return smem;
                        }
                    }
        return 0;
    };

    // gate/up: A = gate and up rows (I per expert), B = x16 rows (slot p -> token p / k)
    p.mode = 0;
    p.K = H;
    p.row_tiles = I / kBM;
    p.item_rows = kBM;
    p.y_off1 = 0;
    p.rows_per_expert = I;
    if (!encode_act_map(&p.mapB, x16, rows, H)) return cudaErrorInvalidValue;
    if (!encode_raw_map(&p.raw0, gate, E, I, H / kQK) || !encode_raw_map(&p.raw1, up, E, I, H / kQK))
        return cudaErrorInvalidValue;
    size_t smem = rings(2);
    if (smem == 0) return cudaErrorInvalidValue;
    launch_pdl(grouped_gemm_kernel, dim3(num_sms), dim3(kThreads), size_t(smem), s, p);

    // down: A = down rows (H per expert), B = h16 rows (slot p)
    p.mode = 1;
    cap = cap_dn;
    p.mh = cap > kBM ? 2 : 1;
    p.mrows = cap <= 64 ? 64 : kBM;
    if (cap_dn != cap_gu) {
        p.chunks = chunks_dn;
        p.nchunks = &hdr->tc_chunks_dn;
    }
    p.timeline = timeline ? timeline + 12 * 256 : nullptr;
    p.K = I;
    p.row_tiles = H / (2 * kBM);
    p.item_rows = 2 * kBM;
    p.y_off1 = kBM;
    p.rows_per_expert = H;
    if (!encode_act_map(&p.mapB, h16, rows, I)) return cudaErrorInvalidValue;
    if (!encode_raw_map(&p.raw0, down, E, H, I / kQK)) return cudaErrorInvalidValue;
    p.raw1 = p.raw0;
    smem = rings(2);
    if (smem == 0) return cudaErrorInvalidValue;
    launch_pdl(grouped_gemm_kernel, dim3(num_sms), dim3(kThreads), size_t(smem), s, p);
    return cudaGetLastError();
}

}  // namespace moeq4k
