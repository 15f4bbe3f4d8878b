// Prefill: the expert FFN of a large batch as two grouped GEMMs on the
// tcgen05 tensor cores, with the Q4_K weights dequantised to fp16 in shared
// memory on the way in.
//
// forward_qwen3_moe.rs (aprender-serve 0.35.0), step 2g of forward_qwen3_moe
// runs every position through the layer on its own; tokens are independent,
// so the slots routed to one expert form the columns of one GEMM per expert:
//   gate/up:  G = Wg[e] X_e^T, U = Wu[e] X_e^T  (M = 128 weight rows per tile,
//             N = up to 256 tokens, K = H), epilogue h = SiLU(G) * U (fp16);
//   down:     O = Wd[e] H_e^T (K = I), epilogue o[p, row] in fp32, followed
//             by the slot-ordered combine kernel.
// The activations are first gathered into expert-sorted rows (fp16), and h
// is written in that order too, so every activation tile is one contiguous
// block of rows.
//
// One persistent CTA per SM takes work items (expert chunk of <= cap slots x
// 128 rows each of gate and up, or 256 rows of down: two A operands that
// share every activation tile) from an atomic counter; cap is 256, or the
// batch's token count rounded up to 32 when that is smaller.  12 warps:
//   thread 32   stages the raw Q4_K bytes of each K stage (64 weights per
//               row: the 16-byte block head and the 32 code bytes) for the
//               tile's 128 rows with two 2-D TMA copies per matrix, into a
//               ring of raw slots as deep as shared memory allows (5 stages
//               at cap 256, up to 16 for small batches): these come from HBM
//               and need the most latency cover;
//   warps 4-11  dequantise them into fp16 K-major tiles with the 128-byte
//               swizzle (generic stores, then a proxy fence), into a ring of
//               weight tiles (2 slots; 4 when cap <= 64, where each stage's
//               MMAs are short and the ring covers their completion latency);
//   thread 64   loads the chunk's activation tile (its sorted rows rounded
//               up to 32, x 64 K, fp16) with 2-D TMA copies of 32 rows that
//               apply the 128-byte swizzle, into a ring of 3 slots of cap
//               rows (4 when cap <= 64);
//   thread 0    issues tcgen05.mma (fp16 x fp16 -> fp32 in tensor memory)
//               once a stage's weight and activation tiles are both in, and
//               commits its completion to both rings' "empty" mbarriers;
//   all warps   read the accumulators back (tcgen05.ld) for the epilogue
//               once the item's MMAs are complete, each warp a third of the
//               columns of its TMEM lane quadrant.
// Every wait is bounded by a global-timer deadline and records
// MOE_ERR_TIMEOUT when it runs out.
#include <cuda.h>
#include <cuda_fp16.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.cuh"
#include "tcgen05.cuh"

namespace moeq4k {
namespace ptc {

constexpr int kThreads = 384;
constexpr int kBM = 128;   // weight rows per tile
constexpr int kBN = 256;   // tokens per tile (max)
constexpr int kBK = 64;    // K per stage
constexpr int kTileA = kBM * kBK * 2;
constexpr int kBoxRows = 32;                   // activation rows per TMA box
constexpr int kBoxB = kBoxRows * kBK * 2;
constexpr int kHead = 2048;  // barriers, item info, token list
constexpr int kDeq = 256;      // warps 4-11
constexpr int kMaxSlots = 16;  // per ring
constexpr int kRawHead = kBM * 16;               // block heads of a tile's rows
constexpr int kRawMat = kBM * (16 + 32);         // one matrix's raw bytes of a stage

struct Params {
    CUtensorMap head0, codes0;  // raw Q4_K bytes of A0 as [E*rows][row bytes] uint8:
    CUtensorMap head1, codes1;  //   boxes of 16 B (block head) and 32 B (codes) x 128 rows
    CUtensorMap mapB;           // activations [T*k sorted rows][K] fp16, 128-byte swizzle
    int mode;                   // 0: gate/up + SwiGLU -> h16; 1: down -> o
    int K;                      // reduction length
    int row_tiles;              // weight rows per expert / item_rows
    int item_rows;              // weight rows per item: 128 (gate/up: 128 of each) or 256
    int y_off1;                 // row offset of the second A operand: 0 (up) or 128 (down)

    const int32_t *offs, *perm;
    const TcChunk *chunks;
    WsHeader *hdr;              // work counters, chunk count, status
    __half *h16;                // mode 0 output [T*k sorted rows][I]
    float *o;                   // mode 1 output [T*k][H]
    int I, H;
    int rows_per_expert;        // I (mode 0) or H (mode 1)
    int nr, r_off;              // raw ring: slots, byte offset (slot = nmat * kRawMat bytes)
    int na, a_off;              // weight-tile ring: slots, byte offset (slot = nmat * kTileA)
    int nb, b_off, b_slot;      // activation-tile ring: slots, byte offset, bytes per slot
                                //   (chunk capacity x 128 B)
    unsigned long long wait_ns;
};

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

__device__ __forceinline__ float u6f(uint32_t v) { return __uint_as_float(0x4B000000u | v) - 8388608.0f; }

// (d*sc, dmin*m) of sub-blocks 2c and 2c+1 from a 16-byte block head.
__device__ __forceinline__ void head_scales(const uint4 &h, int c, float &a0, float &b0, float &a1,
                                            float &b1) {
    const int j0 = 2 * c, j1 = 2 * c + 1;
    uint32_t s0, m0, s1, m1;
    if (c < 2) {
        s0 = (h.y >> (8 * j0)) & 63u;
        m0 = (h.z >> (8 * j0)) & 63u;
        s1 = (h.y >> (8 * j1)) & 63u;
        m1 = (h.z >> (8 * j1)) & 63u;
    } else {
        const int a = j0 - 4, b = j1 - 4;
        s0 = ((h.w >> (8 * a)) & 15u) | (((h.y >> (8 * a + 6)) & 3u) << 4);
        m0 = ((h.w >> (8 * a + 4)) & 15u) | (((h.z >> (8 * a + 6)) & 3u) << 4);
        s1 = ((h.w >> (8 * b)) & 15u) | (((h.y >> (8 * b + 6)) & 3u) << 4);
        m1 = ((h.w >> (8 * b + 4)) & 15u) | (((h.z >> (8 * b + 6)) & 3u) << 4);
    }
    const float2 dd = __half22float2(*reinterpret_cast<const __half2 *>(&h.x));
    a0 = dd.x * u6f(s0);
    a1 = dd.x * u6f(s1);
    b0 = dd.y * u6f(m0);
    b1 = dd.y * u6f(m1);
}

// K order inside the fp16 operand tiles: within each aligned group of four,
// positions 1 and 2 are swapped (the dequantiser below produces that order
// two codes per instruction; the activation operands are written in the same
// order, so every dot product is unchanged).
__host__ __device__ inline int kperm(int k) { return (k & ~3) | ((k & 1) << 1) | ((k >> 1) & 1); }

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }
__device__ __forceinline__ __half2 bits_h2(uint32_t u) { return *reinterpret_cast<__half2 *>(&u); }

// w = q*a - b for the 8 codes of one 16-byte output chunk: nibble `shift`
// (0 low, 4 high) of bytes 0..3 of v0, then of v1.  (v >> s) & 0x000F000F |
// 0x64006400 puts two codes into the low mantissa bits of the fp16 value
// 1024 (bytes 0 and 2, or 1 and 3); subtracting 1024 is exact, then one
// fused multiply-add per pair applies d*sc and dmin*m with one rounding.
// Output order: codes 0, 2, 1, 3, 4, 6, 5, 7.
__device__ __forceinline__ uint4 weights8(uint32_t v0, uint32_t v1, int shift, __half2 a2,
                                          __half2 nb2) {
    const __half2 k1024 = bits_h2(0x64006400u);
    const uint32_t p0 = ((v0 >> shift) & 0x000F000Fu) | 0x64006400u;
    const uint32_t p1 = ((v0 >> (shift + 8)) & 0x000F000Fu) | 0x64006400u;
    const uint32_t p2 = ((v1 >> shift) & 0x000F000Fu) | 0x64006400u;
    const uint32_t p3 = ((v1 >> (shift + 8)) & 0x000F000Fu) | 0x64006400u;
    uint4 r;
    r.x = h2_bits(__hfma2(__hsub2(bits_h2(p0), k1024), a2, nb2));
    r.y = h2_bits(__hfma2(__hsub2(bits_h2(p1), k1024), a2, nb2));
    r.z = h2_bits(__hfma2(__hsub2(bits_h2(p2), k1024), a2, nb2));
    r.w = h2_bits(__hfma2(__hsub2(bits_h2(p3), k1024), a2, nb2));
    return r;
}

struct RawStage {
    uint4 head, q0, q1;  // block head and the 32 code bytes of this stage's 64 weights
};

// Row r of a matrix's raw stage: its 16-byte block head and 32 code bytes.
__device__ __forceinline__ RawStage raw_from_smem(const uint8_t *mat, int r) {
    RawStage v;
    v.head = *reinterpret_cast<const uint4 *>(mat + 16 * r);
    v.q0 = *reinterpret_cast<const uint4 *>(mat + kRawHead + 32 * r);
    v.q1 = *reinterpret_cast<const uint4 *>(mat + kRawHead + 32 * r + 16);
    return v;
}

// Write `nchunks` 16-byte chunks (weights 8j..8j+7 for j in [j0, j0+nchunks),
// in the kperm order) of row `r` of the stage's 64 weights into a swizzled
// tile.
__device__ __forceinline__ void store_row(uint8_t *tile, int r, const RawStage &raw, int s, int j0,
                                          int nchunks) {
    float a0, b0, a1, b1;
    head_scales(raw.head, s & 3, a0, b0, a1, b1);
    const __half2 A0 = __float2half2_rn(a0), A1 = __float2half2_rn(a1);
    const __half2 NB0 = __float2half2_rn(-b0), NB1 = __float2half2_rn(-b1);
    const uint32_t w[8] = {raw.q0.x, raw.q0.y, raw.q0.z, raw.q0.w,
                           raw.q1.x, raw.q1.y, raw.q1.z, raw.q1.w};
#pragma unroll
    for (int jj = 0; jj < 8; ++jj) {
        if (jj < j0 || jj >= j0 + nchunks) continue;
        // chunk jj < 4: low nibbles of code bytes 8jj..8jj+7 (sub-block 2c);
        // chunk jj >= 4: high nibbles of bytes 8(jj-4).. (sub-block 2c+1)
        const int wb = 2 * (jj & 3);
        const uint4 out = jj < 4 ? weights8(w[wb], w[wb + 1], 0, A0, NB0)
                                 : weights8(w[wb], w[wb + 1], 4, A1, NB1);
        *reinterpret_cast<uint4 *>(tile + tc::sw128_offset(r, 8 * jj)) = out;
    }
}

__global__ void __launch_bounds__(kThreads, 1) grouped_gemm_kernel(const __grid_constant__ Params p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t *rfull = reinterpret_cast<uint64_t *>(smem);
    uint64_t *rempty = rfull + kMaxSlots;
    uint64_t *afull = rempty + kMaxSlots;
    uint64_t *aempty = afull + kMaxSlots;
    uint64_t *bfull = aempty + kMaxSlots;
    uint64_t *bempty = bfull + kMaxSlots;
    uint64_t *done = bempty + kMaxSlots;
    uint64_t *drain = done + 1;
    uint32_t *tmem_ptr = reinterpret_cast<uint32_t *>(drain + 1);
    int *info = reinterpret_cast<int *>(tmem_ptr + 4);   // [0] item, [1] abort, [2] accumulators ready
    int *toks = reinterpret_cast<int *>(smem + 1024);    // slot ids of the chunk (<= 256)
    uint8_t *rring = smem + p.r_off;
    uint8_t *aring = smem + p.a_off;
    uint8_t *bring = smem + p.b_off;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int NR = p.nr, NA = p.na, NB = p.nb;
    constexpr int nmat = 2;  // two A operands per item: gate and up, or two 128-row halves
    const int S = p.K / kBK;  // stages per item
    const uint64_t deadline = global_timer_ns() + p.wait_ns;
    const uint32_t tcols = 512u;  // two 128 x 256 fp32 accumulators

    if (tid == 0) {
        for (int i = 0; i < NR; ++i) {
            mbar_init(rfull + i, 1);           // the TMA thread's arrival + its bytes
            mbar_init(rempty + i, kDeq / 32);  // one arrival per dequant warp
        }
        for (int i = 0; i < NA; ++i) {
            mbar_init(afull + i, kDeq / 32);
            mbar_init(aempty + i, 1);          // MMA completion
        }
        for (int i = 0; i < NB; ++i) {
            mbar_init(bfull + i, 1);
            mbar_init(bempty + i, 1);
        }
        mbar_init(done, 1);
        mbar_init(drain, 1);
        info[1] = 0;
        fence_mbar_init();
    }
    if (warp == 0) tc::tmem_alloc(tmem_ptr, tcols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t taddr = *tmem_ptr;
    const int total = p.hdr->tc_chunks * p.row_tiles;

    uint32_t gs = 0;     // stages processed by this CTA (same count in every role)
    uint32_t items = 0;  // items processed by this CTA
    uint32_t issued = 0; // threads 32 and 64: stages whose copies this thread issued
    while (true) {
        if (tid == 0) info[0] = int(atomicAdd(&p.hdr->tc_work[p.mode], 1u));
        __syncthreads();
        const int item = info[0];
        if (item >= total || info[1]) break;
        const TcChunk ch = p.chunks[item / p.row_tiles];
        const int rt = item % p.row_tiles;
        const int ntok = ch.tok_cnt;
        const int nmma = (ntok + 15) & ~15;
        for (int n = tid; n < ntok; n += kThreads) toks[n] = p.perm[p.offs[ch.e] + ch.tok_off + n];
        __syncthreads();

        if (warp >= 4) {
            // ---- dequantise weight rows (raw stage in shared memory) into the A tile(s)
            const int dq = tid - 128;
            const int m = dq >> 7;  // A operand: gate / up, or the first / second 128 rows
            const int r = dq & 127, j0 = 0, nch = 8;
            for (int s = 0; s < S; ++s) {
                const uint32_t g = gs + s, rs = g % NR, as = g % NA;
                if (!wait_bar(rfull + rs, (g / NR) & 1, deadline, p.hdr, 16)) {
                    info[1] = 1;
                    break;
                }
                const RawStage cur = raw_from_smem(rring + size_t(rs) * nmat * kRawMat + m * kRawMat, r);
                // The TMA that refills this slot writes through the async proxy:
                // without a proxy fence after the reads, a refill could land
                // before reads still in flight are performed.
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(rempty + rs);
                if (g >= uint32_t(NA) &&
                    !wait_bar(aempty + as, ((g / NA) - 1) & 1, deadline, p.hdr, 11)) {
                    info[1] = 1;
                    break;
                }
                store_row(aring + size_t(as) * nmat * kTileA + m * kTileA, r, cur, s, j0, nch);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(afull + as);
            }
        } else if (tid == 0) {
            // ---- MMA issue
            const uint32_t idesc = tc::idesc_f16_f32(kBM, nmma);
            for (int s = 0; s < S; ++s) {
                const uint32_t g = gs + s, as = g % NA, bs = g % NB;
                if (!wait_bar(afull + as, (g / NA) & 1, deadline, p.hdr, 13) ||
                    !wait_bar(bfull + bs, (g / NB) & 1, deadline, p.hdr, 18)) {
                    info[1] = 1;
                    break;
                }
                tc::fence_after_sync();
                const uint32_t a0 = smem_addr(aring + size_t(as) * nmat * kTileA), a1 = a0 + kTileA;
                const uint32_t b = smem_addr(bring + size_t(bs) * p.b_slot);
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk) {
                    const uint64_t bd = tc::smem_desc_sw128(b + 32 * kk);
                    const bool acc = s > 0 || kk > 0;
                    tc::mma_f16(taddr, tc::smem_desc_sw128(a0 + 32 * kk), bd, idesc, acc);
                    tc::mma_f16(taddr + 256, tc::smem_desc_sw128(a1 + 32 * kk), bd, idesc, acc);
                }
                tc::commit_arrive(aempty + as);
                tc::commit_arrive(bempty + bs);
            }
            tc::commit_arrive(done);
        } else if (tid == 64) {
            // ---- activation tile of each stage by TMA: the chunk's sorted rows
            // (rounded up to 32) x 64 K, in boxes of 32 rows
            const int row0 = p.offs[ch.e] + ch.tok_off;
            const int nbox = (nmma + kBoxRows - 1) / kBoxRows;
            for (int s = 0; s < S; ++s) {
                const uint32_t g = gs + s, bs = g % NB;
                if (g >= uint32_t(NB) &&
                    !wait_bar(bempty + bs, ((g / NB) - 1) & 1, deadline, p.hdr, 12)) {
                    info[1] = 1;
                    break;
                }
                mbar_arrive_expect_tx(bfull + bs, nbox * kBoxB);
                ++issued;
                for (int i = 0; i < nbox; ++i)
                    tma_load_2d(bring + size_t(bs) * p.b_slot + i * kBoxB, &p.mapB, s * kBK,
                                row0 + i * kBoxRows, bfull + bs);
            }
        } else if (tid == 32) {
            // ---- raw bytes of each stage by TMA: block head + the stage's 32 code bytes
            const int y = ch.e * p.rows_per_expert + rt * p.item_rows;
            for (int s = 0; s < S; ++s) {
                const uint32_t g = gs + s, rs = g % NR;
                if (g >= uint32_t(NR) &&
                    !wait_bar(rempty + rs, ((g / NR) - 1) & 1, deadline, p.hdr, 17)) {
                    info[1] = 1;
                    break;
                }
                uint8_t *dst = rring + size_t(rs) * nmat * kRawMat;
                const int xh = (s >> 2) * kBlockBytes, xq = xh + 16 + 32 * (s & 3);
                mbar_arrive_expect_tx(rfull + rs, nmat * kRawMat);
                ++issued;
                tma_load_2d(dst, &p.head0, xh, y, rfull + rs);
                tma_load_2d(dst + kRawHead, &p.codes0, xq, y, rfull + rs);
                tma_load_2d(dst + kRawMat, &p.head1, xh, y + p.y_off1, rfull + rs);
                tma_load_2d(dst + kRawMat + kRawHead, &p.codes1, xq, y + p.y_off1, rfull + rs);
            }
        }

        // ---- epilogue, by all 12 warps: warp w reads the TMEM lanes of
        // quadrant w % 4 (32 of the tile's weight rows) for column part w / 4
        // of three (in 8-column units)
        __syncthreads();  // every role is past its main loop
        if (tid == 0) info[2] = wait_bar(done, items & 1, deadline, p.hdr, 14) ? 1 : 0;
        __syncthreads();
        tc::fence_after_sync();
        if (info[2] != 0 && !info[1]) {
            const int q = warp & 3, part = warp >> 2;
            const int units = nmma >> 3;
            const int u_lo = units * part / 3, u_hi = units * (part + 1) / 3;
            const int row = rt * p.item_rows + q * 32 + lane;
            const int prow = kperm(row);  // h is the down GEMM's K: stored in kperm order
            const int pos0 = p.offs[ch.e] + ch.tok_off;  // sorted row of column 0
            const uint32_t lanebase = taddr + (uint32_t(q * 32) << 16);
            for (int uu = u_lo; uu < u_hi; ++uu) {
                const int n0 = 8 * uu;
                float g[8], u[8];
                tc::tmem_ld8(lanebase + n0, g);
                tc::tmem_ld8(lanebase + 256 + n0, u);
                if (p.mode == 0) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int n = n0 + j;
                        if (n < ntok) {
                            // SiLU(g) * u with the fast exponential and divide: the
                            // result is rounded to fp16
                            const float e = __expf(fminf(-g[j], 80.0f));
                            p.h16[size_t(pos0 + n) * p.I + prow] =
                                __float2half_rn(__fdividef(g[j], 1.0f + e) * u[j]);
                        }
                    }
                } else {
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int n = n0 + j;
                        if (n < ntok) {
                            float *orow = p.o + size_t(toks[n]) * p.H;
                            orow[row] = g[j];
                            orow[row + kBM] = u[j];
                        }
                    }
                }
            }
        }
        tc::fence_before_sync();
        gs += S;
        ++items;
        __syncthreads();
    }
    // every issued MMA must be complete before the tensor memory is released
    if (tid == 0) {
        tc::commit_arrive(drain);
        wait_bar(drain, 0, global_timer_ns() + p.wait_ns, p.hdr, 15);
    }
    // After a timed-out wait the consumers may have left copies unawaited:
    // each copying thread waits (bounded) for the last phase it started on
    // every slot of its ring, so no copy still targets this CTA's shared
    // memory when it exits.  (Without a time-out every phase was consumed.)
    if (info[1] && (tid == 32 || tid == 64)) {
        uint64_t *bars = tid == 32 ? rfull : bfull;
        const uint32_t n = tid == 32 ? uint32_t(NR) : uint32_t(NB);
        const uint64_t limit = global_timer_ns() + p.wait_ns;
        for (uint32_t i = 0; i < n && i < issued; ++i) {
            const uint32_t g = issued - 1 - i;
            wait_bar(bars + g % n, (g / n) & 1, limit, p.hdr, 19);
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
                                   int T, int k, int H, __half *__restrict__ xs) {
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

// Chunks of <= cap slots per active expert, in active order, and the work
// counters reset.  One warp: lanes take active experts in turns of 32, a
// warp scan gives each expert's first chunk.
__global__ void plan_kernel(const int32_t *__restrict__ offs, const int32_t *__restrict__ active,
                            const int32_t *__restrict__ nactive, int cap, TcChunk *chunks,
                            WsHeader *hdr) {
    const int lane = threadIdx.x & 31;
    if (threadIdx.x >= 32) return;
    const int na = *nactive;
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
    if (lane == 0) {
        hdr->tc_chunks = nc;
        hdr->tc_work[0] = 0;
        hdr->tc_work[1] = 0;
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
// nsb*144 bytes; box = `box_bytes` (16: block head, 32: codes of one stage)
// x 128 rows.  Every x coordinate used (block start, +16 + 32c) is a
// multiple of 16 bytes.
bool encode_raw_map(CUtensorMap *map, const void *base, int E, int rows, int nsb, int box_bytes) {
    const cuuint64_t dims[2] = {cuuint64_t(nsb) * kBlockBytes, cuuint64_t(E) * rows};
    const cuuint64_t strides[1] = {cuuint64_t(nsb) * kBlockBytes};
    const cuuint32_t box[2] = {cuuint32_t(box_bytes), cuuint32_t(ptc::kBM)};
    const cuuint32_t estr[2] = {1, 1};
    return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
bool encode_raw_maps(CUtensorMap *head, CUtensorMap *codes, const void *base, int E, int rows, int nsb) {
    return encode_raw_map(head, base, E, rows, nsb, 16) && encode_raw_map(codes, base, E, rows, nsb, 32);
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

cudaError_t launch_prefill_tc(int dev, const float *x, const uint8_t *gate, const uint8_t *up,
                              const uint8_t *down, int T, int H, int E, int k, int I,
                              const int32_t *offs, const int32_t *perm, const int32_t *slotpos,
                              const int32_t *active, const int32_t *nactive, __half *x16,
                              __half *h16, float *obuf, TcChunk *chunks, WsHeader *hdr,
                              int num_sms, unsigned long long wait_ns, cudaStream_t s) {
    using namespace ptc;
    gather_half_kernel<<<num_sms * 8, 256, 0, s>>>(x, slotpos, T, k, H, x16);
    // Chunk capacity: up to 256 slots, no more than the batch's tokens
    // (rounded to 32) so that small batches get deep rings; a larger expert
    // list (a caller's routing with repeated experts) is split into more chunks.
    const int cap = std::min(kBN, (T + kBoxRows - 1) / kBoxRows * kBoxRows);
    plan_kernel<<<1, 32, 0, s>>>(offs, active, nactive, cap, chunks, hdr);
    const int rows = T * k;

    Params p = {};
    p.offs = offs;
    p.perm = perm;
    p.chunks = chunks;
    p.hdr = hdr;
    p.h16 = h16;
    p.o = obuf;
    p.I = I;
    p.H = H;
    p.wait_ns = wait_ns;
    const int optin = g_tc_smem_optin[dev];

    // Shared memory: header, raw ring, weight-tile ring (1024-aligned), then
    // the activation ring (3 slots of the chunk capacity, 4 for chunks of at
    // most 64 slots); the raw ring takes what is left, up to kMaxSlots stages.
    auto rings = [&](int nmat) -> size_t {
        // small chunks make each stage's MMAs short, so the weight-tile ring
        // must cover the MMA completion round trips: 4 slots instead of 2
        p.na = cap <= 64 ? 4 : 2;
        p.b_slot = cap * kBK * 2;
        p.nb = cap <= 64 ? 4 : 3;
        p.r_off = kHead;
        for (int nr = kMaxSlots; nr >= 2; --nr) {
            p.nr = nr;
            p.a_off = (kHead + nr * nmat * kRawMat + 1023) & ~1023;
            p.b_off = p.a_off + p.na * nmat * kTileA;
            const size_t smem = size_t(p.b_off) + size_t(p.nb) * p.b_slot;
            if (smem <= size_t(optin)) return smem;
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
    if (!encode_raw_maps(&p.head0, &p.codes0, gate, E, I, H / kQK) ||
        !encode_raw_maps(&p.head1, &p.codes1, up, E, I, H / kQK))
        return cudaErrorInvalidValue;
    size_t smem = rings(2);
    if (smem == 0) return cudaErrorInvalidValue;
    grouped_gemm_kernel<<<num_sms, kThreads, smem, s>>>(p);

    // down: A = down rows (H per expert), B = h16 rows (slot p)
    p.mode = 1;
    p.K = I;
    p.row_tiles = H / (2 * kBM);
    p.item_rows = 2 * kBM;
    p.y_off1 = kBM;
    p.rows_per_expert = H;
    if (!encode_act_map(&p.mapB, h16, rows, I)) return cudaErrorInvalidValue;
    if (!encode_raw_maps(&p.head0, &p.codes0, down, E, H, I / kQK)) return cudaErrorInvalidValue;
    p.head1 = p.head0;
    p.codes1 = p.codes0;
    smem = rings(2);
    if (smem == 0) return cudaErrorInvalidValue;
    grouped_gemm_kernel<<<num_sms, kThreads, smem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace moeq4k
