// Token->expert permutation: histogram of the routing, exclusive scan, and a
// stable scatter of slot ids into per-expert lists.
//
// The pages run the layer one position at a time (forward_qwen3_moe.rs,
// aprender-serve 0.35.0, step 2g of forward_qwen3_moe); grouping the slots
// of a batch by expert lets every expert's weights stream from HBM once per
// call whatever the batch size.  The order inside an expert's list is the
// slot order p = t*k + j, so the grouping is deterministic (no atomics
// decide positions).
//
// Batches of up to kSmallPermSlots slots take one single-CTA launch (below);
// larger ones three launches over blocks of kPermSlots consecutive slots
// (either way the launch that knows the expert offsets also writes the
// grouped GEMMs' chunk plans when asked):
//   count    each block's per-expert counts;
//   scan     per expert, the exclusive prefix of the block counts (in
//            place), the totals, their exclusive scan (offs) and the list of
//            active experts;
//   scatter  each block ranks its slots among equal experts (warp
//            __match_any_sync ranks, per-warp counts prefix-summed across the
//            block's warps) and writes every slot to
//              offs[e] + (slots of e in earlier blocks) + (in earlier warps)
//                      + (earlier lanes),
//            recording that position for the slot as well (-1 for a slot
//            whose expert index is invalid).
#include "common.cuh"
#include "kernels.cuh"

namespace moeq4k {

namespace {
constexpr int kWarpsPerBlock = kPermSlots / 32;
}

__global__ void __launch_bounds__(kPermSlots) permute_count_kernel(const int32_t *__restrict__ idx,
                                                                   int n, int E,
                                                                   int32_t *__restrict__ blockcnt,
                                                                   WsHeader *hdr) {
    pdl_enter();
    __shared__ int32_t cnt[kMaxE];
    for (int e = threadIdx.x; e < E; e += blockDim.x) cnt[e] = 0;
    __syncthreads();
    const int p = blockIdx.x * kPermSlots + threadIdx.x;
    if (p < n) {
        const int e = idx[p];
        if (e >= 0 && e < E) {
            atomicAdd(&cnt[e], 1);
        } else {
            record_status(hdr, MOE_ERR_EXPERT_RANGE, e);
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) blockcnt[size_t(blockIdx.x) * E + e] = cnt[e];
}

// One CTA of 1024 threads.  The block counts pass through shared memory 32
// blocks at a time (coalesced loads and stores); thread e keeps expert e's
// running total and rewrites its column of the tile as exclusive prefixes.
// Then warp 0 scans the expert totals, and warps 0 and 1 write the chunk
// plans asked for.
__global__ void __launch_bounds__(1024) permute_scan_kernel(int nblocks, int E,
                                                            int32_t *__restrict__ blockcnt,
                                                            int32_t *__restrict__ counts,
                                                            int32_t *__restrict__ offs,
                                                            int32_t *__restrict__ active,
                                                            int32_t *__restrict__ nactive,
                                                            ChunkPlan pa, ChunkPlan pb) {
    pdl_enter();
    __shared__ int32_t tile[32][kMaxE + 1];
    __shared__ int32_t tot[kMaxE];
    __shared__ int32_t s_offs[kMaxE + 1];
    __shared__ int32_t s_active[kMaxE];
    __shared__ int32_t s_na;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int run = 0;  // thread e < E: slots of expert e in the blocks so far
    for (int b0 = 0; b0 < nblocks; b0 += 32) {
        const int nb = min(32, nblocks - b0);
        int32_t *src = blockcnt + size_t(b0) * E;
        for (int i = tid; i < nb * E; i += blockDim.x) tile[i / E][i % E] = src[i];
        __syncthreads();
        if (tid < E) {
            for (int b = 0; b < nb; ++b) {
                const int c = tile[b][tid];
                tile[b][tid] = run;
                run += c;
            }
        }
        __syncthreads();
        for (int i = tid; i < nb * E; i += blockDim.x) src[i] = tile[i / E][i % E];
        __syncthreads();
    }
    if (tid < E) tot[tid] = run;
    __syncthreads();
    if (warp == 0) {
        int carry = 0, na = 0;
        for (int base = 0; base < E; base += 32) {
            const int ee = base + lane;
            const int v = (ee < E) ? tot[ee] : 0;
            int incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += u;
            }
            if (ee < E) {
                offs[ee] = carry + incl - v;
                s_offs[ee] = carry + incl - v;
                counts[ee] = v;
            }
            carry += __shfl_sync(0xffffffffu, incl, 31);
            // active experts in ascending order
            const bool on = (ee < E) && v > 0;
            const unsigned m = __ballot_sync(0xffffffffu, on);
            if (on) {
                const int a = na + __popc(m & ((1u << lane) - 1u));
                active[a] = ee;
                s_active[a] = ee;
            }
            na += __popc(m);
        }
        if (lane == 0) {
            offs[E] = carry;
            s_offs[E] = carry;
            *nactive = na;
            s_na = na;
        }
    }
    __syncthreads();
    if (warp == 0 && pa.cap > 0) warp_plan_chunks(s_offs, s_active, s_na, pa.cap, pa.chunks, pa.count);
    if (warp == 1 && pb.cap > 0) warp_plan_chunks(s_offs, s_active, s_na, pb.cap, pb.chunks, pb.count);
}

__global__ void __launch_bounds__(kPermSlots) permute_scatter_kernel(
    const int32_t *__restrict__ idx, int n, int E, const int32_t *__restrict__ blockcnt,
    const int32_t *__restrict__ offs, int32_t *__restrict__ perm, int32_t *__restrict__ slotpos,
    WsHeader *hdr) {
    pdl_enter();
    __shared__ int32_t table[kWarpsPerBlock][kMaxE];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int p = blockIdx.x * kPermSlots + tid;
    const int e = (p < n) ? idx[p] : -1;
    const bool ok = (e >= 0 && e < E);
    const unsigned peers = __match_any_sync(0xffffffffu, ok ? e : -1);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    for (int i = tid; i < kWarpsPerBlock * E; i += blockDim.x) table[i / E][i % E] = 0;
    __syncthreads();
    if (ok && rank == 0) table[warp][e] = __popc(peers);
    __syncthreads();
    // per-expert exclusive prefix across the block's warps, plus the block's base
    for (int ee = tid; ee < E; ee += blockDim.x) {
        int run = offs[ee] + blockcnt[size_t(blockIdx.x) * E + ee];
        for (int w = 0; w < kWarpsPerBlock; ++w) {
            const int c = table[w][ee];
            table[w][ee] = run;
            run += c;
        }
    }
    __syncthreads();
    if (ok) {
        const int pos = table[warp][e] + rank;
        if (pos >= 0 && pos < n) {
            perm[pos] = p;
            slotpos[p] = pos;
        } else {
            record_status(hdr, MOE_ERR_INTERNAL, 400000000 + (pos & 0xffffff));
        }
    } else if (p < n) {
        slotpos[p] = -1;  // an invalid expert index: the slot has no sorted row
    }
}

// Up to kSmallPermSlots slots, one CTA of 1024 threads does it all: shared
// per-expert counts, the scan of the totals (offs, counts, the active list),
// then the slots in passes of 1024 in slot order: warp ranks among equal
// experts (__match_any_sync), per-warp counts prefix-summed across the 32
// warps on top of each expert's running base, positions written.  Stable by
// construction, so the result equals the multi-launch path's.  Warps 0 and
// 1 then write the chunk plans asked for.
constexpr int kSmallPerSlot = kSmallPermSlots / 1024;  // slots per thread

__global__ void __launch_bounds__(1024) permute_small_kernel(
    const int32_t *__restrict__ idx, int n, int E, int32_t *__restrict__ counts,
    int32_t *__restrict__ offs, int32_t *__restrict__ perm, int32_t *__restrict__ slotpos,
    int32_t *__restrict__ active, int32_t *__restrict__ nactive, WsHeader *hdr, ChunkPlan pa,
    ChunkPlan pb) {
    pdl_enter();
    __shared__ int32_t run[kMaxE];          // counts, then each expert's next position
    __shared__ int32_t s_offs[kMaxE + 1];
    __shared__ int32_t s_active[kMaxE];
    __shared__ int32_t s_na;
    __shared__ int32_t table[32][kMaxE];    // per-warp counts of one pass
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int e = tid; e < E; e += 1024) run[e] = 0;
    __syncthreads();
    int ev[kSmallPerSlot];
#pragma unroll
    for (int i = 0; i < kSmallPerSlot; ++i) {
        const int p = 1024 * i + tid;
        ev[i] = p < n ? idx[p] : -1;
        if (ev[i] >= 0 && ev[i] < E) {
            atomicAdd(&run[ev[i]], 1);
        } else if (p < n) {
            record_status(hdr, MOE_ERR_EXPERT_RANGE, ev[i]);
            ev[i] = -1;
        } else {
            ev[i] = -1;
        }
    }
    __syncthreads();
    if (warp == 0) {
        int carry = 0, na = 0;
        for (int base = 0; base < E; base += 32) {
            const int ee = base + lane;
            const int v = (ee < E) ? run[ee] : 0;
            int incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += u;
            }
            if (ee < E) {
                s_offs[ee] = carry + incl - v;
                offs[ee] = carry + incl - v;
                counts[ee] = v;
            }
            carry += __shfl_sync(0xffffffffu, incl, 31);
            const bool on = (ee < E) && v > 0;
            const unsigned m = __ballot_sync(0xffffffffu, on);
            if (on) {
                const int a = na + __popc(m & ((1u << lane) - 1u));
                active[a] = ee;
                s_active[a] = ee;
            }
            na += __popc(m);
        }
        if (lane == 0) {
            s_offs[E] = carry;
            offs[E] = carry;
            *nactive = na;
            s_na = na;
        }
    }
    __syncthreads();
    for (int e = tid; e < E; e += 1024) run[e] = s_offs[e];
    for (int i = 0; i < kSmallPerSlot; ++i) {
        if (1024 * i >= n) break;  // uniform
        for (int q = tid; q < 32 * E; q += 1024) table[q / E][q % E] = 0;
        __syncthreads();
        const int p = 1024 * i + tid;
        const int e = ev[i];
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        const int rank = __popc(peers & ((1u << lane) - 1u));
        if (e >= 0 && rank == 0) table[warp][e] = __popc(peers);
        __syncthreads();
        for (int ee = tid; ee < E; ee += 1024) {
            int r = run[ee];
            for (int w = 0; w < 32; ++w) {
                const int c = table[w][ee];
                table[w][ee] = r;
                r += c;
            }
            run[ee] = r;
        }
        __syncthreads();
        if (e >= 0) {
            const int pos = table[warp][e] + rank;
            if (pos >= 0 && pos < n) {
                perm[pos] = p;
                slotpos[p] = pos;
            } else {
                record_status(hdr, MOE_ERR_INTERNAL, 410000000 + (pos & 0xffffff));
            }
        } else if (p < n) {
            slotpos[p] = -1;  // an invalid expert index: the slot has no sorted row
        }
        __syncthreads();  // before the next pass clears the table
    }
    if (warp == 0 && pa.cap > 0) warp_plan_chunks(s_offs, s_active, s_na, pa.cap, pa.chunks, pa.count);
    if (warp == 1 && pb.cap > 0) warp_plan_chunks(s_offs, s_active, s_na, pb.cap, pb.chunks, pb.count);
}

cudaError_t launch_permute(const int32_t *idx, int T, int k, int E, int32_t *counts, int32_t *offs,
                           int32_t *perm, int32_t *active, int32_t *nactive, int32_t *blockcnt,
                           int32_t *slotpos, WsHeader *hdr, cudaStream_t s, const ChunkPlan &pa,
                           const ChunkPlan &pb) {
    const int n = T * k;
    if (n <= kSmallPermSlots) {
        launch_pdl(permute_small_kernel, dim3(1), dim3(1024), size_t(0), s, idx, n, E, counts, offs,
                   perm, slotpos, active, nactive, hdr, pa, pb);
        return cudaGetLastError();
    }
    const int nb = (n + kPermSlots - 1) / kPermSlots;
    launch_pdl(permute_count_kernel, dim3(nb), dim3(kPermSlots), size_t(0), s, idx, n, E, blockcnt, hdr);
    launch_pdl(permute_scan_kernel, dim3(1), dim3(1024), size_t(0), s, nb, E, blockcnt, counts, offs,
               active, nactive, pa, pb);
    launch_pdl(permute_scatter_kernel, dim3(nb), dim3(kPermSlots), size_t(0), s, idx, n, E, blockcnt, offs, perm, slotpos, hdr);
    return cudaGetLastError();
}

}  // namespace moeq4k
