// Token->expert permutation: histogram of the routing, exclusive scan, and a
// stable scatter of slot ids into per-expert lists.
//
// The pages run the layer one position at a time (forward_qwen3_moe.rs,
// aprender-serve 0.35.0, step 2g of forward_qwen3_moe); grouping the slots
// of a batch by expert lets every expert's weights stream from HBM once per
// call whatever the batch size.  The order inside an expert's list is the
// slot order p = t*k + j, so the grouping is deterministic (no atomics
// decide positions).
#include "common.cuh"
#include "kernels.cuh"

namespace moeq4k {

// One CTA of 1024 threads.  Slots are processed in chunks of 1024 in slot
// order; inside a chunk each warp ranks its lanes among equal experts with
// __match_any_sync, per-warp counts are prefix-summed per expert across the
// 32 warps, and every slot lands at
//   offs[e] + (slots of e in earlier chunks) + (in earlier warps) + (earlier lanes).
__global__ void __launch_bounds__(1024) permute_kernel(const int32_t *__restrict__ idx, int n,
                                                       int E, int32_t *__restrict__ counts,
                                                       int32_t *__restrict__ offs,
                                                       int32_t *__restrict__ perm,
                                                       int32_t *__restrict__ active,
                                                       int32_t *__restrict__ nactive,
                                                       WsHeader *hdr) {
    __shared__ int32_t cnt[kMaxE];
    __shared__ int32_t cursor[kMaxE];
    __shared__ int32_t table[32][kMaxE];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    for (int e = tid; e < E; e += blockDim.x) cnt[e] = 0;
    __syncthreads();
    for (int p = tid; p < n; p += blockDim.x) {
        int e = idx[p];
        if (e >= 0 && e < E) {
            atomicAdd(&cnt[e], 1);
        } else {
            record_status(hdr, MOE_ERR_EXPERT_RANGE, e);
        }
    }
    __syncthreads();
    // exclusive scan of cnt over E <= 256 entries: one warp
    if (warp == 0) {
        int carry = 0;
        for (int base = 0; base < E; base += 32) {
            int e = base + lane;
            int v = (e < E) ? cnt[e] : 0;
            int incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                int u = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += u;
            }
            if (e < E) {
                cursor[e] = carry + incl - v;
                offs[e] = carry + incl - v;
                counts[e] = v;
            }
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) offs[E] = carry;
        // active experts in ascending order
        int na = 0;
        for (int base = 0; base < E; base += 32) {
            int e = base + lane;
            bool on = (e < E) && cnt[e] > 0;
            unsigned m = __ballot_sync(0xffffffffu, on);
            if (on) active[na + __popc(m & ((1u << lane) - 1u))] = e;
            na += __popc(m);
        }
        if (lane == 0) *nactive = na;
    }
    __syncthreads();

    for (int base = 0; base < n; base += blockDim.x) {
        const int p = base + tid;
        int e = (p < n) ? idx[p] : -1;
        bool ok = (e >= 0 && e < E);
        int key = ok ? e : -1;
        unsigned peers = __match_any_sync(0xffffffffu, key);
        int rank = __popc(peers & ((1u << lane) - 1u));
        bool leader = ok && (rank == 0);
        for (int i = tid; i < 32 * E; i += blockDim.x) table[i / E][i % E] = 0;
        __syncthreads();
        if (leader) table[warp][e] = __popc(peers);
        __syncthreads();
        // per-expert exclusive prefix across warps; cnt[] now holds chunk totals
        for (int ee = tid; ee < E; ee += blockDim.x) {
            int run = 0;
            for (int w = 0; w < 32; ++w) {
                int c = table[w][ee];
                table[w][ee] = run;
                run += c;
            }
            cnt[ee] = run;
        }
        __syncthreads();
        if (ok) {
            const int pos = cursor[e] + table[warp][e] + rank;
            if (pos >= 0 && pos < n) {
                perm[pos] = p;
            } else {
                record_status(hdr, MOE_ERR_INTERNAL, 400000000 + (pos & 0xffffff));
            }
        }
        __syncthreads();
        for (int ee = tid; ee < E; ee += blockDim.x) cursor[ee] += cnt[ee];
        __syncthreads();
    }
}

cudaError_t launch_permute(const int32_t *idx, int T, int k, int E, int32_t *counts, int32_t *offs,
                           int32_t *perm, int32_t *active, int32_t *nactive, WsHeader *hdr,
                           cudaStream_t s) {
    permute_kernel<<<1, 1024, 0, s>>>(idx, T * k, E, counts, offs, perm, active, nactive, hdr);
    return cudaGetLastError();
}

}  // namespace moeq4k
