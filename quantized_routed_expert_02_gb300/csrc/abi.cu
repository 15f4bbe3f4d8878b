// C ABI of the moeq4k library: argument checks, workspace carving and launch
// order.  Every entry point checks its arguments before anything is enqueued
// and returns a moe_status; nothing here allocates device memory.
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "kernels.cuh"

using namespace moeq4k;

namespace {

struct DevInfo {
    bool ready = false;
    int sms = 0;
    int id = 0;
};
constexpr int kMaxDevices = 64;
DevInfo g_dev[kMaxDevices];
std::mutex g_mu;

// Test hooks (see moe_debug_set_wait_limit / moe_debug_withhold_arrivals).
unsigned long long g_wait_ns = 1000000000ull;  // 1 s: far above any healthy wait
int g_withhold = 0;

}  // namespace

// Per-device one-time set-up (kernel attributes, SM count) for the current device.
moe_status moeq4k::device_info(int *sms, int *dev_out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_dev[dev].ready) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return MOE_ERR_CUDA;
        if (init_expert_ffn() != cudaSuccess) return MOE_ERR_CUDA;
        if (init_router() != cudaSuccess) return MOE_ERR_CUDA;
        if (init_decode_fused(dev, n) != cudaSuccess) return MOE_ERR_CUDA;
        if (init_prefill_tc(dev) != cudaSuccess) return MOE_ERR_CUDA;
        if (init_router_tc() != cudaSuccess) return MOE_ERR_CUDA;
        if (init_decode_stream(dev) != cudaSuccess) return MOE_ERR_CUDA;
        g_dev[dev].sms = n;
        g_dev[dev].id = dev;
        g_dev[dev].ready = true;
    }
    *sms = g_dev[dev].sms;
    if (dev_out) *dev_out = dev;
    return MOE_OK;
}

namespace {

inline bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

moe_status check_shape(int T, int H, int E, int k, int I) {
    if (T < 1 || H < 1 || E < 1 || k < 1 || I < 1) return MOE_ERR_INVALID_SHAPE;
    if (k > E || E > kMaxE || k > kMaxK) return MOE_ERR_INVALID_SHAPE;
    if (H % kQK != 0 || I % kQK != 0 || H > kMaxHI || I > kMaxHI) return MOE_ERR_INVALID_SHAPE;
    if (int64_t(T) * k > (int64_t(1) << 22)) return MOE_ERR_INVALID_SHAPE;
    return MOE_OK;
}

moe_status check_ptr(const void *p, size_t align) {
    if (p == nullptr) return MOE_ERR_NULL;
    if (!aligned(p, align)) return MOE_ERR_MISALIGNED;
    return MOE_OK;
}

#define MOE_TRY(expr)                        \
    do {                                     \
        moe_status _s = (expr);              \
        if (_s != MOE_OK) return _s;         \
    } while (0)

struct Ws {
    uint8_t *base;
    WsLayout L;
    WsHeader *hdr() const { return reinterpret_cast<WsHeader *>(base); }
    int32_t *i32(size_t off) const { return reinterpret_cast<int32_t *>(base + off); }
    float *f32(size_t off) const { return reinterpret_cast<float *>(base + off); }
    unsigned long long *u64(size_t off) const {
        return reinterpret_cast<unsigned long long *>(base + off);
    }
    // the single-token kernel's profiling timeline: the per-slot output
    // region, which that kernel does not use
    int timeline_cap() const { return int((L.x16 - L.o) / sizeof(unsigned long long)); }
};

// Profiling builds: the grouped GEMMs' per-stage stamps go to the fp32
// expert-activation region, which the tensor-core path does not use.
unsigned long long *gemm_timeline(const Ws &ws) {
#ifdef MOEQ4K_TIMELINE
    if (ws.L.o - ws.L.h >= 2 * 12 * 256 * sizeof(unsigned long long)) return ws.u64(ws.L.h);
#else
    (void)ws;
#endif
    return nullptr;
}

moe_status check_ws(void *ws, size_t ws_bytes, const WsLayout &L) {
    MOE_TRY(check_ptr(ws, 256));
    if (ws_bytes < L.total) return MOE_ERR_WORKSPACE;
    return MOE_OK;
}

inline moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

moe_status ffn_enqueue(const float *x, const int32_t *idx, const float *w, const void *gate,
                       const void *up, const void *down, int T, int H, int E, int k, int I,
                       float *y, const Ws &ws, int sms, int dev, const OutEpilogue &ep,
                       cudaStream_t s) {
    const WsLayout &L = ws.L;
    const bool tensor = prefill_tc_supported(T, H, E, k, I);
    // the tensor-core path's chunk plans, written by the permutation
    ChunkPlan pa, pb;
    if (tensor) {
        int cap_gu = 0, cap_dn = 0;
        prefill_tc_caps(T, &cap_gu, &cap_dn);
        pa.cap = cap_gu;
        pa.chunks = reinterpret_cast<TcChunk *>(ws.base + L.chunks);
        pa.count = &ws.hdr()->tc_chunks;
        if (cap_dn != cap_gu) {
            pb.cap = cap_dn;
            pb.chunks = reinterpret_cast<TcChunk *>(ws.base + L.chunks_dn);
            pb.count = &ws.hdr()->tc_chunks_dn;
        }
    }
    MOE_TRY(cuda_status(launch_permute(idx, T, k, E, ws.i32(L.counts), ws.i32(L.offs),
                                       ws.i32(L.perm), ws.i32(L.active), ws.i32(L.nactive),
                                       ws.i32(L.blockcnt), ws.i32(L.slotpos), ws.hdr(), s, pa, pb)));
    if (tensor) {
        MOE_TRY(cuda_status(launch_prefill_tc(
            dev, x, static_cast<const uint8_t *>(gate), static_cast<const uint8_t *>(up),
            static_cast<const uint8_t *>(down), T, H, E, k, I, ws.i32(L.offs), ws.i32(L.perm),
            ws.i32(L.slotpos), ws.i32(L.active), ws.i32(L.nactive), reinterpret_cast<__half *>(ws.base + L.x16),
            reinterpret_cast<__half *>(ws.base + L.h16), ws.f32(L.o),
            reinterpret_cast<TcChunk *>(ws.base + L.chunks),
            reinterpret_cast<TcChunk *>(ws.base + L.chunks_dn),
            reinterpret_cast<unsigned int *>(ws.base + L.ready), ws.hdr(), sms, g_wait_ns, g_withhold,
            gemm_timeline(ws), s)));
        return cuda_status(launch_combine(ws.f32(L.o), idx, w, T, H, E, k, y, ep, sms, s));
    }
    return cuda_status(launch_expert_ffn(
        x, idx, w, static_cast<const uint8_t *>(gate), static_cast<const uint8_t *>(up),
        static_cast<const uint8_t *>(down), T, H, E, k, I, y, ws.i32(L.offs), ws.i32(L.perm),
        ws.i32(L.active), ws.i32(L.nactive), ws.f32(L.h), ws.f32(L.o), ws.hdr(), ep, sms, s));
}

// Router then FFN for every shape (moe_layer and moe_layer_block): x is the
// FFN input; norm_w (nullable) asks the single-token fused kernel to
// RMS-normalise x itself (the other paths get an already normalised x).
moe_status layer_enqueue(const float *x, const float *norm_w, float eps, const float *Wr,
                         const float *bias, const void *gate, const void *up, const void *down,
                         int T, int H, int E, int k, int I, int32_t *idx, float *w, float *y,
                         const Ws &W, int sms, int dev, const OutEpilogue &ep, cudaStream_t s) {
    const WsLayout &L = W.L;
    if (decode_fused_supported(dev, T, H, E, k, I)) {
        return cuda_status(launch_decode_fused(
            dev, x, norm_w, eps, ep, Wr, bias, nullptr, nullptr, idx, w,
            static_cast<const uint8_t *>(gate), static_cast<const uint8_t *>(up),
            static_cast<const uint8_t *>(down), H, E, k, I, y, W.u64(L.sync), W.f32(L.h), W.hdr(),
            g_withhold, g_wait_ns, W.u64(L.o), W.timeline_cap(), s));
    }
    MOE_TRY(cuda_status(launch_router(x, Wr, bias, T, H, E, k, idx, w, W.f32(L.logits), W.hdr(), sms, g_wait_ns, s)));
    if (decode_stream_supported(dev, T, H, E, k, I)) {
        return cuda_status(launch_decode_stream(
            x, idx, w, static_cast<const uint8_t *>(gate), static_cast<const uint8_t *>(up),
            static_cast<const uint8_t *>(down), H, E, k, I, y, W.f32(L.h), W.hdr(), ep, sms, s));
    }
    return ffn_enqueue(x, idx, w, gate, up, down, T, H, E, k, I, y, W, sms, dev, ep, s);
}

// The Q8_K-activation FFN's scratch inside the fp16 activation regions,
// which that path does not otherwise use: codes, then block scales, then
// sub-block code sums (1.14 n bytes for n values; the regions hold 2 n).
struct Q8Scratch {
    int8_t *xq, *hq;
    float *xd, *hd;
    int32_t *xs, *hs;
};

Q8Scratch q8_scratch(const Ws &W, int T, int H, int k, int I) {
    const size_t nx = size_t(T) * H, nh = size_t(T) * k * I;
    Q8Scratch q;
    q.xq = reinterpret_cast<int8_t *>(W.base + W.L.x16);
    q.xd = reinterpret_cast<float *>(W.base + W.L.x16 + nx);
    q.xs = reinterpret_cast<int32_t *>(W.base + W.L.x16 + nx + nx / 64);
    q.hq = reinterpret_cast<int8_t *>(W.base + W.L.h16);
    q.hd = reinterpret_cast<float *>(W.base + W.L.h16 + nh);
    q.hs = reinterpret_cast<int32_t *>(W.base + W.L.h16 + nh + nh / 64);
    return q;
}

moe_status q8k_ffn_enqueue(const float *x, const int32_t *idx, const float *w, const void *gate,
                           const void *up, const void *down, int T, int H, int E, int k, int I,
                           float *y, const Ws &W, int sms, cudaStream_t s) {
    const Q8Scratch q = q8_scratch(W, T, H, k, I);
    return cuda_status(launch_q8k_ffn(x, idx, w, static_cast<const uint8_t *>(gate),
                                      static_cast<const uint8_t *>(up),
                                      static_cast<const uint8_t *>(down), T, H, E, k, I, y, q.xq,
                                      q.xd, q.xs, W.f32(W.L.h), q.hq, q.hd, q.hs, W.hdr(), sms, s));
}

}  // namespace

moe_status moeq4k::validate_shape(int T, int H, int E, int k, int I) {
    return check_shape(T, H, E, k, I);
}

extern "C" {

const char *moe_status_str(moe_status s) {
    switch (s) {
        case MOE_OK: return "MOE_OK";
        case MOE_ERR_INVALID_SHAPE: return "MOE_ERR_INVALID_SHAPE";
        case MOE_ERR_NULL: return "MOE_ERR_NULL";
        case MOE_ERR_MISALIGNED: return "MOE_ERR_MISALIGNED";
        case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
        case MOE_ERR_EXPERT_RANGE: return "MOE_ERR_EXPERT_RANGE";
        case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
        case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
        case MOE_ERR_INTERNAL: return "MOE_ERR_INTERNAL";
        case MOE_ERR_SCRATCH_LIMIT: return "MOE_ERR_SCRATCH_LIMIT";
    }
    return "MOE_ERR_UNKNOWN";
}

int moe_version(void) { return 100; }

size_t moe_workspace_bytes(int T, int H, int E, int k, int I) {
    if (check_shape(T, H, E, k, I) != MOE_OK) return 0;
    return ws_layout(T, H, E, k, I, false).total;
}

size_t moe_workspace_bytes_host(int T, int H, int E, int k, int I) {
    if (check_shape(T, H, E, k, I) != MOE_OK) return 0;
    return ws_layout(T, H, E, k, I, true).total;
}

int moe_layer_launch_count(int T, int H, int E, int k, int I) {
    if (check_shape(T, H, E, k, I) != MOE_OK) return 0;
    int sms = 0, dev = 0;
    if (device_info(&sms, &dev) != MOE_OK) return 0;
    if (decode_fused_supported(dev, T, H, E, k, I)) return 1;
    if (decode_stream_supported(dev, T, H, E, k, I)) return 1 /* router */ + 2;
    const int router = 1;
    // one launch up to kSmallPermSlots routed slots, else count, scan,
    // scatter (the permutation also writes the GEMMs' chunk plans)
    const int permutation = int64_t(T) * k <= kSmallPermSlots ? 1 : 3;
    if (prefill_tc_supported(T, H, E, k, I)) {
        // fp16 rows, GEMMs, combine
        return router + permutation + 1 + 2 + 1;
    }
    return router + permutation + 3 /* gate/up, down, combine */;
}

int moe_layer_q8k_launch_count(int T, int H, int E, int k, int I) {
    if (check_shape(T, H, E, k, I) != MOE_OK) return 0;
    return 1 /* router */ + 4;  // quantise x, gate/up, quantise h, down (with the combine)
}

void moe_debug_set_wait_limit(unsigned long long ns) { g_wait_ns = ns ? ns : 1000000000ull; }

void moe_debug_withhold_arrivals(int n) { g_withhold = n < 0 ? 0 : n; }

moe_status moe_workspace_init(void *ws, size_t ws_bytes, void *stream) {
    MOE_TRY(check_ptr(ws, 256));
    if (ws_bytes < sizeof(WsHeader)) return MOE_ERR_WORKSPACE;
    // the header and the tag region (the same place for every shape)
    const size_t keep = sizeof(WsHeader) + align256(sizeof(unsigned long long) * kSyncWords);
    return cuda_status(cudaMemsetAsync(ws, 0, std::min(ws_bytes, keep),
                                       static_cast<cudaStream_t>(stream)));
}

moe_status moe_router(const float *x, const float *Wr, const float *bias, int T, int H, int E,
                      int k, int32_t *idx, float *w, void *ws, size_t ws_bytes, void *stream) {
    MOE_TRY(check_shape(T, H, E, k, 256));
    MOE_TRY(check_ptr(x, 16));
    MOE_TRY(check_ptr(Wr, 16));
    if (bias && !aligned(bias, 16)) return MOE_ERR_MISALIGNED;
    MOE_TRY(check_ptr(idx, 16));
    MOE_TRY(check_ptr(w, 16));
    WsLayout L = ws_layout(T, H, E, k, 256, false);
    // the router only needs the header and the logits region
    MOE_TRY(check_ptr(ws, 256));
    if (ws_bytes < L.logits + sizeof(float) * size_t(T) * E) return MOE_ERR_WORKSPACE;
    int sms = 0;
    MOE_TRY(device_info(&sms, nullptr));
    Ws W{static_cast<uint8_t *>(ws), L};
    return cuda_status(launch_router(x, Wr, bias, T, H, E, k, idx, w, W.f32(L.logits), W.hdr(),
                                     sms, g_wait_ns, static_cast<cudaStream_t>(stream)));
}

moe_status moe_permute(const int32_t *idx, int T, int k, int E, int32_t *counts, int32_t *offs,
                       int32_t *perm, void *ws, size_t ws_bytes, void *stream) {
    MOE_TRY(check_shape(T, 256, E, k, 256));
    MOE_TRY(check_ptr(idx, 16));
    MOE_TRY(check_ptr(counts, 16));
    MOE_TRY(check_ptr(offs, 16));
    MOE_TRY(check_ptr(perm, 16));
    MOE_TRY(check_ptr(ws, 256));
    WsLayout L = ws_layout(T, 256, E, k, 256, false);
    if (ws_bytes < L.perm) return MOE_ERR_WORKSPACE;
    int sms = 0;
    MOE_TRY(device_info(&sms, nullptr));
    Ws W{static_cast<uint8_t *>(ws), L};
    return cuda_status(launch_permute(idx, T, k, E, counts, offs, perm, W.i32(L.active),
                                      W.i32(L.nactive), W.i32(L.blockcnt), W.i32(L.slotpos),
                                      W.hdr(), static_cast<cudaStream_t>(stream)));
}

moe_status moe_ffn(const float *x, const int32_t *idx, const float *w, const void *gate,
                   const void *up, const void *down, int T, int H, int E, int k, int I, float *y,
                   void *ws, size_t ws_bytes, void *stream) {
    MOE_TRY(check_shape(T, H, E, k, I));
    MOE_TRY(check_ptr(x, 16));
    MOE_TRY(check_ptr(idx, 16));
    MOE_TRY(check_ptr(w, 16));
    MOE_TRY(check_ptr(gate, 16));
    MOE_TRY(check_ptr(up, 16));
    MOE_TRY(check_ptr(down, 16));
    MOE_TRY(check_ptr(y, 16));
    WsLayout L = ws_layout(T, H, E, k, I, false);
    MOE_TRY(check_ws(ws, ws_bytes, L));
    int sms = 0, dev = 0;
    MOE_TRY(device_info(&sms, &dev));
    Ws W{static_cast<uint8_t *>(ws), L};
    const OutEpilogue none;
    if (decode_fused_supported(dev, T, H, E, k, I)) {
        return cuda_status(launch_decode_fused(
            dev, x, nullptr, 0.f, none, nullptr, nullptr, idx, w, nullptr, nullptr,
            static_cast<const uint8_t *>(gate), static_cast<const uint8_t *>(up),
            static_cast<const uint8_t *>(down), H, E, k, I, y, W.u64(L.sync), W.f32(L.h), W.hdr(),
            g_withhold, g_wait_ns, W.u64(L.o), W.timeline_cap(), static_cast<cudaStream_t>(stream)));
    }
    if (decode_stream_supported(dev, T, H, E, k, I)) {
        return cuda_status(launch_decode_stream(
            x, idx, w, static_cast<const uint8_t *>(gate), static_cast<const uint8_t *>(up),
            static_cast<const uint8_t *>(down), H, E, k, I, y, W.f32(L.h), W.hdr(), none, sms,
            static_cast<cudaStream_t>(stream)));
    }
    return ffn_enqueue(x, idx, w, gate, up, down, T, H, E, k, I, y, W, sms, dev, none,
                       static_cast<cudaStream_t>(stream));
}

moe_status moe_layer(const float *x, const float *Wr, const float *bias, const void *gate,
                     const void *up, const void *down, int T, int H, int E, int k, int I,
                     int32_t *idx, float *w, float *y, void *ws, size_t ws_bytes, void *stream) {
    MOE_TRY(check_shape(T, H, E, k, I));
    MOE_TRY(check_ptr(x, 16));
    MOE_TRY(check_ptr(Wr, 16));
    if (bias && !aligned(bias, 16)) return MOE_ERR_MISALIGNED;
    MOE_TRY(check_ptr(gate, 16));
    MOE_TRY(check_ptr(up, 16));
    MOE_TRY(check_ptr(down, 16));
    MOE_TRY(check_ptr(idx, 16));
    MOE_TRY(check_ptr(w, 16));
    MOE_TRY(check_ptr(y, 16));
    WsLayout L = ws_layout(T, H, E, k, I, false);
    MOE_TRY(check_ws(ws, ws_bytes, L));
    int sms = 0, dev = 0;
    MOE_TRY(device_info(&sms, &dev));
    Ws W{static_cast<uint8_t *>(ws), L};
    return layer_enqueue(x, nullptr, 0.f, Wr, bias, gate, up, down, T, H, E, k, I, idx, w, y, W,
                         sms, dev, OutEpilogue{}, static_cast<cudaStream_t>(stream));
}

moe_status moe_layer_block(const float *hidden, const float *norm_w, float norm_eps,
                           const float *Wr, const float *bias, const void *gate, const void *up,
                           const void *down, int T, int H, int E, int k, int I, int32_t *idx,
                           float *w, float *out, int add_residual, int capture_token,
                           int32_t *cap_idx, float *cap_w, float *cap_ffn, void *ws,
                           size_t ws_bytes, void *stream) {
    MOE_TRY(check_shape(T, H, E, k, I));
    MOE_TRY(check_ptr(hidden, 16));
    if (norm_w && !aligned(norm_w, 16)) return MOE_ERR_MISALIGNED;
    if (!(norm_eps >= 0.f) || !(norm_eps <= 3.402823466e38f)) return MOE_ERR_INVALID_SHAPE;
    MOE_TRY(check_ptr(Wr, 16));
    if (bias && !aligned(bias, 16)) return MOE_ERR_MISALIGNED;
    MOE_TRY(check_ptr(gate, 16));
    MOE_TRY(check_ptr(up, 16));
    MOE_TRY(check_ptr(down, 16));
    MOE_TRY(check_ptr(idx, 16));
    MOE_TRY(check_ptr(w, 16));
    MOE_TRY(check_ptr(out, 16));
    if (capture_token < -1 || capture_token >= T) return MOE_ERR_INVALID_SHAPE;
    if ((cap_idx && !aligned(cap_idx, 4)) || (cap_w && !aligned(cap_w, 4)) ||
        (cap_ffn && !aligned(cap_ffn, 16)))
        return MOE_ERR_MISALIGNED;
    WsLayout L = ws_layout(T, H, E, k, I, false);
    MOE_TRY(check_ws(ws, ws_bytes, L));
    int sms = 0, dev = 0;
    MOE_TRY(device_info(&sms, &dev));
    Ws W{static_cast<uint8_t *>(ws), L};
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    OutEpilogue ep;
    ep.residual = add_residual ? hidden : nullptr;
    ep.capture = capture_token >= 0 ? cap_ffn : nullptr;
    ep.cap_t = capture_token;
    // The fused single-token kernel normalises x while staging it; every
    // other path reads a normalised copy from the workspace.
    const float *ffn_in = hidden;
    const float *fused_norm = nullptr;
    if (norm_w != nullptr) {
        if (decode_fused_supported(dev, T, H, E, k, I)) {
            fused_norm = norm_w;
        } else {
            MOE_TRY(cuda_status(launch_rmsnorm(hidden, norm_w, norm_eps, T, H, W.f32(L.xn), s)));
            ffn_in = W.f32(L.xn);
        }
    }
    MOE_TRY(layer_enqueue(ffn_in, fused_norm, norm_eps, Wr, bias, gate, up, down, T, H, E, k, I,
                          idx, w, out, W, sms, dev, ep, s));
    // the router stage of the captured token: its k expert ids and weights
    if (capture_token >= 0 && cap_idx != nullptr)
        MOE_TRY(cuda_status(cudaMemcpyAsync(cap_idx, idx + size_t(capture_token) * k,
                                            sizeof(int32_t) * k, cudaMemcpyDeviceToDevice, s)));
    if (capture_token >= 0 && cap_w != nullptr)
        MOE_TRY(cuda_status(cudaMemcpyAsync(cap_w, w + size_t(capture_token) * k,
                                            sizeof(float) * k, cudaMemcpyDeviceToDevice, s)));
    return MOE_OK;
}

// Host memory that kernels may address with the same pointer: page-locked
// (cudaHostAlloc / cudaHostRegister) and mapped into the unified address
// space.  Pageable memory, device memory and unknown pointers are not.
static bool host_mapped(const void *p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        (void)cudaGetLastError();  // an unknown pointer is not an error here
        return false;
    }
    return a.type == cudaMemoryTypeHost && a.devicePointer == p;
}

moe_status moe_layer_host(const float *x_host, const float *Wr, const float *bias,
                          const void *gate, const void *up, const void *down, int T, int H, int E,
                          int k, int I, int32_t *idx, float *w, float *y_host, void *ws,
                          size_t ws_bytes, void *stream) {
    MOE_TRY(check_shape(T, H, E, k, I));
    if (x_host == nullptr || y_host == nullptr) return MOE_ERR_NULL;
    WsLayout L = ws_layout(T, H, E, k, I, true);
    MOE_TRY(check_ws(ws, ws_bytes, L));
    Ws W{static_cast<uint8_t *>(ws), L};
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // A single token on the fused kernel reads x once per CTA and writes y
    // once: with both buffers mapped host memory it reads and writes them in
    // place over the chip-to-chip link, with no staging copies (measured on
    // GB300 at the A3B single token: 39.5 -> 36.3 us per call, outputs
    // bitwise the same).
    int sms = 0, dev = 0;
    MOE_TRY(device_info(&sms, &dev));
    if (decode_fused_supported(dev, T, H, E, k, I) && aligned(x_host, 16) && aligned(y_host, 16) &&
        host_mapped(x_host) && host_mapped(y_host)) {
        MOE_TRY(moe_layer(x_host, Wr, bias, gate, up, down, T, H, E, k, I, idx, w, y_host, ws,
                          ws_bytes, stream));
        return cuda_status(cudaStreamSynchronize(s));
    }
    const size_t bytes = sizeof(float) * size_t(T) * H;
    float *xd = W.f32(L.xstage), *yd = W.f32(L.ystage);
    MOE_TRY(cuda_status(cudaMemcpyAsync(xd, x_host, bytes, cudaMemcpyHostToDevice, s)));
    MOE_TRY(moe_layer(xd, Wr, bias, gate, up, down, T, H, E, k, I, idx, w, yd, ws, ws_bytes,
                      stream));
    MOE_TRY(cuda_status(cudaMemcpyAsync(y_host, yd, bytes, cudaMemcpyDeviceToHost, s)));
    return cuda_status(cudaStreamSynchronize(s));
}

moe_status moe_quantize_q8k(const float *v, int rows, int n, int8_t *q, float *d, int32_t *sums,
                            void *stream) {
    if (rows < 1 || n < kQK || n % kQK != 0 || int64_t(rows) * n > (int64_t(1) << 31))
        return MOE_ERR_INVALID_SHAPE;
    MOE_TRY(check_ptr(v, 16));
    MOE_TRY(check_ptr(q, 16));
    MOE_TRY(check_ptr(d, 4));
    MOE_TRY(check_ptr(sums, 4));
    int sms = 0;
    MOE_TRY(device_info(&sms, nullptr));
    return cuda_status(launch_q8k_quantize(v, rows, n, q, d, sums, sms,
                                           static_cast<cudaStream_t>(stream)));
}

moe_status moe_ffn_q8k(const float *x, const int32_t *idx, const float *w, const void *gate,
                       const void *up, const void *down, int T, int H, int E, int k, int I,
                       float *y, void *ws, size_t ws_bytes, void *stream) {
    MOE_TRY(check_shape(T, H, E, k, I));
    MOE_TRY(check_ptr(x, 16));
    MOE_TRY(check_ptr(idx, 16));
    MOE_TRY(check_ptr(w, 16));
    MOE_TRY(check_ptr(gate, 16));
    MOE_TRY(check_ptr(up, 16));
    MOE_TRY(check_ptr(down, 16));
    MOE_TRY(check_ptr(y, 16));
    WsLayout L = ws_layout(T, H, E, k, I, false);
    MOE_TRY(check_ws(ws, ws_bytes, L));
    int sms = 0;
    MOE_TRY(device_info(&sms, nullptr));
    Ws W{static_cast<uint8_t *>(ws), L};
    return q8k_ffn_enqueue(x, idx, w, gate, up, down, T, H, E, k, I, y, W, sms,
                           static_cast<cudaStream_t>(stream));
}

moe_status moe_layer_q8k(const float *x, const float *Wr, const float *bias, const void *gate,
                         const void *up, const void *down, int T, int H, int E, int k, int I,
                         int32_t *idx, float *w, float *y, void *ws, size_t ws_bytes,
                         void *stream) {
    MOE_TRY(check_shape(T, H, E, k, I));
    MOE_TRY(check_ptr(x, 16));
    MOE_TRY(check_ptr(Wr, 16));
    if (bias && !aligned(bias, 16)) return MOE_ERR_MISALIGNED;
    MOE_TRY(check_ptr(gate, 16));
    MOE_TRY(check_ptr(up, 16));
    MOE_TRY(check_ptr(down, 16));
    MOE_TRY(check_ptr(idx, 16));
    MOE_TRY(check_ptr(w, 16));
    MOE_TRY(check_ptr(y, 16));
    WsLayout L = ws_layout(T, H, E, k, I, false);
    MOE_TRY(check_ws(ws, ws_bytes, L));
    int sms = 0;
    MOE_TRY(device_info(&sms, nullptr));
    Ws W{static_cast<uint8_t *>(ws), L};
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    MOE_TRY(cuda_status(launch_router(x, Wr, bias, T, H, E, k, idx, w, W.f32(L.logits), W.hdr(), sms, g_wait_ns, s)));
    return q8k_ffn_enqueue(x, idx, w, gate, up, down, T, H, E, k, I, y, W, sms, s);
}

moe_status moe_read_device_status(const void *ws, void *stream, int32_t *detail) {
    MOE_TRY(check_ptr(ws, 256));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    WsHeader h;
    MOE_TRY(cuda_status(cudaMemcpyAsync(&h, ws, sizeof(h), cudaMemcpyDeviceToHost, s)));
    MOE_TRY(cuda_status(cudaStreamSynchronize(s)));
    if (detail) *detail = h.detail;
    return static_cast<moe_status>(h.status);
}

}  // extern "C"
