// Allocation-free variant of the single-token layer call.
//
// Some callers cannot allocate device memory at all: a plugin whose host
// framework owns every device allocation, or a decode loop that must not
// touch an allocator (cudaMalloc, or a caching allocator behind it) on its
// hot path.  They still own x, the weights and the outputs, but cannot
// provide the scratch workspace the other entry points take.  This entry
// point runs the same single-token kernel with its scratch (status word,
// call counters, tagged router logits and expert activations h) in a fixed
// array in device global memory that the library itself defines.
//
// The array lives for as long as the library is loaded, on every GPU that
// loads it; it starts zeroed.  All calls share it and it keeps the previous
// call's contents, which is what the kernel needs: the call counters only
// grow, so the tags left by earlier calls never match a later call's.  The
// call clears the status word itself.  Calls that overlap on the GPU
// (different streams, or several host threads) race on the array and must
// be serialised by the caller.
#include <cstddef>
#include <mutex>

#include "common.cuh"
#include "kernels.cuh"

namespace moeq4k {
namespace {

// Header (256 B), then the tagged router logits (kSyncWords words), then h
// (k*I floats).
constexpr size_t kNoallocScratchBytes = 256 * 1024;
constexpr size_t kNoallocSyncOff = 256;
constexpr size_t kNoallocHOff = kNoallocSyncOff + sizeof(unsigned long long) * kSyncWords;
constexpr size_t kNoallocMaxKI = (kNoallocScratchBytes - kNoallocHOff) / sizeof(float);

__device__ __align__(256) uint8_t g_noalloc_scratch[kNoallocScratchBytes];

// Device address of the array, looked up once per device.  In host code
// the array's name is only a host-side stand-in, never a device pointer.
void *g_noalloc_ptr[64];
std::mutex g_noalloc_mu;

moe_status noalloc_scratch(int dev, uint8_t **out) {
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (g_noalloc_ptr[dev] == nullptr) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
            return MOE_ERR_CUDA;
        g_noalloc_ptr[dev] = ptr;
    }
    *out = static_cast<uint8_t *>(g_noalloc_ptr[dev]);
    return MOE_OK;
}

}  // namespace
}  // namespace moeq4k

using namespace moeq4k;

extern "C" moe_status moe_layer_noalloc(const float *x, const float *Wr, const float *bias,
                                        const void *gate, const void *up, const void *down,
                                        int T, int H, int E, int k, int I, int32_t *idx, float *w,
                                        float *y, void *stream) {
    moe_status st = validate_shape(T, H, E, k, I);
    if (st != MOE_OK) return st;
    if (T != 1) return MOE_ERR_INVALID_SHAPE;
    if (size_t(k) * I > kNoallocMaxKI) return MOE_ERR_SCRATCH_LIMIT;
    const void *ptrs[] = {x, Wr, gate, up, down, idx, w, y};
    for (const void *q : ptrs) {
        if (q == nullptr) return MOE_ERR_NULL;
        if (reinterpret_cast<uintptr_t>(q) % 16 != 0) return MOE_ERR_MISALIGNED;
    }
    if (bias && reinterpret_cast<uintptr_t>(bias) % 16 != 0) return MOE_ERR_MISALIGNED;
    int sms = 0, dev = 0;
    st = device_info(&sms, &dev);
    if (st != MOE_OK) return st;
    if (!decode_fused_supported(dev, T, H, E, k, I)) return MOE_ERR_INVALID_SHAPE;
    uint8_t *scratch = nullptr;
    st = noalloc_scratch(dev, &scratch);
    if (st != MOE_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the status word starts at zero on every call; the call counters must not
    static_assert(offsetof(WsHeader, status) == 0 && offsetof(WsHeader, detail) == 4,
                  "status and detail lead the header");
    if (cudaMemsetAsync(scratch, 0, 8, s) != cudaSuccess) return MOE_ERR_CUDA;
    cudaError_t err = launch_decode_fused(
        dev, x, nullptr, 0.f, OutEpilogue{}, Wr, bias, nullptr, nullptr, idx, w,
        static_cast<const uint8_t *>(gate),
        static_cast<const uint8_t *>(up), static_cast<const uint8_t *>(down), H, E, k, I, y,
        reinterpret_cast<unsigned long long *>(scratch + kNoallocSyncOff),
        reinterpret_cast<float *>(scratch + kNoallocHOff), reinterpret_cast<WsHeader *>(scratch), 0,
        1000000000ull, nullptr, 0, s);
    return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
