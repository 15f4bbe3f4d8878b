// Launch wrappers of the moeq4k kernels (host side).
#pragma once

#include <cuda.h>

#include "common.cuh"

namespace moeq4k {

// Per-device one-time set-up (kernel attributes, SM count) for the current
// device; returns the SM count and the device ordinal.
moe_status device_info(int *sms, int *dev_out);
// Shape limits shared by every entry point.
moe_status validate_shape(int T, int H, int E, int k, int I);

cudaError_t init_router();
// `hdr` carries the one- and two-token router's running CTA count.
cudaError_t launch_router(const float *x, const float *Wr, const float *bias, int T, int H, int E,
                          int k, int32_t *idx, float *w, float *logits, WsHeader *hdr, int num_sms,
                          unsigned long long wait_ns, cudaStream_t s);

// Three launches (count, scan, scatter); blockcnt holds ceil(T*k / kPermSlots)
// x E ints of scratch, slotpos receives each slot's sorted position.
// Up to kSmallPermSlots routed slots the permutation is one launch of one
// CTA, above that three launches; either way the chunk plans `pa` / `pb` are
// written on the way when their cap is non-zero.
cudaError_t launch_permute(const int32_t *idx, int T, int k, int E, int32_t *counts, int32_t *offs,
                           int32_t *perm, int32_t *active, int32_t *nactive, int32_t *blockcnt,
                           int32_t *slotpos, WsHeader *hdr, cudaStream_t s,
                           const ChunkPlan &pa = ChunkPlan{}, const ChunkPlan &pb = ChunkPlan{});

cudaError_t init_expert_ffn();
cudaError_t launch_expert_ffn(const float *x, const int32_t *idx, const float *w,
                              const uint8_t *gate, const uint8_t *up, const uint8_t *down, int T,
                              int H, int E, int k, int I, float *y, const int32_t *offs,
                              const int32_t *perm, const int32_t *active, const int32_t *nactive,
                              float *hbuf, float *obuf, WsHeader *hdr, const OutEpilogue &ep,
                              int num_sms, cudaStream_t s);

cudaError_t launch_combine(const float *obuf, const int32_t *idx, const float *w, int T, int H,
                           int E, int k, float *y, const OutEpilogue &ep, int num_sms,
                           cudaStream_t s);

// Pre-FFN RMSNorm of T rows: xn = x / sqrt(mean(x^2) + eps) * gamma.
cudaError_t launch_rmsnorm(const float *x, const float *gamma, float eps, int T, int H, float *xn,
                           cudaStream_t s);

cudaError_t init_prefill_tc(int dev);
bool prefill_tc_supported(int T, int H, int E, int k, int I);
// A 2-D TMA map of a row-major fp32 matrix [rows][cols] (cols a multiple of
// 4, base 16-byte aligned): boxes of 32 columns (one 128-byte row) x
// box_rows rows with the 128-byte swizzle; out-of-range elements read as
// zero.  Needs init_prefill_tc first.  False on failure.
bool encode_fp32_sw128_map(CUtensorMap *map, const float *base, int rows, int cols, int box_rows);
bool encode_fp32_box_map(CUtensorMap *map, const float *base, int rows, int cols, int box_cols,
                         int box_rows);

// Router logits of T >= 256 tokens (E <= 128, H a multiple of 128) on the
// tensor cores (three-pass TF32), with the top-k fused.
bool router_tc_supported(int T, int H, int E);
cudaError_t init_router_tc();
cudaError_t launch_router_tc(const float *x, const float *Wr, const float *bias, int T, int H, int E,
                             int k, int32_t *idx, float *w, WsHeader *hdr,
                             unsigned long long wait_ns, cudaStream_t s);

// The chunk capacities of the gate/up and down GEMMs for a batch of T tokens.
void prefill_tc_caps(int T, int *cap_gu, int *cap_dn);
// The chunk plans (`chunks`, `chunks_dn`) are written by the permutation.
cudaError_t launch_prefill_tc(int dev, const float *x, const uint8_t *gate, const uint8_t *up,
                              const uint8_t *down, int T, int H, int E, int k, int I,
                              const int32_t *offs, const int32_t *perm, const int32_t *slotpos,
                              const int32_t *active,
                              const int32_t *nactive, __half *x16, __half *h16, float *obuf,
                              TcChunk *chunks, TcChunk *chunks_dn, unsigned int *ready, WsHeader *hdr,
                              int num_sms, unsigned long long wait_ns, int withhold,
                              unsigned long long *timeline,
                              cudaStream_t s);

cudaError_t init_decode_fused(int dev, int num_sms);
bool decode_fused_supported(int dev, int T, int H, int E, int k, int I);
// Wr == nullptr: routing comes from idx_in / w_in (moe_ffn); otherwise the
// kernel routes and writes idx_out / w_out (moe_layer).  `sync` is the tag
// region (kSyncWords words, zero or tags of earlier calls of this header),
// `hbuf` k*I floats of scratch; `timeline` (timeline_cap words) is written
// only by profiling builds.  `norm_w` (nullable): x is RMS-normalised with
// it (and `eps`) before anything uses it; `ep`: the output epilogue.
cudaError_t launch_decode_fused(int dev, const float *x, const float *norm_w, float eps,
                                const OutEpilogue &ep, const float *Wr, const float *bias,
                                const int32_t *idx_in, const float *w_in, int32_t *idx_out,
                                float *w_out, const uint8_t *gate, const uint8_t *up,
                                const uint8_t *down, int H, int E, int k, int I, float *y,
                                unsigned long long *sync, float *hbuf, WsHeader *hdr, int withhold,
                                unsigned long long wait_ns, unsigned long long *timeline,
                                int timeline_cap, cudaStream_t s);

// One token whose rows do not fit the fused kernel: gate/up then down with
// the slot-ordered combine folded in (two launches; idx / w from the router
// or the caller; `hbuf` k*I floats of scratch).
cudaError_t init_decode_stream(int dev);
bool decode_stream_supported(int dev, int T, int H, int E, int k, int I);
cudaError_t launch_decode_stream(const float *x, const int32_t *idx, const float *w,
                                 const uint8_t *gate, const uint8_t *up, const uint8_t *down,
                                 int H, int E, int k, int I, float *y, float *hbuf, WsHeader *hdr,
                                 const OutEpilogue &ep, int num_sms, cudaStream_t s);

// Q8_K activations: `rows` fp32 rows of n values (n a multiple of 256) ->
// codes [rows, n], block scales [rows, n/256], sub-block code sums
// [rows, n/32]; and the expert FFN on them (x and h quantised; `hbuf`
// T*k*I floats of scratch; xq/xd/xs and hq/hd/hs the quantised x and h).
cudaError_t launch_q8k_quantize(const float *v, long rows, int n, int8_t *q, float *d,
                                int32_t *sums, int num_sms, cudaStream_t s);
cudaError_t launch_q8k_ffn(const float *x, const int32_t *idx, const float *w, const uint8_t *gate,
                           const uint8_t *up, const uint8_t *down, int T, int H, int E, int k,
                           int I, float *y, int8_t *xq, float *xd, int32_t *xs, float *hbuf,
                           int8_t *hq, float *hd, int32_t *hs, WsHeader *hdr, int num_sms,
                           cudaStream_t s);

}  // namespace moeq4k
