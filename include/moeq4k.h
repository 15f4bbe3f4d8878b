/*
 * moeq4k — routed-expert MoE FFN over GGUF Q4_K expert weights, for one GB300
 * (sm_103a).  C ABI.
 *
 * The operation is one Qwen3-MoE routed-expert FFN layer
 * (forward_qwen3_moe.rs, aprender-serve 0.35.0, step 2h of
 * forward_single_qwen3_moe_with_cache and step 2g of forward_qwen3_moe):
 *
 *   router:   l[t,e] = sum_h x[t,h] Wr[e,h] (+ bias[e])
 *             p[t,:] = softmax over all E experts of l[t,:]
 *             idx[t,0..k) = the k largest p, descending, ties -> lowest index
 *             w[t,j] = p[t,idx[t,j]] / sum_j' p[t,idx[t,j']]
 *             (forward_qwen3_moe_cuda_traced.rs, aprender-serve 0.34.0, doc of
 *             forward_qwen3_moe_cuda_traced_with_plan: the router stage is the
 *             k post-softmax, renormalised top-k weights)
 *   expert e: g = Wg[e] x, u = Wu[e] x, h = SiLU(g) * u, o = Wd[e] h,
 *             SiLU(z) = z / (1 + exp(-z))
 *   output:   y[t] = sum over slots j = 0..k-1, in slot order, of w[t,j] o_{t,j}
 *             (the output stage is [H] per token)
 *
 * Each expert matrix is consumed in place in the Q4_K block format (fused
 * dequant + matvec; forward_qwen3_moe.rs, doc of forward_qwen3_moe, argument
 * `data`).  Activations are fp32 and are not quantised
 * (qwen3_moe_dispatch.rs, aprender-serve 0.70.2, doc of cpu_reference).
 *
 * Q4_K block: 144 bytes per 256 weights — fp16 d, fp16 dmin, 12 bytes of
 * packed 6-bit scales sc[8] and mins m[8], 128 bytes of 4-bit codes q;
 * weight = d * sc[j] * q - dmin * m[j] for sub-block j (32 weights).
 *
 * Conventions for every entry point:
 *  - Pointers named *_dev are device pointers, owned by the caller, never
 *    freed or retained by the library.  Expert blobs are borrowed in place.
 *  - Every device pointer must be 16-byte aligned; the workspace 256-byte
 *    aligned.
 *  - Row-major layouts: x [T,H] fp32, Wr [E,H] fp32, bias [E] fp32,
 *    idx [T,k] int32, w [T,k] fp32, y [T,H] fp32.
 *    gate/up blobs: [E][I rows][H/256 blocks] x 144 B; down blob:
 *    [E][H rows][I/256 blocks] x 144 B (blocks contiguous along the
 *    reduction dimension, rows contiguous, experts contiguous).
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default).
 *    Calls only enqueue work on it: they never allocate, free or
 *    synchronise, except moe_read_device_status (which synchronises the
 *    stream) and moe_layer_host (which synchronises before returning).
 *  - Argument errors are returned before anything is enqueued.  Problems
 *    only the device can see (an expert index outside [0,E) in a
 *    caller-given idx) are recorded in a sticky status word inside the
 *    workspace; the offending slot contributes nothing to y.  Read the word
 *    with moe_read_device_status, reset it with moe_workspace_init.
 *  - Limits: 1 <= T, 1 <= k <= E <= 256, k <= 32, H and I multiples of 256,
 *    H <= 8192, I <= 8192, T*k <= 2^22.  Shapes outside them return
 *    MOE_ERR_INVALID_SHAPE (forward_qwen3_moe.rs, forward_qwen3_moe: an
 *    incomplete or mismatched MoE shape is an InvalidShape error).
 */
#ifndef MOEQ4K_H
#define MOEQ4K_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_SHAPE = 1,  /* a dimension is out of range or inconsistent */
    MOE_ERR_NULL = 2,           /* a required pointer is NULL */
    MOE_ERR_MISALIGNED = 3,     /* a pointer breaks the alignment rule */
    MOE_ERR_WORKSPACE = 4,      /* workspace smaller than moe_workspace_bytes() */
    MOE_ERR_EXPERT_RANGE = 5,   /* device saw an expert index outside [0,E) */
    MOE_ERR_TIMEOUT = 6,        /* a bounded device-side wait expired */
    MOE_ERR_CUDA = 7,           /* the CUDA runtime reported an error */
    MOE_ERR_INTERNAL = 8,       /* a device-side consistency check failed (a library fault) */
    MOE_ERR_SCRATCH_LIMIT = 9   /* the shape needs more than moe_layer_noalloc's fixed scratch */
} moe_status;

/* Human-readable name of a status code (static string, never NULL). */
MOE_API const char *moe_status_str(moe_status s);

/* Library version as major*10000 + minor*100 + patch. */
MOE_API int moe_version(void);

/*
 * Bytes of device workspace that moe_router / moe_permute / moe_ffn /
 * moe_layer need for this shape (0 when the shape is invalid).  The
 * workspace holds the sticky status word, call and work counters and a
 * 2 KB region of tagged router logits that single-token calls keep between
 * calls (both at the same place for every shape), the permutation, the
 * expert activations h [T*k, I], the per-slot outputs [T*k, H], and the
 * fp16 activation rows, chunk plans and per-expert readiness counts of the
 * tensor-core path.
 */
MOE_API size_t moe_workspace_bytes(int T, int H, int E, int k, int I);

/*
 * Number of kernel launches one moe_layer call enqueues for this shape
 * (0 when the shape is invalid); moe_ffn enqueues all but the router's.
 */
MOE_API int moe_layer_launch_count(int T, int H, int E, int k, int I);

/*
 * Zero the workspace header (status word, counters) and the region of
 * tagged values that single-token calls keep between calls: the first
 * min(ws_bytes, 256 B + 2 KB) bytes.  Call once after allocating a
 * workspace, before its first use (single-token calls rely on that region
 * and the one- and two-token router on a header count starting at zero),
 * and whenever the sticky status should be cleared.  A
 * workspace large enough for several shapes may serve all of them.
 * Enqueued on `stream`.
 */
MOE_API moe_status moe_workspace_init(void *ws_dev, size_t ws_bytes, void *stream);

/*
 * Router (logits, softmax, top-k, renormalise) for T tokens
 * (forward_qwen3_moe_cuda_traced.rs, aprender-serve 0.34.0, doc of
 * forward_qwen3_moe_cuda_traced_with_plan: the router stage is the k
 * post-softmax, renormalised top-k weights of a token).
 *  x_dev [T,H] fp32, Wr_dev [E,H] fp32, bias_dev [E] fp32 or NULL.
 *  Writes idx_dev [T,k] int32 (descending logit, ties -> lowest index; a
 *  NaN logit ranks below every number) and w_dev [T,k] fp32 (sums to 1 per
 *  token).  The logits are fp32 sums; from 256 tokens with E <= 128 they
 *  come from the tensor cores as a three-pass tf32 split product
 *  (hi.hi + lo.hi + hi.lo of each operand's exact hi/lo split, fp32
 *  accumulation), within about 1e-6 of sum |x_h Wr_eh| of the fp32 value.
 *  One launch at every T.  The workspace must have been initialised
 *  (moe_workspace_init); calls that share a workspace must not overlap on
 *  the GPU (true of every call taking a workspace).
 */
MOE_API moe_status moe_router(const float *x_dev, const float *Wr_dev, const float *bias_dev,
                      int T, int H, int E, int k,
                      int32_t *idx_dev, float *w_dev,
                      void *ws_dev, size_t ws_bytes, void *stream);

/*
 * Token->expert permutation of a routing (the pages run the layer one
 * position at a time, forward_qwen3_moe.rs, aprender-serve 0.35.0, step 2g
 * of forward_qwen3_moe; grouping a batch's slots by expert lets each
 * expert's bytes stream once per call): counts_dev [E], offs_dev [E+1]
 * (exclusive prefix sum of counts) and perm_dev [T*k] = slot ids p = t*k+j
 * grouped by expert, ascending p within an expert (stable).  Slots whose
 * expert index is outside [0,E) are left out (perm has offs[E] valid
 * entries) and set the sticky status.
 */
MOE_API moe_status moe_permute(const int32_t *idx_dev, int T, int k, int E,
                       int32_t *counts_dev, int32_t *offs_dev, int32_t *perm_dev,
                       void *ws_dev, size_t ws_bytes, void *stream);

/*
 * Expert FFN and combine for a given routing (forward_qwen3_moe.rs,
 * aprender-serve 0.35.0, step 2h of forward_single_qwen3_moe_with_cache: the
 * gate x up SwiGLU of each selected expert, weighted by the router weights
 * and summed; doc of forward_qwen3_moe, argument `data`: each expert is a
 * fused dequant + matvec over its Q4_K bytes in place).
 *  x_dev [T,H] fp32; idx_dev [T,k] int32; w_dev [T,k] fp32 (any values;
 *  they need not sum to 1); gate/up/down: Q4_K blobs as above.
 *  Writes y_dev [T,H] fp32: y[t] = sum_j w[t,j] * expert_{idx[t,j]}(x[t]),
 *  summed in slot order j = 0..k-1.  Duplicate experts in a row are legal.
 *  An index outside [0,E) contributes nothing and sets the sticky status
 *  MOE_ERR_EXPERT_RANGE (same page, Errors of forward_qwen3_moe: an
 *  out-of-range expert is an error).  Argument errors as for every call.
 */
MOE_API moe_status moe_ffn(const float *x_dev, const int32_t *idx_dev, const float *w_dev,
                   const void *gate_dev, const void *up_dev, const void *down_dev,
                   int T, int H, int E, int k, int I, float *y_dev,
                   void *ws_dev, size_t ws_bytes, void *stream);

/*
 * The whole layer: moe_router then moe_ffn (forward_qwen3_moe.rs,
 * aprender-serve 0.35.0, step 2h of forward_single_qwen3_moe_with_cache and
 * of forward_qwen3_moe: route, then the weighted SwiGLU experts).  idx_dev
 * / w_dev receive the routing (the router stage), y_dev the output stage.  One difference from
 * moe_router, for a single token on the fused kernel: a NaN logit ranks
 * with -inf (below every finite logit, ties to the lowest index) rather
 * than below -inf.
 */
MOE_API moe_status moe_layer(const float *x_dev, const float *Wr_dev, const float *bias_dev,
                     const void *gate_dev, const void *up_dev, const void *down_dev,
                     int T, int H, int E, int k, int I,
                     int32_t *idx_dev, float *w_dev, float *y_dev,
                     void *ws_dev, size_t ws_bytes, void *stream);

/*
 * The layer with the steps on each side of it in a decoder block
 * (forward_qwen3_moe.rs, aprender-serve 0.35.0, steps 2f-2h of
 * forward_qwen3_moe and 2g-2i of forward_single_qwen3_moe_with_cache):
 *   ffn_in = RMSNorm(hidden) = hidden / sqrt(mean(hidden^2) + norm_eps) * norm_w
 *            (per token row; ffn_in = hidden when norm_w_dev is NULL),
 *   the router and the expert FFN of moe_layer on ffn_in (idx_dev, w_dev,
 *   and the FFN output y),
 *   out = hidden + y when add_residual != 0 (hidden += ffn_output), else y.
 *  hidden_dev [T,H] fp32; norm_w_dev [H] fp32 or NULL; norm_eps >= 0 and
 *  finite; out_dev [T,H] fp32 may be hidden_dev itself (an in-place
 *  residual update: every read of hidden precedes the write of its element).
 *  The single-token fused kernel applies the norm while staging the row and
 *  adds the residual at its output store; the other paths run one extra
 *  launch for the norm (into the workspace) and add the residual in the
 *  final combine.
 * Stage capture (forward_qwen3_moe_cuda_traced.rs, aprender-serve 0.34.0, doc
 * of forward_qwen3_moe_cuda_traced_with_plan: the MoeRouter stage is the
 * chosen token's k post-softmax, renormalised weights, MoeFfnOut its [H]
 * FFN output before the residual): when 0 <= capture_token < T, cap_idx_dev
 * [k] int32 and cap_w_dev [k] fp32 receive that token's routing and
 * cap_ffn_dev [H] fp32 its FFN output before the residual add (each
 * pointer NULL to skip it); capture_token = -1 captures nothing and costs
 * nothing.  capture_token outside [-1, T) is MOE_ERR_INVALID_SHAPE.
 *  Workspace: moe_workspace_bytes(T, H, E, k, I), as for moe_layer.
 */
MOE_API moe_status moe_layer_block(const float *hidden_dev, const float *norm_w_dev, float norm_eps,
                                   const float *Wr_dev, const float *bias_dev,
                                   const void *gate_dev, const void *up_dev, const void *down_dev,
                                   int T, int H, int E, int k, int I,
                                   int32_t *idx_dev, float *w_dev, float *out_dev, int add_residual,
                                   int capture_token, int32_t *cap_idx_dev, float *cap_w_dev,
                                   float *cap_ffn_dev, void *ws_dev, size_t ws_bytes, void *stream);

/*
 * The whole layer for a caller whose activations live in host memory:
 * copies x_host [T,H] fp32 to the device, runs moe_layer, copies y back to
 * y_host [T,H] fp32, and synchronises `stream` before returning.  Page-locked
 * host buffers make the copies asynchronous DMA; pageable ones work too.
 * When T = 1 runs on the single-token fused kernel and both buffers are
 * page-locked host memory mapped into the unified address space
 * (cudaHostAlloc, cudaHostRegister, torch's pin_memory), the kernel reads
 * x_host and writes y_host in place instead, with no staging copies; the
 * results are the same.  Device staging for x and y lives in the workspace:
 * size it with moe_workspace_bytes_host().  idx_dev / w_dev are device
 * outputs as in moe_layer.
 */
MOE_API size_t moe_workspace_bytes_host(int T, int H, int E, int k, int I);
MOE_API moe_status moe_layer_host(const float *x_host, const float *Wr_dev, const float *bias_dev,
                          const void *gate_dev, const void *up_dev, const void *down_dev,
                          int T, int H, int E, int k, int I,
                          int32_t *idx_dev, float *w_dev, float *y_host,
                          void *ws_dev, size_t ws_bytes, void *stream);

/*
 * Synchronise `stream`, then return the first device-side error recorded in
 * the workspace since the last moe_workspace_init (MOE_OK if none).  If
 * `detail` is not NULL it receives the offending value (e.g. the expert
 * index seen).
 */
MOE_API moe_status moe_read_device_status(const void *ws_dev, void *stream, int32_t *detail);

/*
 * Q8_K activations (qwen3_moe_dispatch.rs, aprender-serve 0.70.2, doc of
 * cpu_reference: the production CPU path runs the layer on Q8_K
 * activations, as opposed to the fp32-activation path of moe_layer).  Every
 * activation vector that meets a Q4_K matrix is quantised per block of 256
 * consecutive values to one fp32 scale d and 256 signed 8-bit codes q
 * (v ~= d q):  amax = max |v|;  amax = 0 gives d = 0 and all codes 0;
 * otherwise d = amax / 127 and q_i = v_i * (127 / amax) rounded to the
 * nearest integer, halves to even, every step in fp32.
 *
 * moe_quantize_q8k: `rows` rows of n fp32 values (n a multiple of 256,
 * rows * n <= 2^31) at v_dev [rows, n] (16-byte aligned) -> q_dev int8
 * [rows, n] (16-byte aligned), d_dev fp32 [rows, n/256], sums_dev int32
 * [rows, n/32] (each 32-value sub-block's code sum).  Errors:
 * MOE_ERR_INVALID_SHAPE, MOE_ERR_NULL, MOE_ERR_MISALIGNED.
 */
MOE_API moe_status moe_quantize_q8k(const float *v_dev, int rows, int n, int8_t *q_dev,
                                    float *d_dev, int32_t *sums_dev, void *stream);

/*
 * moe_ffn with Q8_K activations: x[t] is quantised; each routed expert's
 * g = W_gate x and u = W_up x are integer Q4_K x Q8_K dot products (per
 * sub-block of 32: d8 (d4 sc P - dmin m S), P the integer dot of the 4-bit
 * and 8-bit codes, S the 8-bit codes' sum); h = SiLU(g) u in fp32 is
 * quantised the same way; o = W_down h likewise; y[t] = sum_j w_j o_j.
 * Arguments, layouts, workspace and errors as moe_ffn (the same workspace
 * size; a slot with an expert index outside [0, E) contributes 0 and is
 * recorded as MOE_ERR_EXPERT_RANGE).  Four launches.
 */
MOE_API moe_status moe_ffn_q8k(const float *x_dev, const int32_t *idx_dev, const float *w_dev,
                       const void *gate_dev, const void *up_dev, const void *down_dev,
                       int T, int H, int E, int k, int I, float *y_dev,
                       void *ws_dev, size_t ws_bytes, void *stream);

/*
 * moe_router (fp32 logits: the router is a dense f32 matvec, not a Q4_K one)
 * then moe_ffn_q8k.  Arguments as moe_layer.
 */
MOE_API moe_status moe_layer_q8k(const float *x_dev, const float *Wr_dev, const float *bias_dev,
                         const void *gate_dev, const void *up_dev, const void *down_dev,
                         int T, int H, int E, int k, int I,
                         int32_t *idx_dev, float *w_dev, float *y_dev,
                         void *ws_dev, size_t ws_bytes, void *stream);

/* Number of kernel launches one moe_layer_q8k call enqueues (0: invalid shape). */
MOE_API int moe_layer_q8k_launch_count(int T, int H, int E, int k, int I);

/*
 * moe_layer for one token without any workspace, for callers that cannot
 * allocate device memory (for example a plugin whose host framework owns
 * every device allocation, or a decode loop that must not reach an
 * allocator on its hot path).  No step of the layer needs it: it exists for
 * those callers only.  Same arguments as moe_layer with T = 1 and no
 * workspace; x, weights, idx, w and y are still the caller's device buffers.
 *
 * Scratch: a fixed 256 KB array in device global memory defined by the
 * library (held on every GPU that loads it until the process exits).  It
 * fits k*I <= 64960 and E <= 256; larger shapes return
 * MOE_ERR_SCRATCH_LIMIT.  Shapes the single-token kernel does not take
 * return MOE_ERR_INVALID_SHAPE.  The call allocates and frees nothing; it
 * clears the scratch's status word with an async memset on `stream`, then
 * launches one kernel.  All calls share the array: calls
 * that overlap on the GPU race and must be serialised by the caller.
 * The first call on each device looks up the array's device address; make
 * that first call before any stream capture.  Only argument and launch
 * errors are returned; device-side errors of this path are not reported.
 */
MOE_API moe_status moe_layer_noalloc(const float *x_dev, const float *Wr_dev, const float *bias_dev,
                                     const void *gate_dev, const void *up_dev, const void *down_dev,
                                     int T, int H, int E, int k, int I,
                                     int32_t *idx_dev, float *w_dev, float *y_dev, void *stream);

/*
 * Test hooks for the bounded device-side waits (not for production use).
 * moe_debug_set_wait_limit: upper bound, in ns, of every device-side wait
 * of later calls (0 restores the default of 1 s).  moe_debug_withhold_arrivals:
 * n != 0 makes CTA 0 of later single-token calls publish none of its router
 * logits and h values, so the other CTAs' waits for them run out; such a
 * call records MOE_ERR_TIMEOUT in the workspace status and writes no output.
 * On the tensor-core batch path, CTA 0 of the gate/up GEMM then counts none
 * of its finished h rows, so the down GEMM's waits for those experts run
 * out: MOE_ERR_TIMEOUT again, and y holds no valid output.
 * Re-initialise the workspace (moe_workspace_init) afterwards to clear the
 * sticky status.
 */
MOE_API void moe_debug_set_wait_limit(unsigned long long ns);
MOE_API void moe_debug_withhold_arrivals(int n);

#ifdef __cplusplus
}
#endif

#endif /* MOEQ4K_H */
