/*
 * CPU oracle for the routed-expert Q4_K MoE FFN layer.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, fp64 statement of
 * what the layer computes.  Only the test-suite, the smoke check and the
 * benchmark's CPU-baseline leg load it; the product path never does.  It
 * shares no code, header or table with the CUDA library.
 *
 * What it follows (page title, then the item on the page):
 *  - forward_qwen3_moe.rs (aprender-serve 0.35.0), step 2h of
 *    forward_single_qwen3_moe_with_cache: the MoE FFN output is the gate x up
 *    SwiGLU of each selected expert, weighted by the softmax-normalised top-k
 *    router weights;
 *  - same page, doc of forward_qwen3_moe ("Arguments", `data`): each
 *    selected expert is a dequant+matvec over the Q4_K bytes in place;
 *  - same page, step 2g of forward_qwen3_moe: every position goes through
 *    the layer on its own (tokens are independent);
 *  - forward_qwen3_moe_cuda_traced.rs (aprender-serve 0.34.0), doc of
 *    forward_qwen3_moe_cuda_traced_with_plan: the router stage is the k
 *    post-softmax, renormalised top-k weights, the output stage is [H];
 *  - qwen3_moe_dispatch.rs (aprender-serve 0.70.2), doc of cpu_reference:
 *    activations enter as exact fp32 values (no Q8_K quantisation).
 * The Q4_K block layout is the GGUF format named by those pages ("Q4_K_M");
 * the pages do not spell it out, so the field placement below is the format's
 * public definition, restated.
 *
 * Readings where the pages leave a step open:
 *  - softmax over all E logits, then the k largest probabilities in
 *    descending order, equal values by lowest expert index; the k weights are
 *    the selected probabilities divided by their sum;
 *  - SiLU applies to the gate projection, SiLU(z) = z / (1 + exp(-z));
 *    the up projection is linear; h = SiLU(g) * u; o = W_down h;
 *  - y = sum over slots j = 0..k-1, in slot order, of w_j * o_j;
 *  - a slot whose expert index is outside [0, E) contributes nothing and is
 *    reported through the status count.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define QK 256
#define BLK 144

/* IEEE binary16 -> double, exactly, subnormals included. */
static double half_bits_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 31;
    int mant = h & 1023;
    double v;
    if (expo == 0)
        v = ldexp((double)mant, -24);            /* subnormal or zero */
    else if (expo == 31)
        v = mant ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + mant), expo - 25);
    return sign ? -v : v;
}

/* The 6-bit scale and min of sub-block j (0..7) from the 12 packed bytes. */
static void scale_min(const uint8_t *scales, int j, int *sc, int *m)
{
    if (j < 4) {
        *sc = scales[j] & 63;
        *m = scales[j + 4] & 63;
    } else {
        *sc = (scales[j + 4] & 15) | ((scales[j - 4] >> 6) << 4);
        *m = (scales[j + 4] >> 4) | ((scales[j] >> 6) << 4);
    }
}

/* Decode one 144-byte block into its 256 weights, in weight order. */
void moq_decode_block(const uint8_t *blk, double *out)
{
    uint16_t dbits = (uint16_t)(blk[0] | (blk[1] << 8));
    uint16_t mbits = (uint16_t)(blk[2] | (blk[3] << 8));
    double d = half_bits_to_double(dbits);
    double dmin = half_bits_to_double(mbits);
    const uint8_t *scales = blk + 4;
    const uint8_t *qs = blk + 16;
    for (int i = 0; i < QK; i++) {
        int j = i / 32;               /* sub-block */
        int c = i / 64;               /* 32-byte chunk of qs */
        int l = i % 32;               /* position inside the sub-block */
        int hi = (i % 64) >= 32;      /* second sub-block of the chunk -> high nibble */
        uint8_t byte = qs[32 * c + l];
        int q = hi ? (byte >> 4) : (byte & 15);
        int sc, m;
        scale_min(scales, j, &sc, &m);
        out[i] = d * (double)sc * (double)q - dmin * (double)m;
    }
}

/* Decode `nrows` rows of `ncols` weights (ncols a multiple of 256). */
void moq_decode_rows(const uint8_t *blob, long nrows, int ncols, double *out)
{
    int nsb = ncols / QK;
    for (long r = 0; r < nrows; r++)
        for (int s = 0; s < nsb; s++)
            moq_decode_block(blob + (r * nsb + s) * BLK, out + r * ncols + (long)s * QK);
}

/* Dot product of one Q4_K row (ncols weights) with a double vector. */
static double row_dot(const uint8_t *row, int ncols, const double *v, double *tmp)
{
    int nsb = ncols / QK;
    double acc = 0.0;
    for (int s = 0; s < nsb; s++) {
        moq_decode_block(row + (long)s * BLK, tmp);
        for (int i = 0; i < QK; i++)
            acc += tmp[i] * v[s * QK + i];
    }
    return acc;
}

/*
 * Router: logits l = x Wr^T (+ bias), p = softmax over all E, the k largest
 * p (ties -> lowest index) in descending order, w = p_sel / sum(p_sel).
 * x [T,H], Wr [E,H] fp32, bias [E] fp32 or NULL.
 * Outputs: logits [T,E] (biased, fp64), p [T,E], idx [T,k], w [T,k].
 */
void moq_router(const float *x, const float *Wr, const float *bias,
                int T, int H, int E, int k,
                double *logits, double *p, int32_t *idx, double *w)
{
#pragma omp parallel for schedule(dynamic)
    for (int t = 0; t < T; t++) {
        double *l = logits + (long)t * E;
        double *pt = p + (long)t * E;
        for (int e = 0; e < E; e++) {
            double acc = 0.0;
            for (int h = 0; h < H; h++)
                acc += (double)x[(long)t * H + h] * (double)Wr[(long)e * H + h];
            l[e] = acc + (bias ? (double)bias[e] : 0.0);
        }
        double mx = l[0];
        for (int e = 1; e < E; e++)
            if (l[e] > mx) mx = l[e];
        double z = 0.0;
        for (int e = 0; e < E; e++) {
            pt[e] = exp(l[e] - mx);
            z += pt[e];
        }
        for (int e = 0; e < E; e++)
            pt[e] /= z;
        /* selection by repeated maximum: strict '>' keeps the lowest index on ties */
        char *taken = calloc((size_t)E, 1);
        double sel_sum = 0.0;
        for (int j = 0; j < k; j++) {
            int best = -1;
            for (int e = 0; e < E; e++)
                if (!taken[e] && (best < 0 || pt[e] > pt[best]))
                    best = e;
            taken[best] = 1;
            idx[(long)t * k + j] = best;
            sel_sum += pt[best];
        }
        for (int j = 0; j < k; j++)
            w[(long)t * k + j] = pt[idx[(long)t * k + j]] / sel_sum;
        free(taken);
    }
}

/*
 * One expert applied to one activation row: g = W_gate x, u = W_up x,
 * h = SiLU(g) * u, o = W_down h.  gate/up: [I rows x H], down: [H rows x I].
 */
void moq_expert(const double *xv, const uint8_t *gate_e, const uint8_t *up_e,
                const uint8_t *down_e, int H, int I, double *h, double *o)
{
    int nsb_h = H / QK, nsb_i = I / QK;
    /* Rows are independent: when this runs outside a parallel region (fewer
     * tokens than threads), the rows are shared out over the threads.  Each
     * row's dot product is the same sequential sum either way. */
#ifdef _OPENMP
    int outer = !omp_in_parallel();
#else
    int outer = 0;
#endif
#pragma omp parallel for schedule(static) if (outer)
    for (int r = 0; r < I; r++) {
        double tmp[QK];
        double g = row_dot(gate_e + (long)r * nsb_h * BLK, H, xv, tmp);
        double u = row_dot(up_e + (long)r * nsb_h * BLK, H, xv, tmp);
        h[r] = g / (1.0 + exp(-g)) * u;
    }
#pragma omp parallel for schedule(static) if (outer)
    for (int r = 0; r < H; r++) {
        double tmp[QK];
        o[r] = row_dot(down_e + (long)r * nsb_i * BLK, I, h, tmp);
    }
}

/*
 * The FFN for the listed tokens (all T when `tokens` is NULL, else
 * `ntok` entries of `tokens`): y[t] = sum_j w[t,j] * expert_{idx[t,j]}(x[t]).
 * y is [T,H] (only the listed rows are written).  Returns the number of
 * slots skipped for an out-of-range expert index.
 */
long moq_ffn(const float *x, const int32_t *idx, const double *w,
             const uint8_t *gate, const uint8_t *up, const uint8_t *down,
             int T, int H, int E, int k, int I,
             const int32_t *tokens, int ntok, double *y)
{
    long gate_bytes = (long)I * (H / QK) * BLK;
    long down_bytes = (long)H * (I / QK) * BLK;
    int n = tokens ? ntok : T;
    long skipped = 0;
    /* Tokens in parallel when there are at least as many as threads; else
     * one token at a time, with each expert's rows in parallel. */
#ifdef _OPENMP
    int by_token = n >= omp_get_max_threads();
#else
    int by_token = 0;
#endif
#pragma omp parallel for schedule(dynamic) reduction(+ : skipped) if (by_token)
    for (int a = 0; a < n; a++) {
        int t = tokens ? tokens[a] : a;
        double *xv = malloc(sizeof(double) * (size_t)H);
        double *h = malloc(sizeof(double) * (size_t)I);
        double *o = malloc(sizeof(double) * (size_t)H);
        double *yt = y + (long)t * H;
        for (int i = 0; i < H; i++) {
            xv[i] = (double)x[(long)t * H + i];
            yt[i] = 0.0;
        }
        for (int j = 0; j < k; j++) {
            int e = idx[(long)t * k + j];
            if (e < 0 || e >= E) {
                skipped++;
                continue;
            }
            moq_expert(xv, gate + e * gate_bytes, up + e * gate_bytes, down + e * down_bytes,
                       H, I, h, o);
            double wj = w[(long)t * k + j];
            for (int i = 0; i < H; i++)
                yt[i] += wj * o[i];
        }
        free(xv);
        free(h);
        free(o);
    }
    return skipped;
}

/*
 * Q8_K activations (qwen3_moe_dispatch.rs, aprender-serve 0.70.2, doc of
 * cpu_reference: the production CPU path quantises activations to Q8_K for
 * its integer dot products; the fp32-activation path above is the other
 * scope).  The pages name the format, not its arithmetic.  Reading: every
 * block of 256 consecutive activations gets one fp32 scale d and 256 signed
 * 8-bit codes q with v ~= d q, symmetric around zero, the block's largest
 * magnitude at +-127:
 *     amax = max_i |v_i|;   amax = 0 gives d = 0 and all codes 0;
 *     otherwise s = 127 / amax and d = amax / 127 (fp32 divisions, rounded
 *     to nearest), q_i = v_i * s (fp32 product) rounded to the nearest
 *     integer, halves to even.
 * Every step is fp32, so a kernel taking the same steps decides the same
 * codes.  `sums` receives each 32-element sub-block's code sum.
 */
void moq_q8k_quantize(const float *v, long nblocks, int8_t *q, float *d, int32_t *sums)
{
    for (long b = 0; b < nblocks; b++) {
        const float *vb = v + b * QK;
        int8_t *qb = q + b * QK;
        float amax = 0.0f;
        for (int i = 0; i < QK; i++)
            if (fabsf(vb[i]) > amax)
                amax = fabsf(vb[i]);
        if (amax == 0.0f) {
            d[b] = 0.0f;
            for (int i = 0; i < QK; i++)
                qb[i] = 0;
        } else {
            float s = 127.0f / amax;
            d[b] = amax / 127.0f;
            for (int i = 0; i < QK; i++) {
                float t = vb[i] * s;
                qb[i] = (int8_t)rintf(t);   /* default rounding mode: halves to even */
            }
        }
        for (int j = 0; j < QK / 32; j++) {
            int32_t acc = 0;
            for (int i = 0; i < 32; i++)
                acc += qb[32 * j + i];
            sums[b * (QK / 32) + j] = acc;
        }
    }
}

/*
 * Dot product of one Q4_K row (nsb blocks) with a Q8_K vector of the same
 * length: per block b and sub-block j, with the exact integers
 * P = sum_i q4_i q8_i and S = sum_i q8_i (the sub-block's code sum),
 *     sum_b d8_b * sum_j (d4_b sc_j P - dmin_b m_j S)
 * in fp64, i.e. the dot of the dequantised row with the vector d8 q8.
 */
double moq_row_dot_q8k(const uint8_t *row, int nsb, const int8_t *q, const float *d,
                       const int32_t *sums)
{
    double acc = 0.0;
    for (int b = 0; b < nsb; b++) {
        const uint8_t *blk = row + (long)b * BLK;
        double d4 = half_bits_to_double((uint16_t)(blk[0] | (blk[1] << 8)));
        double dmin = half_bits_to_double((uint16_t)(blk[2] | (blk[3] << 8)));
        const uint8_t *qs = blk + 16;
        const int8_t *qb = q + (long)b * QK;
        double bacc = 0.0;
        for (int j = 0; j < QK / 32; j++) {
            int sc, m;
            scale_min(blk + 4, j, &sc, &m);
            long P = 0;
            for (int l = 0; l < 32; l++) {
                uint8_t byte = qs[32 * (j / 2) + l];   /* sub-blocks 2c, 2c+1 share 32 bytes */
                int q4 = (j % 2) ? (byte >> 4) : (byte & 15);
                P += (long)q4 * qb[32 * j + l];
            }
            bacc += d4 * (double)sc * (double)P - dmin * (double)m * (double)sums[b * (QK / 32) + j];
        }
        acc += (double)d[b] * bacc;
    }
    return acc;
}

/*
 * One expert on one token with Q8_K activations: g, u = Q4_K x Q8_K dots
 * with the quantised x; h = SiLU(g) u in fp64, rounded to fp32 and quantised
 * (the down projection's input is an activation vector too); o = the
 * Q4_K x Q8_K dots of the down rows with the quantised h.
 */
static void expert_q8k(const int8_t *xq, const float *xd, const int32_t *xs, const uint8_t *gate_e,
                       const uint8_t *up_e, const uint8_t *down_e, int H, int I, float *hf,
                       int8_t *hq, float *hd, int32_t *hs, double *o)
{
    int nsb_h = H / QK, nsb_i = I / QK;
#ifdef _OPENMP
    int outer = !omp_in_parallel();
#else
    int outer = 0;
#endif
#pragma omp parallel for schedule(static) if (outer)
    for (int r = 0; r < I; r++) {
        double g = moq_row_dot_q8k(gate_e + (long)r * nsb_h * BLK, nsb_h, xq, xd, xs);
        double u = moq_row_dot_q8k(up_e + (long)r * nsb_h * BLK, nsb_h, xq, xd, xs);
        hf[r] = (float)(g / (1.0 + exp(-g)) * u);
    }
    moq_q8k_quantize(hf, nsb_i, hq, hd, hs);
#pragma omp parallel for schedule(static) if (outer)
    for (int r = 0; r < H; r++)
        o[r] = moq_row_dot_q8k(down_e + (long)r * nsb_i * BLK, nsb_i, hq, hd, hs);
}

/*
 * The FFN with Q8_K activations for the listed tokens (all T when `tokens`
 * is NULL): x[t] is quantised, each routed expert runs expert_q8k, and
 * y[t] = sum_j w[t,j] o_j in slot order.  Returns the number of slots
 * skipped for an out-of-range expert index.
 */
long moq_ffn_q8k(const float *x, const int32_t *idx, const double *w,
                 const uint8_t *gate, const uint8_t *up, const uint8_t *down,
                 int T, int H, int E, int k, int I,
                 const int32_t *tokens, int ntok, double *y)
{
    long gate_bytes = (long)I * (H / QK) * BLK;
    long down_bytes = (long)H * (I / QK) * BLK;
    int n = tokens ? ntok : T;
    long skipped = 0;
#ifdef _OPENMP
    int by_token = n >= omp_get_max_threads();
#else
    int by_token = 0;
#endif
#pragma omp parallel for schedule(dynamic) reduction(+ : skipped) if (by_token)
    for (int a = 0; a < n; a++) {
        int t = tokens ? tokens[a] : a;
        int8_t *xq = malloc((size_t)H);
        float *xd = malloc(sizeof(float) * (size_t)(H / QK));
        int32_t *xs = malloc(sizeof(int32_t) * (size_t)(H / 32));
        float *hf = malloc(sizeof(float) * (size_t)I);
        int8_t *hq = malloc((size_t)I);
        float *hd = malloc(sizeof(float) * (size_t)(I / QK));
        int32_t *hs = malloc(sizeof(int32_t) * (size_t)(I / 32));
        double *o = malloc(sizeof(double) * (size_t)H);
        double *yt = y + (long)t * H;
        moq_q8k_quantize(x + (long)t * H, H / QK, xq, xd, xs);
        for (int i = 0; i < H; i++)
            yt[i] = 0.0;
        for (int j = 0; j < k; j++) {
            int e = idx[(long)t * k + j];
            if (e < 0 || e >= E) {
                skipped++;
                continue;
            }
            expert_q8k(xq, xd, xs, gate + e * gate_bytes, up + e * gate_bytes, down + e * down_bytes,
                       H, I, hf, hq, hd, hs, o);
            double w_slot = w[(long)t * k + j];
            for (int i = 0; i < H; i++)
                yt[i] += w_slot * o[i];
        }
        free(xq);
        free(xd);
        free(xs);
        free(hf);
        free(hq);
        free(hd);
        free(hs);
        free(o);
    }
    return skipped;
}

/*
 * Pre-FFN RMSNorm (forward_qwen3_moe.rs, aprender-serve 0.35.0, step 2f of
 * forward_qwen3_moe and step 2g of forward_single_qwen3_moe_with_cache:
 * ffn_input = rms_norm(hidden, ffn_norm_weight, eps)).  The pages name the
 * operation, not its formula; the reading is the usual root-mean-square
 * norm, per token row:
 *     out[i] = x[i] / sqrt(mean_i(x[i]^2) + eps) * gamma[i]
 * computed in fp64 and rounded once to fp32 at the end, because the pages'
 * ffn_input is an f32 vector that the MoE FFN then consumes.
 */
void moq_rmsnorm(const float *x, const float *gamma, double eps, int T, int H, float *out)
{
    for (int t = 0; t < T; t++) {
        const float *xt = x + (long)t * H;
        double ss = 0.0;
        for (int i = 0; i < H; i++)
            ss += (double)xt[i] * (double)xt[i];
        double inv = 1.0 / sqrt(ss / (double)H + eps);
        for (int i = 0; i < H; i++)
            out[(long)t * H + i] = (float)((double)xt[i] * inv * (double)gamma[i]);
    }
}

/*
 * Residual after the MoE FFN (same page, step 2h of forward_qwen3_moe and
 * step 2i of forward_single_qwen3_moe_with_cache: hidden += ffn_output):
 * out = hidden + y, elementwise, in fp64.
 */
void moq_add_residual(const float *hidden, const double *y, long n, double *out)
{
    for (long i = 0; i < n; i++)
        out[i] = (double)hidden[i] + y[i];
}

/*
 * Token->expert permutation: counts[e] = number of (t,j) slots routed to e,
 * offs = exclusive prefix sum of counts (E+1 entries), perm = slot ids
 * p = t*k + j ordered by (expert, p).  Out-of-range slots are left out.
 */
void moq_permutation(const int32_t *idx, int T, int k, int E,
                     int32_t *counts, int32_t *offs, int32_t *perm)
{
    long n = (long)T * k;
    for (int e = 0; e < E; e++)
        counts[e] = 0;
    for (long p = 0; p < n; p++)
        if (idx[p] >= 0 && idx[p] < E)
            counts[idx[p]]++;
    offs[0] = 0;
    for (int e = 0; e < E; e++)
        offs[e + 1] = offs[e] + counts[e];
    int32_t *cursor = malloc(sizeof(int32_t) * (size_t)E);
    for (int e = 0; e < E; e++)
        cursor[e] = offs[e];
    for (long p = 0; p < n; p++)
        if (idx[p] >= 0 && idx[p] < E)
            perm[cursor[idx[p]]++] = (int32_t)p;
    free(cursor);
}

void moq_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int moq_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
