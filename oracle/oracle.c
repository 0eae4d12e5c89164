/*
 * oracle.c -- fp64 CPU oracle for the multi-LoRA fused MoE layer forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline / reference legs load this library.  The product
 * (the CUDA library and its binding) never calls it, and the two share no
 * code, header, table or helper.
 *
 * Source of the method: the AWS machine-learning blog post "Efficiently serve
 * dozens of fine-tuned models with vLLM on Amazon SageMaker AI and Amazon
 * Bedrock" (read in its Spanish and Chinese reprints), section "Implementing
 * multi-LoRA inference for MoE models in vLLM" and Figure 1:
 *   - a router sends each token to its top experts and their outputs are
 *     aggregated;
 *   - each expert is a two-stage feed-forward block: gate_up widens the
 *     hidden state, down narrows it back;
 *   - a LoRA adapter adds to a frozen projection y = xW the product x A B,
 *     computed as a shrink z = x A (h_in -> r) followed by an expand z B
 *     (r -> h_out), with no extra scale;
 *   - with MoE, A and B exist per adapter and per expert, for both gate_up
 *     and down.
 * The pages leave the activation, the aggregation weights and the adapter
 * semantics open; this oracle takes: act = SiLU(gate) * up with
 * SiLU(u) = u / (1 + exp(-u)); gate = the first I outputs of gate_up and up =
 * the last I; out[t] = sum_j w[t][j] * down_j; adapter id l is per token and
 * l = -1 means no LoRA delta.
 *
 * Layout (row-major, "[out][in]": the stored arrays are the transposes of the
 * pages' h_in x h_out matrices): x[T][H], W1[E][2I][H], W2[E][H][I],
 * A1[L][E][r][H], B1[L][E][2I][r], A2[L][E][r][I], B2[L][E][H][r].  Every
 * floating-point input is bfloat16 bits, widened exactly to double.  All
 * arithmetic is fp64 in the plain order of the definition: no blocking, no
 * fusion, no reassociation beyond "base sum, then delta sum, then add".
 *
 * Pairs with an expert id outside [0, E) or a token adapter id outside
 * [-1, L) contribute nothing and are counted in the return value.
 *
 * oracle_forward_w8 is the same layer with FP8 base expert weights (the
 * fused-MoE news item's second optimisation moves MoE weights to FP8): E4M3
 * codes with one fp32 scale per output row, each weight scale * value(code)
 * in fp64, decoded from the format's definition (oracle_e4m3).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int T, H, I, E, k, L, r;
} oracle_dims;

/*
 * FP8 base expert weights (the fused-MoE news item's second optimisation,
 * FP8 MoE weights): W1q [E][2I][H] and W2q [E][H][I] hold 8-bit E4M3 codes,
 * W1s [E][2I] and W2s [E][H] one fp32 scale per output row; the weight is
 * scale * value(code).  The LoRA A and B stay bfloat16.
 */
typedef struct {
    const uint8_t *W1q, *W2q;
    const float *W1s, *W2s;
} oracle_w8;

static double bf(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * Value of an E4M3 code (OCP 8-bit floating point, the finite "fn" variant):
 * sign bit s, 4-bit exponent field f with bias 7, 3-bit mantissa m.  f = 0:
 * subnormal (-1)^s * (m / 8) * 2^-6; f = 15 with m = 7: not a number (the
 * format has no infinities); otherwise (-1)^s * (1 + m / 8) * 2^(f - 7).
 */
double oracle_e4m3(uint8_t c)
{
    const int s = c >> 7, f = (c >> 3) & 15, m = c & 7;
    double v;
    if (f == 15 && m == 7)
        return NAN;
    if (f == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, f - 7);
    return s ? -v : v;
}

/* dot(row of E4M3 codes times the row's scale, vector of double), in index order */
static double dot_w8(const uint8_t *row, float scale, const double *v, long n)
{
    double s = 0.0;
    for (long i = 0; i < n; i++)
        s += ((double)scale * oracle_e4m3(row[i])) * v[i];
    return s;
}

/* SiLU(u) = u * sigmoid(u) = u / (1 + e^{-u}) */
static double silu(double u) { return u / (1.0 + exp(-u)); }

static int pair_valid(const oracle_dims *d, int e, int l)
{
    return e >= 0 && e < d->E && l >= -1 && l < d->L;
}

/* dot(row of bf16, vector of double), length n, summed in index order */
static double dot_bf(const uint16_t *row, const double *v, long n)
{
    double s = 0.0;
    for (long i = 0; i < n; i++)
        s += bf(row[i]) * v[i];
    return s;
}

/*
 * One (token, slot) pair: the expert FFN of expert e with the LoRA deltas of
 * adapter l, for the token's hidden state xd[H] (already widened).
 * Outputs (each may be NULL): z1[r], g[2I], act[I], z2[r], dv[H].
 * work must hold 2I + I + H + 2r doubles.
 */
static void pair_ffn(const oracle_dims *d, const double *xd, int e, int l,
                     const uint16_t *W1, const uint16_t *W2, const oracle_w8 *q,
                     const uint16_t *A1,
                     const uint16_t *B1, const uint16_t *A2, const uint16_t *B2,
                     double *work, double *z1_out, double *g_out, double *act_out,
                     double *z2_out, double *d_out)
{
    const long H = d->H, I = d->I, E = d->E, r = d->r;
    double *g = work;            /* 2I */
    double *act = g + 2 * I;     /* I  */
    double *dv = act + I;        /* H  */
    double *z1 = dv + H;         /* r  */
    double *z2 = z1 + r;         /* r  */
    const int lora = (l >= 0) && A1 && B1 && A2 && B2 && r > 0;

    /* gate_up base: g = W1[e] x (bf16 weights, or FP8 codes times their row's scale) */
    if (!q) {
        for (long o = 0; o < 2 * I; o++)
            g[o] = dot_bf(W1 + ((long)e * 2 * I + o) * H, xd, H);
    } else {
        for (long o = 0; o < 2 * I; o++)
            g[o] = dot_w8(q->W1q + ((long)e * 2 * I + o) * H, q->W1s[(long)e * 2 * I + o], xd, H);
    }
    /* gate_up LoRA: shrink z1 = A1[l][e] x, expand g += B1[l][e] z1 */
    if (lora) {
        for (long q = 0; q < r; q++)
            z1[q] = dot_bf(A1 + (((long)l * E + e) * r + q) * H, xd, H);
        for (long o = 0; o < 2 * I; o++)
            g[o] += dot_bf(B1 + (((long)l * E + e) * 2 * I + o) * r, z1, r);
    } else {
        for (long q = 0; q < r; q++)
            z1[q] = 0.0;
    }
    /* activation: SiLU(gate) * up */
    for (long i = 0; i < I; i++)
        act[i] = silu(g[i]) * g[I + i];
    /* down base: dv = W2[e] act */
    if (!q) {
        for (long h = 0; h < H; h++)
            dv[h] = dot_bf(W2 + ((long)e * H + h) * I, act, I);
    } else {
        for (long h = 0; h < H; h++)
            dv[h] = dot_w8(q->W2q + ((long)e * H + h) * I, q->W2s[(long)e * H + h], act, I);
    }
    /* down LoRA: shrink z2 = A2[l][e] act, expand dv += B2[l][e] z2 */
    if (lora) {
        for (long q = 0; q < r; q++)
            z2[q] = dot_bf(A2 + (((long)l * E + e) * r + q) * I, act, I);
        for (long h = 0; h < H; h++)
            dv[h] += dot_bf(B2 + (((long)l * E + e) * H + h) * r, z2, r);
    } else {
        for (long q = 0; q < r; q++)
            z2[q] = 0.0;
    }
    if (z1_out) memcpy(z1_out, z1, sizeof(double) * r);
    if (g_out) memcpy(g_out, g, sizeof(double) * 2 * I);
    if (act_out) memcpy(act_out, act, sizeof(double) * I);
    if (z2_out) memcpy(z2_out, z2, sizeof(double) * r);
    if (d_out) memcpy(d_out, dv, sizeof(double) * H);
}

static int dims_ok(const oracle_dims *d)
{
    return d && d->T >= 0 && d->H > 0 && d->I > 0 && d->E > 0 && d->k > 0 &&
           d->L >= 0 && d->r >= 0;
}

/*
 * Layer forward for a list of tokens (tokens == NULL: all T tokens in order).
 * out[n][H] receives the unrounded fp64 result of token tokens[n].
 * Returns the number of invalid pairs met, or -1 on bad arguments.
 */
static long forward_impl(const oracle_dims *d, const uint16_t *x, const int32_t *topk_ids,
                         const float *topk_weights, const int32_t *lora_ids,
                         const uint16_t *W1, const uint16_t *W2, const oracle_w8 *q,
                         const uint16_t *A1, const uint16_t *B1, const uint16_t *A2,
                         const uint16_t *B2, const int32_t *tokens, int n_tokens, double *out,
                         int n_threads)
{
    if (!dims_ok(d) || !x || !topk_ids || !topk_weights || !lora_ids || !out)
        return -1;
    if (q ? !(q->W1q && q->W2q && q->W1s && q->W2s) : !(W1 && W2))
        return -1;
    if (!tokens)
        n_tokens = d->T;
    for (int n = 0; n < n_tokens; n++)
        if (tokens && (tokens[n] < 0 || tokens[n] >= d->T))
            return -1;
    const long H = d->H, I = d->I, r = d->r;
    long invalid = 0;
    if (n_threads <= 0)
        n_threads = 1;

#pragma omp parallel num_threads(n_threads) reduction(+ : invalid)
    {
        double *work = (double *)malloc(sizeof(double) * (size_t)(2 * I + I + H + 2 * r));
        double *xd = (double *)malloc(sizeof(double) * (size_t)H);
        double *dv = (double *)malloc(sizeof(double) * (size_t)H);
#pragma omp for schedule(dynamic, 1)
        for (int n = 0; n < n_tokens; n++) {
            const int t = tokens ? tokens[n] : n;
            double *acc = out + (long)n * H;
            for (long h = 0; h < H; h++) {
                acc[h] = 0.0;
                xd[h] = bf(x[(long)t * H + h]);
            }
            const int l = lora_ids[t];
            for (int j = 0; j < d->k; j++) {
                const int e = topk_ids[(long)t * d->k + j];
                if (!pair_valid(d, e, l)) {
                    invalid++;
                    continue;
                }
                const double w = (double)topk_weights[(long)t * d->k + j];
                pair_ffn(d, xd, e, l, W1, W2, q, A1, B1, A2, B2, work, NULL, NULL, NULL, NULL, dv);
                /* weighted aggregation over the token's k experts, in slot order */
                for (long h = 0; h < H; h++)
                    acc[h] += w * dv[h];
            }
        }
        free(work);
        free(xd);
        free(dv);
    }
    return invalid;
}

long oracle_forward(const oracle_dims *d, const uint16_t *x, const int32_t *topk_ids,
                    const float *topk_weights, const int32_t *lora_ids,
                    const uint16_t *W1, const uint16_t *W2, const uint16_t *A1,
                    const uint16_t *B1, const uint16_t *A2, const uint16_t *B2,
                    const int32_t *tokens, int n_tokens, double *out, int n_threads)
{
    return forward_impl(d, x, topk_ids, topk_weights, lora_ids, W1, W2, NULL, A1, B1, A2, B2,
                        tokens, n_tokens, out, n_threads);
}

/*
 * The same forward with FP8 base expert weights: W1q [E][2I][H], W2q [E][H][I]
 * E4M3 codes, W1s [E][2I], W2s [E][H] fp32 row scales (weight = scale *
 * value(code)); the LoRA matrices stay bf16.
 */
long oracle_forward_w8(const oracle_dims *d, const uint16_t *x, const int32_t *topk_ids,
                       const float *topk_weights, const int32_t *lora_ids,
                       const uint8_t *W1q, const float *W1s, const uint8_t *W2q,
                       const float *W2s, const uint16_t *A1, const uint16_t *B1,
                       const uint16_t *A2, const uint16_t *B2, const int32_t *tokens,
                       int n_tokens, double *out, int n_threads)
{
    const oracle_w8 q = {W1q, W2q, W1s, W2s};
    return forward_impl(d, x, topk_ids, topk_weights, lora_ids, NULL, NULL, &q, A1, B1, A2, B2,
                        tokens, n_tokens, out, n_threads);
}

/*
 * Intermediates of pair p = t*k + j (each output may be NULL):
 * z1[r], g[2I] (gate_up after the LoRA add), act[I], z2[r], dvec[H] (down
 * after the LoRA add, before the top-k weight).
 * Returns 0, 1 if the pair is invalid (outputs zero-filled), -1 on bad args.
 */
int oracle_pair(const oracle_dims *d, const uint16_t *x, const int32_t *topk_ids,
                const int32_t *lora_ids, const uint16_t *W1, const uint16_t *W2,
                const uint16_t *A1, const uint16_t *B1, const uint16_t *A2, const uint16_t *B2,
                long p, double *z1, double *g, double *act, double *z2, double *dvec)
{
    if (!dims_ok(d) || !x || !topk_ids || !lora_ids || !W1 || !W2)
        return -1;
    if (p < 0 || p >= (long)d->T * d->k)
        return -1;
    const long H = d->H, I = d->I, r = d->r;
    const long t = p / d->k;
    const int e = topk_ids[p], l = lora_ids[t];
    if (!pair_valid(d, e, l)) {
        if (z1) memset(z1, 0, sizeof(double) * r);
        if (g) memset(g, 0, sizeof(double) * 2 * I);
        if (act) memset(act, 0, sizeof(double) * I);
        if (z2) memset(z2, 0, sizeof(double) * r);
        if (dvec) memset(dvec, 0, sizeof(double) * H);
        return 1;
    }
    double *work = (double *)malloc(sizeof(double) * (size_t)(2 * I + I + H + 2 * r));
    double *xd = (double *)malloc(sizeof(double) * (size_t)H);
    for (long h = 0; h < H; h++)
        xd[h] = bf(x[t * H + h]);
    pair_ffn(d, xd, e, l, W1, W2, NULL, A1, B1, A2, B2, work, z1, g, act, z2, dvec);
    free(work);
    free(xd);
    return 0;
}

/*
 * Expert x adapter bucketing of the (token, slot) pairs -- the "extra grid
 * dimension for the active adapters" of the blog's section "Implementing
 * multi-LoRA inference for MoE models in vLLM", written as a stable counting
 * sort.  Pair p = t*k + j has expert e = topk_ids[p] and adapter
 * l = lora_ids[t]; its bucket is b = e*(L+1) + (l+1), so buckets run
 * expert-major, adapters from -1 to L-1.  Within a bucket pairs keep
 * ascending p.  Each non-empty bucket is padded up to a multiple of bm with
 * the sentinel value P = T*k; empty buckets take no room.  Invalid pairs are
 * left out.
 *
 * Outputs: sorted_ids[cap] (entries past *num_post_padded untouched),
 * tile_expert / tile_lora (one entry per bm-row tile), *num_post_padded,
 * bucket_count[E*(L+1)] (valid pairs per bucket), bucket_offset[E*(L+1)+1]
 * (padded start of each bucket).  Returns the number of invalid pairs, -1 on
 * bad arguments, -2 if cap is too small.
 */
long oracle_align(int T, int k, int E, int L, int bm, const int32_t *topk_ids,
                  const int32_t *lora_ids, int32_t *sorted_ids, long cap,
                  int32_t *tile_expert, int32_t *tile_lora, int32_t *num_post_padded,
                  int32_t *bucket_count, int32_t *bucket_offset)
{
    if (T < 0 || k <= 0 || E <= 0 || L < 0 || bm <= 0 || !topk_ids || !lora_ids ||
        !sorted_ids || !tile_expert || !tile_lora || !num_post_padded || !bucket_count ||
        !bucket_offset)
        return -1;
    const long P = (long)T * k;
    const long NB = (long)E * (L + 1);
    long invalid = 0;

    /* 1. count */
    for (long b = 0; b < NB; b++)
        bucket_count[b] = 0;
    for (long p = 0; p < P; p++) {
        const int e = topk_ids[p], l = lora_ids[p / k];
        if (e < 0 || e >= E || l < -1 || l >= L) {
            invalid++;
            continue;
        }
        bucket_count[(long)e * (L + 1) + (l + 1)]++;
    }
    /* 2. padded offsets */
    long off = 0;
    for (long b = 0; b < NB; b++) {
        bucket_offset[b] = (int32_t)off;
        off += ((bucket_count[b] + bm - 1) / bm) * (long)bm;
    }
    bucket_offset[NB] = (int32_t)off;
    if (off > cap)
        return -2;
    /* 3. stable placement: walking p upward keeps ascending p within a bucket */
    long *cursor = (long *)malloc(sizeof(long) * (size_t)(NB > 0 ? NB : 1));
    for (long b = 0; b < NB; b++)
        cursor[b] = bucket_offset[b];
    for (long p = 0; p < P; p++) {
        const int e = topk_ids[p], l = lora_ids[p / k];
        if (e < 0 || e >= E || l < -1 || l >= L)
            continue;
        const long b = (long)e * (L + 1) + (l + 1);
        sorted_ids[cursor[b]++] = (int32_t)p;
    }
    /* 4. padding and per-tile (expert, adapter) labels */
    for (long b = 0; b < NB; b++) {
        for (long q = cursor[b]; q < bucket_offset[b + 1]; q++)
            sorted_ids[q] = (int32_t)P;
        for (long q = bucket_offset[b]; q < bucket_offset[b + 1]; q += bm) {
            tile_expert[q / bm] = (int32_t)(b / (L + 1));
            tile_lora[q / bm] = (int32_t)(b % (L + 1)) - 1;
        }
    }
    free(cursor);
    *num_post_padded = (int32_t)off;
    return invalid;
}

/* Capacity that always suffices for oracle_align: P + min(NB, P) * (bm - 1). */
long oracle_align_capacity(int T, int k, int E, int L, int bm)
{
    const long P = (long)T * k, NB = (long)E * (L + 1);
    const long nonempty = NB < P ? NB : P;
    return P + nonempty * (long)(bm - 1);
}
