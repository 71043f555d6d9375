/*
 * dg_oracle.c -- plain, slow, single-threaded fp64 oracle for one
 * block-diffusion denoising step (DiffusionGemma-style sampler).
 *
 * TEST INFRASTRUCTURE ONLY.  This file exists to check the CUDA library
 * against the method as the pages describe it.  Only the test-suite, the
 * smoke check and the CPU-baseline leg of the benchmark may load it.  It
 * shares no code, header, table or constant generator with the CUDA path.
 *
 * Sources (web pages, by title and section):
 *   [Lab]  "DiffusionGemma Lab", section 2 "The generation algorithm, as
 *          written in the code", items 1-7.
 *   [PD]   "DiffusionGemma: Parallel Denoising From an Autoregressive
 *          Checkpoint", section "Finding", the three sampler bullets
 *          (entropy-bounded acceptance, temperature annealing, adaptive
 *          stopping) and the architecture paragraph.
 *   [SC11] Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as
 *          1, 2, 3" (SC'11): the Philox4x32 bijection, 10 rounds.
 *
 * Floating point: everything is fp64 except the Gumbel score, which the
 * method (as read here) defines as an fp32 sequence so that two independent
 * implementations agree bit for bit on identical fp32 logits.  Build with
 * -ffp-contract=off and without -ffast-math: every fused multiply-add below
 * is an explicit fmaf().
 *
 * Parity status: every function below is pinned by a CPU test against a
 * closed form, a published known-answer vector, a library routine or brute
 * force, except the end-to-end step count of a converging block loop, which
 * has no page value ("parity unpinned" for that number only).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* Philox4x32-10 [SC11]: 4x32-bit counter, 2x32-bit key, 10 rounds.     */
/* Round: (L0,R0,L1,R1) -> (hi(M1*L1)^R0^k0, lo(M1*L1),                 */
/*                          hi(M0*L0)^R1^k1, lo(M0*L0)); the key is      */
/* bumped by the Weyl constants between rounds.                          */
/* ------------------------------------------------------------------ */
#define ORC_PHILOX_M0 0xD2511F53u
#define ORC_PHILOX_M1 0xCD9E8D57u
#define ORC_PHILOX_W0 0x9E3779B9u
#define ORC_PHILOX_W1 0xBB67AE85u

void orc_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4])
{
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int round = 0; round < 10; ++round) {
        uint64_t p0 = (uint64_t)ORC_PHILOX_M0 * (uint64_t)c0;
        uint64_t p1 = (uint64_t)ORC_PHILOX_M1 * (uint64_t)c2;
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        uint32_t n0 = hi1 ^ c1 ^ k0;
        uint32_t n1 = lo1;
        uint32_t n2 = hi0 ^ c3 ^ k1;
        uint32_t n3 = lo0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
        k0 += ORC_PHILOX_W0;
        k1 += ORC_PHILOX_W1;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* Counter layout used by the sampler (a reading: the pages only say the   */
/* sample is multinomial and the renoise uniform).  key = (seed lo, hi);   */
/* counter = (lane, row, step, stream): stream 0 = Gumbel noise, word v&3  */
/* of lane v>>2 belongs to vocabulary entry v; stream 1 = renoise and      */
/* stream 2 = canvas initialisation, word 0 of lane 0.                     */
static uint32_t orc_philox_word(uint64_t seed, uint32_t lane, uint32_t row, uint32_t step,
                                uint32_t stream, int word)
{
    uint32_t ctr[4] = {lane, row, step, stream};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t out[4];
    orc_philox4x32_10(ctr, key, out);
    return out[word];
}

uint32_t orc_gumbel_bits(uint64_t seed, uint32_t row, uint32_t step, uint32_t v)
{
    return orc_philox_word(seed, v >> 2, row, step, 0u, (int)(v & 3u));
}

/* Uniform token in [0, V): multiply-shift of one 32-bit word. */
static int32_t orc_token_from_word(uint32_t x, int32_t V)
{
    return (int32_t)(((uint64_t)x * (uint64_t)(uint32_t)V) >> 32);
}

int32_t orc_renoise_token(uint64_t seed, uint32_t row, uint32_t step, int32_t V)
{
    return orc_token_from_word(orc_philox_word(seed, 0u, row, step, 1u, 0), V);
}

/* [Lab] item 1: the canvas starts as uniform random tokens, not [MASK]. */
int32_t orc_init_token(uint64_t seed, uint32_t row, int32_t V)
{
    return orc_token_from_word(orc_philox_word(seed, 0u, row, 0u, 2u, 0), V);
}

void orc_init_canvas(int32_t *canvas, int32_t n, int32_t V, uint64_t seed)
{
    for (int32_t r = 0; r < n; ++r) canvas[r] = orc_init_token(seed, (uint32_t)r, V);
}

/* ------------------------------------------------------------------ */
/* fp32 natural logarithm as a fixed sequence of IEEE operations.      */
/* x = 2^e * m with m in [sqrt(1/2), sqrt(2)); f = m - 1 (exact);      */
/* ln(1+f) = 2 atanh(s), s = f/(2+f), by the series                    */
/* 2s (1 + s^2/3 + s^4/5 + ... + s^10/11); then + e*ln2 with ln2 split */
/* into a short high part (exact products) and a low correction.       */
/* Valid for positive normal x.                                          */
/* ------------------------------------------------------------------ */
static float orc_bits_to_float(uint32_t b) { float f; memcpy(&f, &b, 4); return f; }
static uint32_t orc_float_to_bits(float f) { uint32_t b; memcpy(&b, &f, 4); return b; }

float orc_logf(float x)
{
    uint32_t bits = orc_float_to_bits(x);
    int32_t e = (int32_t)(bits >> 23) - 127;
    uint32_t mb = (bits & 0x007FFFFFu) | 0x3F800000u;   /* m in [1, 2) */
    if (mb > 0x3FB504F3u) {                              /* m > sqrt(2): use m/2 */
        mb -= 0x00800000u;
        e += 1;
    }
    float m = orc_bits_to_float(mb);
    float f = m - 1.0f;
    float s = f / (2.0f + f);
    float w = s * s;
    float p = 1.0f / 11.0f;
    p = fmaf(p, w, 1.0f / 9.0f);
    p = fmaf(p, w, 1.0f / 7.0f);
    p = fmaf(p, w, 1.0f / 5.0f);
    p = fmaf(p, w, 1.0f / 3.0f);
    float t = s + s;
    float tw = t * w;
    float r = fmaf(tw, p, t);
    float ef = (float)e;
    const float ln2_hi = 0.693145751953125f;          /* 0x3F317200 */
    const float ln2_lo = 1.428606765330187e-06f;      /* ln2 - ln2_hi */
    return fmaf(ef, ln2_hi, fmaf(ef, ln2_lo, r));
}

/* u = ((x >> 9) + 1/2) * 2^-23, in (0, 1), exact in fp32. */
float orc_uniform_open(uint32_t x)
{
    float hi = (float)(x >> 9);
    return (hi + 0.5f) * 1.1920928955078125e-07f;
}

/* Standard Gumbel variate G = -ln(-ln u). */
float orc_gumbel_from_bits(uint32_t x)
{
    float u = orc_uniform_open(x);
    float e1 = -orc_logf(u);
    return -orc_logf(e1);
}

/* ------------------------------------------------------------------ */
/* Per-position sampler of one row of logits.                           */
/* [Lab] item 2 / [PD] "Entropy-bounded acceptance": the ranking key is */
/* the entropy (nats) of the sampling distribution softmax(logit / T).  */
/* [Lab] item 5: the multinomial sample decides what is committed, the  */
/* argmax canvas is the output.  The sample is drawn by Gumbel-max:     */
/* argmax_v fp32(fmaf(logit_v, invT, G_v)), invT = fp32(1/T), ties to    */
/* the lowest v.  The fp64 logits are rounded to fp32 for the score     */
/* only; entropy and argmax use them as given.                          */
/* ------------------------------------------------------------------ */
void orc_sampler_row(const double *logits, int32_t V, double T, uint64_t seed,
                     uint32_t row, uint32_t step,
                     double *H_out, int32_t *sample_out, int32_t *argmax_out,
                     double *gumbel_margin_out, double *argmax_margin_out)
{
    /* entropy of softmax(logits / T), fp64 */
    double zmax = -INFINITY;
    for (int32_t v = 0; v < V; ++v) {
        double z = logits[v] / T;
        if (z > zmax) zmax = z;
    }
    double S = 0.0, A = 0.0;
    for (int32_t v = 0; v < V; ++v) {
        double d = logits[v] / T - zmax;
        double e = exp(d);
        S += e;
        A += e * d;
    }
    *H_out = log(S) - A / S;

    /* plain argmax, ties -> lowest index; margin to the runner-up */
    int32_t am = 0;
    double best = logits[0];
    for (int32_t v = 1; v < V; ++v)
        if (logits[v] > best) { best = logits[v]; am = v; }
    double second = -INFINITY;
    for (int32_t v = 0; v < V; ++v)
        if (v != am && logits[v] > second) second = logits[v];
    *argmax_out = am;
    *argmax_margin_out = (V > 1) ? best - second : INFINITY;

    /* Gumbel-max sample in the fp32 score */
    float invT = (float)(1.0 / T);
    int32_t smp = 0;
    float sbest = -INFINITY;
    double s1 = -INFINITY, s2 = -INFINITY;
    for (int32_t v = 0; v < V; ++v) {
        float g = orc_gumbel_from_bits(orc_gumbel_bits(seed, row, step, (uint32_t)v));
        float sc = fmaf((float)logits[v], invT, g);
        if (sc > sbest) { sbest = sc; smp = v; }
        double scd = (double)sc;
        if (scd > s1) { s2 = s1; s1 = scd; }
        else if (scd > s2) { s2 = scd; }
    }
    *sample_out = smp;
    *gumbel_margin_out = (V > 1) ? s1 - s2 : INFINITY;
}

/* ------------------------------------------------------------------ */
/* Entropy-bounded acceptance + uniform renoise of one canvas.          */
/* [Lab] item 2: sort positions by entropy ascending, commit the        */
/* largest prefix with cumsum(H) - max(H) <= b; at least one commits.   */
/* Reading: max(H) is the prefix maximum, i.e. the last sorted entry,   */
/* so the test on a prefix of length k is sum_{j<k} H_(j) <= b, with    */
/* the sum taken in fp64 in sorted order.  Ties in H go to the lower    */
/* position.  [PD] "Entropy-bounded acceptance": the rest is renoised   */
/* uniformly over the vocabulary.  Accepted positions take the sampled  */
/* token ([Lab] item 5).                                                */
/* ------------------------------------------------------------------ */
static const float *orc_sort_keys;
static int orc_cmp_pos(const void *pa, const void *pb)
{
    int32_t a = *(const int32_t *)pa, b = *(const int32_t *)pb;
    float ha = orc_sort_keys[a], hb = orc_sort_keys[b];
    if (ha < hb) return -1;
    if (ha > hb) return 1;
    return (a > b) - (a < b);
}

int32_t orc_accept_renoise(const float *H, const int32_t *sample, int32_t *canvas,
                           uint8_t *accepted, int32_t L, int32_t V, double b,
                           uint64_t seed, uint32_t row_base, uint32_t step,
                           int32_t *order_out, double *boundary_gap_out)
{
    int32_t *order = (int32_t *)malloc(sizeof(int32_t) * (size_t)L);
    for (int32_t i = 0; i < L; ++i) order[i] = i;
    orc_sort_keys = H;
    qsort(order, (size_t)L, sizeof(int32_t), orc_cmp_pos);

    /* k* = max { k in [1, L] : sum_{j<k} H_(j) <= b } */
    int32_t kstar = 0;
    double run = 0.0;                 /* sum of the first k-1 sorted entries */
    double gap = INFINITY;
    for (int32_t k = 1; k <= L; ++k) {
        if (k > 1) run += (double)H[order[k - 2]];
        double d = fabs(run - b);
        if (k > 1 && d < gap) gap = d;
        if (run <= b) kstar = k;
    }
    if (kstar < 1) kstar = 1;         /* b < 0 only; the rule always commits one */

    for (int32_t rank = 0; rank < L; ++rank) {
        int32_t i = order[rank];
        if (rank < kstar) {
            canvas[i] = sample[i];
            accepted[i] = 1;
        } else {
            canvas[i] = orc_renoise_token(seed, row_base + (uint32_t)i, step, V);
            accepted[i] = 0;
        }
    }
    if (order_out) memcpy(order_out, order, sizeof(int32_t) * (size_t)L);
    if (boundary_gap_out) *boundary_gap_out = gap;
    free(order);
    return kstar;
}

/* ------------------------------------------------------------------ */
/* Adaptive stop. [Lab] item 3: argmax canvas unchanged from the        */
/* previous step AND mean entropy < threshold (0.005).  Step 0 has no   */
/* previous step and never stops.  Mean in fp64, sequential.            */
/* ------------------------------------------------------------------ */
int32_t orc_stop(const int32_t *argmax, const int32_t *prev_argmax, const float *H,
                 int32_t L, int32_t step, double threshold, double *mean_out)
{
    double sum = 0.0;
    for (int32_t i = 0; i < L; ++i) sum += (double)H[i];
    double mean = sum / (double)L;
    if (mean_out) *mean_out = mean;
    if (step < 1) return 0;
    for (int32_t i = 0; i < L; ++i)
        if (argmax[i] != prev_argmax[i]) return 0;
    return mean < threshold ? 1 : 0;
}

/* [Lab] item 4 / [PD] "Temperature annealing": linear 0.8 -> 0.4 across */
/* the N steps; step k of N uses t0 + (t1 - t0) * k / (N - 1).            */
double orc_temperature(int32_t k, int32_t N, double t0, double t1)
{
    if (N <= 1) return t0;
    return t0 + (t1 - t0) * (double)k / (double)(N - 1);
}

/* ------------------------------------------------------------------ */
/* Canvas attention [Lab] item 6, [PD] "Finding": the decoder attends   */
/* bidirectionally across the canvas (no mask) and to the cached        */
/* context.  For query row (b, i, h): keys are the P cached rows then   */
/* the L canvas rows of kv head g = h / (Hq/Hkv);                       */
/* O = softmax(scale * q K^T) V.  bf16 inputs, fp64 arithmetic.          */
/* Layouts: q, out [B, L, Hq, D]; kp, vp [B, P, Hkv, D];                 */
/* kc, vc [B, L, Hkv, D].  rows[] lists flat query rows (b*L+i)*Hq+h.    */
/* ------------------------------------------------------------------ */
static double orc_bf16(uint16_t h)
{
    uint32_t b = (uint32_t)h << 16;
    return (double)orc_bits_to_float(b);
}

/* With causal != 0 (the encoder's cache-append forward, "Parallel Denoising
   From an Autoregressive Checkpoint", section "Finding": the causal encoder
   extends the append-only cache with the committed block), the query at
   canvas position i sees the P cached keys and the canvas keys 0 .. i only. */
void orc_attention_rows_ex(const uint16_t *q, const uint16_t *kp, const uint16_t *vp,
                           const uint16_t *kc, const uint16_t *vc,
                           int32_t B, int32_t L, int32_t P, int32_t Hq, int32_t Hkv, int32_t D,
                           double scale, int32_t causal, const int64_t *rows, int64_t nrows,
                           double *out)
{
    int32_t group = Hq / Hkv;
    int64_t nk_all = (int64_t)P + L;
    double *s = (double *)malloc(sizeof(double) * (size_t)(nk_all > 0 ? nk_all : 1));
    (void)B;
    for (int64_t t = 0; t < nrows; ++t) {
        int64_t flat = rows[t];
        int64_t h = flat % Hq;
        int64_t bi = flat / Hq;            /* b*L + i */
        int64_t b = bi / L;
        int64_t i = bi % L;
        int64_t g = h / group;
        int64_t nk = causal ? (int64_t)P + i + 1 : nk_all;
        const uint16_t *qr = q + flat * D;
        double smax = -INFINITY;
        for (int64_t j = 0; j < nk; ++j) {
            const uint16_t *kr = (j < P) ? kp + ((b * P + j) * Hkv + g) * D
                                         : kc + ((b * L + (j - P)) * Hkv + g) * D;
            double acc = 0.0;
            for (int32_t d = 0; d < D; ++d) acc += orc_bf16(qr[d]) * orc_bf16(kr[d]);
            s[j] = scale * acc;
            if (s[j] > smax) smax = s[j];
        }
        double den = 0.0;
        for (int64_t j = 0; j < nk; ++j) { s[j] = exp(s[j] - smax); den += s[j]; }
        double *o = out + t * D;
        for (int32_t d = 0; d < D; ++d) o[d] = 0.0;
        for (int64_t j = 0; j < nk; ++j) {
            const uint16_t *vr = (j < P) ? vp + ((b * P + j) * Hkv + g) * D
                                         : vc + ((b * L + (j - P)) * Hkv + g) * D;
            double p = s[j] / den;
            for (int32_t d = 0; d < D; ++d) o[d] += p * orc_bf16(vr[d]);
        }
    }
    free(s);
}

void orc_attention_rows(const uint16_t *q, const uint16_t *kp, const uint16_t *vp,
                        const uint16_t *kc, const uint16_t *vc,
                        int32_t B, int32_t L, int32_t P, int32_t Hq, int32_t Hkv, int32_t D,
                        double scale, const int64_t *rows, int64_t nrows, double *out)
{
    orc_attention_rows_ex(q, kp, vp, kc, vc, B, L, P, Hq, Hkv, D, scale, 0, rows, nrows, out);
}

/* Gumbel variates of vocabulary entries v0 .. v0+n-1 of one (row, step). */
void orc_gumbel_fill(uint64_t seed, uint32_t row, uint32_t step, uint32_t v0, int32_t n, float *out)
{
    for (int32_t t = 0; t < n; ++t)
        out[t] = orc_gumbel_from_bits(orc_gumbel_bits(seed, row, step, v0 + (uint32_t)t));
}

/* ---------------------------------------------------------------------------
 * FP8 (E4M3) weight and hidden-state streams for the LM head.  The pages
 * quote their H100 throughput for an FP8 model ("DiffusionGemma Lab",
 * section 1; "Parallel Denoising From an Autoregressive Checkpoint", section
 * "Finding"); the format is OCP FP8 E4M3: 1 sign, 4 exponent (bias 7), 3
 * mantissa bits, no infinities, 0x7F / 0xFF NaN, largest finite 448.
 * Quantisation of a row of n values x (bf16): amax = max |x|; if amax == 0
 * every code is 0 and the scale 1, else inv = fp32(448 / amax), scale =
 * fp32(amax / 448), code_j = E4M3 nearest-even of fp32(x_j * inv), saturated
 * to +-448.  The row then stands for decode(code_j) * scale.
 * ------------------------------------------------------------------------- */
double orc_e4m3_decode(uint8_t c)
{
    const int s = c >> 7, e = (c >> 3) & 0xF, m = c & 7;
    double v;
    if (e == 0xF && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);                 /* subnormal: m/8 * 2^-6 */
    else v = ldexp(8.0 + m, e - 10);                     /* (1 + m/8) * 2^(e-7) */
    return s ? -v : v;
}

uint8_t orc_e4m3_encode(float x)
{
    /* nearest of the 127 non-negative finite codes to |x| (ties: even code),
       saturating at 448; a plain search over the code table */
    const uint8_t sign = (signbit(x) ? 0x80 : 0x00);
    double a = fabs((double)x);
    if (isnan(x)) return 0x7F;
    if (a > 448.0) a = 448.0;
    static double table[0x7F];           /* decoded non-negative codes, filled once */
    static int have_table = 0;
    if (!have_table) {
        for (int c = 0; c <= 0x7E; ++c) table[c] = orc_e4m3_decode((uint8_t)c);
        have_table = 1;
    }
    uint8_t best = 0;
    double bd = INFINITY;
    for (int c = 0; c <= 0x7E; ++c) {
        const double d = fabs(table[c] - a);
        if (d < bd || (d == bd && (c & 1) == 0)) {
            bd = d;
            best = (uint8_t)c;
        }
    }
    return (uint8_t)(best | sign);
}

void orc_quantize_rows_e4m3(const uint16_t *x, int64_t rows, int64_t cols, uint8_t *q, float *scale)
{
    for (int64_t r = 0; r < rows; ++r) {
        const uint16_t *xr = x + r * cols;
        float amax = 0.0f;
        for (int64_t j = 0; j < cols; ++j) {
            const float v = fabsf((float)orc_bf16(xr[j]));
            if (v > amax) amax = v;
        }
        if (amax == 0.0f) {
            scale[r] = 1.0f;
            for (int64_t j = 0; j < cols; ++j) q[r * cols + j] = 0;
            continue;
        }
        const float inv = 448.0f / amax;
        scale[r] = amax / 448.0f;
        for (int64_t j = 0; j < cols; ++j) {
            const float v = (float)orc_bf16(xr[j]) * inv;
            q[r * cols + j] = orc_e4m3_encode(v);
        }
    }
}

/* ------------------------------------------------------------------ */
/* Self-conditioning read-out of one canvas row.                        */
/* [PD] "Finding", architecture paragraph: a small self-conditioning    */
/* block (7.8M parameters) feeds the previous step's prediction back    */
/* into the model; the hardware paragraph places its matmul, in full    */
/* precision, in the sampling stage next to the full-vocabulary softmax.*/
/* Reading: the fed-back prediction is the expected embedding under the */
/* step's sampling distribution,                                        */
/*   sc[j] = sum_v softmax(logits / T)_v E[v, j],   j < R,              */
/* with a table E [V, R] (V R = 262144 x 30 = 7.86M at the full vocab-  */
/* ulary).  fp64 throughout: the softmax weights exp(z_v - zmax) / S    */
/* with z = logits / T, then the weighted sum over v in order.          */
/* ------------------------------------------------------------------ */
void orc_self_cond_row(const double *logits, int32_t V, double T, const float *E, int32_t R,
                       double *sc_out)
{
    double zmax = -INFINITY;
    for (int32_t v = 0; v < V; ++v) {
        double z = logits[v] / T;
        if (z > zmax) zmax = z;
    }
    double S = 0.0;
    for (int32_t j = 0; j < R; ++j) sc_out[j] = 0.0;
    for (int32_t v = 0; v < V; ++v) {
        double e = exp(logits[v] / T - zmax);
        S += e;
        for (int32_t j = 0; j < R; ++j) sc_out[j] += e * (double)E[(int64_t)v * R + j];
    }
    for (int32_t j = 0; j < R; ++j) sc_out[j] /= S;
}

/* ------------------------------------------------------------------ */
/* Round to the nearest bf16 (8 significant bits), ties to even: the   */
/* bf16 value a model stores for an activation computed in higher     */
/* precision.  Returns the bit pattern.  Finite normal inputs within   */
/* the bf16 range (the activations here); +-0 maps to +-0.             */
/* ------------------------------------------------------------------ */
uint16_t orc_round_bf16(double x)
{
    if (x == 0.0) return signbit(x) ? 0x8000u : 0u;
    const int neg = x < 0.0;
    double a = fabs(x);
    int e;
    (void)frexp(a, &e);                 /* a = f 2^e, f in [0.5, 1) */
    /* 8 significant bits: the unit in the last place is 2^(e - 8) */
    double q = ldexp(a, 8 - e);         /* in [128, 256) */
    double fl = floor(q);
    double rem = q - fl;
    if (rem > 0.5 || (rem == 0.5 && fmod(fl, 2.0) != 0.0)) fl += 1.0;
    double r = ldexp(fl, e - 8);
    float rf = (float)r;                /* exact: 8 significant bits */
    uint32_t b = orc_float_to_bits(rf);
    uint16_t h = (uint16_t)(b >> 16);
    if (neg) h |= 0x8000u;
    return h;
}
