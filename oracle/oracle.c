/*
 * oracle.c -- plain fp64 CPU reference of grouped-query causal attention
 * with rotary positions, q/k RMSNorm, a tanh logit softcap, a sliding
 * window and a key/value cache.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the package smoke check and the
 * benchmark's CPU-baseline leg load this library. The CUDA library never
 * calls it and shares no code, header or table with it.
 *
 * Every step is written straight from its definition, in double precision:
 * there is no tiling, no fusion and no online softmax. Sources (web pages,
 * cited by title and section):
 *   [mojo]  "mojolearn.transformer": TransformerBlock parameters (window,
 *           rope_theta, rope_scaling, rope_dim, qk_norm, attn_softcap,
 *           norm_eps), TransformerBlock.step, TransformerState.
 *   [dx]    "Core Layers -- Deep Reference": "RMSNorm", "RoPE (Rotary
 *           Positional Embedding)", "Multi-Head (MHA) and Grouped-Query
 *           Attention (GQA)", "Sliding window attention".
 *   [dew]   "dew.nn.backbones.causal_transformer": LayerKind.window,
 *           CausalTransformer (partial_rotary_factor, attention_scale).
 *
 * Readings taken where the pages are silent or disagree:
 *   - rotary pairs are "rotate half" (i, i + R/2), the Hugging Face Llama
 *     convention that [mojo] says it computes; [dx] prints interleaved pairs;
 *   - the window admits W keys, its own included ([mojo] window, [dew]
 *     LayerKind.window), not the W + 1 of [dx]'s printed mask;
 *   - the frequency exponent under partial rotary uses R, not D;
 *   - Llama-3 scaling follows the published Llama 3.1 frequency ramp, of
 *     which [mojo] names only the fields;
 *   - softcap c*tanh(s/c) acts on the scaled score, before masking;
 *   - the default scale is 1/sqrt(D), with D the full head dimension.
 *
 * The interior of the Llama-3 ramp (0 < s < 1 in orc_inv_freq) is pinned by
 * three frequencies of the Llama-3-8B-shaped workload worked by hand from the
 * published Llama 3.1 rule (tests/golden/llama3_ramp_interior.txt) and by
 * f'/f being affine in f there, besides both ends of the ramp.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

#ifndef M_PI
#define M_PI 3.14159265358979323846
#endif

typedef struct orc_cfg {
    int B, H, Hkv, L, D;
    int rope_dim;                 /* R rotary dims; 0 means no rotation */
    double theta;                 /* RoPE base */
    int scaling_type;             /* 0 none, 1 linear, 2 llama3 */
    double factor;
    double low_freq_factor;
    double high_freq_factor;
    double original_max_positions;
    double norm_eps;
    int window;                   /* 0 full causal, W > 0 sliding window */
    double softcap;               /* <= 0: off */
    double scale;                 /* <= 0: 1/sqrt(D) */
} orc_cfg;

int orc_num_threads(void)
{
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Rotary frequencies, [dx] "RoPE": theta_i = base^(-2i/d), here with d = R
 * (the rotary width). Linear scaling divides every frequency by the factor
 * ([mojo] rope_scaling "linear"). Llama-3 scaling ([mojo] rope_scaling
 * "llama3"): a frequency whose wavelength 2*pi/f is shorter than
 * orig/high_freq_factor is kept, one longer than orig/low_freq_factor is
 * divided by the factor, and in between the two are blended linearly in
 * s = (orig/wavelength - low) / (high - low).
 */
void orc_inv_freq(const orc_cfg* c, double* inv)
{
    int R = c->rope_dim;
    for (int i = 0; i < R / 2; ++i) {
        double f = pow(c->theta, -(2.0 * i) / (double)R);
        if (c->scaling_type == 1) {
            f = f / c->factor;
        } else if (c->scaling_type == 2) {
            double wavelength = 2.0 * M_PI / f;
            double short_wl = c->original_max_positions / c->high_freq_factor;
            double long_wl = c->original_max_positions / c->low_freq_factor;
            if (wavelength < short_wl) {
                /* high frequency: unchanged */
            } else if (wavelength > long_wl) {
                f = f / c->factor;
            } else {
                double s = (c->original_max_positions / wavelength - c->low_freq_factor) /
                           (c->high_freq_factor - c->low_freq_factor);
                f = (1.0 - s) * f / c->factor + s * f;
            }
        }
        inv[i] = f;
    }
}

/* [dx] "RMSNorm": y = x / sqrt(mean(x^2) + eps) * w, no bias. */
static void rmsnorm(const double* x, const double* w, int D, double eps, double* y)
{
    double ss = 0.0;
    for (int i = 0; i < D; ++i) ss += x[i] * x[i];
    double rms = sqrt(ss / D + eps);
    for (int i = 0; i < D; ++i) y[i] = x[i] / rms * w[i];
}

/*
 * Rotation of one head vector at absolute position p, [dx] "RoPE": pair
 * (a, b) turns by the angle p*theta_i into (a cos - b sin, a sin + b cos).
 * Pair i is (i, i + R/2); dims R..D-1 are left as they are.
 */
static void rope_vec(double* x, int R, const double* inv, long p)
{
    int half = R / 2;
    for (int i = 0; i < half; ++i) {
        double ang = (double)p * inv[i];
        double cs = cos(ang), sn = sin(ang);
        double a = x[i], b = x[i + half];
        x[i] = a * cs - b * sn;
        x[i + half] = a * sn + b * cs;
    }
}

/*
 * Normalise (if norm_w) then rotate every row of x [B, NH, L, D] at
 * position start[b] + l. q/k RMSNorm comes before RoPE ([mojo] qk_norm).
 */
void orc_rotate_rows(const orc_cfg* c, const double* x, int NH, const int* start,
                     const double* norm_w, double* y)
{
    int B = c->B, L = c->L, D = c->D, R = c->rope_dim;
    double* inv = (double*)malloc(sizeof(double) * (R > 0 ? R / 2 : 1));
    if (R > 0) orc_inv_freq(c, inv);
    long rows = (long)B * NH * L;
#pragma omp parallel for schedule(static)
    for (long r = 0; r < rows; ++r) {
        int b = (int)(r / ((long)NH * L));
        int l = (int)(r % L);
        const double* xr = x + r * D;
        double* yr = y + r * D;
        if (norm_w) rmsnorm(xr, norm_w, D, c->norm_eps, yr);
        else memcpy(yr, xr, sizeof(double) * D);
        if (R > 0) rope_vec(yr, R, inv, (long)start[b] + l);
    }
    free(inv);
}

static double attn_scale(const orc_cfg* c)
{
    return c->scale > 0.0 ? c->scale : 1.0 / sqrt((double)c->D);
}

/* Key position m is visible from query position p: causal, and inside the
 * window [p - W + 1, p] when W > 0 ([mojo] window). */
static int visible(long m, long p, int W)
{
    if (m > p) return 0;
    if (W > 0 && m < p - W + 1) return 0;
    return 1;
}

/*
 * softmax(q.k_m * scale, capped) over the visible keys, times v_m.
 * keys[j], vals[j] point at the rows of key position pos[j]; n entries.
 * Two passes in fp64: maximum, then exp-sum and weighted sum.
 */
static void attend(const orc_cfg* c, const double* q, const double* const* keys,
                   const double* const* vals, const long* pos, int n, long p, double* out,
                   double* scratch)
{
    int D = c->D;
    double sc = attn_scale(c);
    double mx = -INFINITY;
    for (int j = 0; j < n; ++j) {
        if (!visible(pos[j], p, c->window)) { scratch[j] = NAN; continue; }
        double s = 0.0;
        for (int d = 0; d < D; ++d) s += q[d] * keys[j][d];
        s *= sc;
        if (c->softcap > 0.0) s = c->softcap * tanh(s / c->softcap);
        scratch[j] = s;
        if (s > mx) mx = s;
    }
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    double den = 0.0;
    for (int j = 0; j < n; ++j) {
        if (!visible(pos[j], p, c->window)) continue;
        double w = exp(scratch[j] - mx);
        den += w;
        for (int d = 0; d < D; ++d) out[d] += w * vals[j][d];
    }
    for (int d = 0; d < D; ++d) out[d] /= den;
}

/*
 * One query row (b, h, l) of a prefill from an empty cache: the keys are the
 * chunk's own rows, at positions start[b] + l'. Query head h reads key/value
 * head h / G with G = H / Hkv ([dx] "MHA and GQA": contiguous groups of
 * n_heads // kv_heads query heads share one key/value head).
 */
static void prefill_row(const orc_cfg* c, const double* qr, const double* kr,
                        const double* v, const int* start, int b, int h, int l, double* out,
                        const double** kp, const double** vp, long* pos, double* scratch)
{
    int H = c->H, Hkv = c->Hkv, L = c->L, D = c->D;
    int G = H / Hkv, hk = h / G;
    long p = (long)start[b] + l;
    const double* q = qr + (((long)b * H + h) * L + l) * D;
    for (int j = 0; j < L; ++j) {
        long off = (((long)b * Hkv + hk) * L + j) * D;
        kp[j] = kr + off;
        vp[j] = v + off;
        pos[j] = (long)start[b] + j;
    }
    attend(c, q, kp, vp, pos, L, p, out, scratch);
}

/* Whole prefill: out [B, H, L, D] from rotated q [B, H, L, D], rotated k and
 * raw v [B, Hkv, L, D]. */
void orc_prefill(const orc_cfg* c, const double* qr, const double* kr, const double* v,
                 const int* start, double* out)
{
    int B = c->B, H = c->H, L = c->L, D = c->D;
    long rows = (long)B * H * L;
#pragma omp parallel
    {
        const double** kp = (const double**)malloc(sizeof(double*) * L);
        const double** vp = (const double**)malloc(sizeof(double*) * L);
        long* pos = (long*)malloc(sizeof(long) * L);
        double* scratch = (double*)malloc(sizeof(double) * L);
#pragma omp for schedule(dynamic, 16)
        for (long r = 0; r < rows; ++r) {
            int b = (int)(r / ((long)H * L));
            int h = (int)((r / L) % H);
            int l = (int)(r % L);
            prefill_row(c, qr, kr, v, start, b, h, l, out + r * D, kp, vp, pos, scratch);
        }
        free(kp); free(vp); free(pos); free(scratch);
    }
}

/* Selected rows of the same prefill: rows[3i..3i+2] = (b, h, l); out [n, D]. */
void orc_prefill_rows(const orc_cfg* c, const double* qr, const double* kr, const double* v,
                      const int* start, int n, const int* rows, double* out)
{
    int L = c->L, D = c->D;
#pragma omp parallel
    {
        const double** kp = (const double**)malloc(sizeof(double*) * L);
        const double** vp = (const double**)malloc(sizeof(double*) * L);
        long* pos = (long*)malloc(sizeof(long) * L);
        double* scratch = (double*)malloc(sizeof(double) * L);
#pragma omp for schedule(dynamic, 1)
        for (int i = 0; i < n; ++i)
            prefill_row(c, qr, kr, v, start, rows[3 * i], rows[3 * i + 1], rows[3 * i + 2],
                        out + (long)i * D, kp, vp, pos, scratch);
        free(kp); free(vp); free(pos); free(scratch);
    }
}

/* Cache slot of absolute position m: m itself, or m mod W in a ring of W
 * slots ([mojo] TransformerState, sliding window). */
static long slot_of(long m, int W)
{
    return W > 0 ? m % W : m;
}

/*
 * Cache append ([mojo] TransformerState; [dx] "Static KV-Cache": the new
 * rows go in at the current index). Rotated k and raw v of positions
 * start[b] + l are stored at their slot of caches [B, Hkv, capacity, D].
 * Under a ring, a later position overwrites an earlier one that maps to the
 * same slot, so only the last W positions of the chunk survive. written
 * [B, Hkv, capacity] receives the position stored in each slot (entries of
 * slots not written keep their value).
 */
void orc_append(const orc_cfg* c, const double* kr, const double* v, const int* start,
                int capacity, double* kc, double* vc, long* written)
{
    int B = c->B, Hkv = c->Hkv, L = c->L, D = c->D, W = c->window;
    for (int b = 0; b < B; ++b)
        for (int hk = 0; hk < Hkv; ++hk)
            for (int l = 0; l < L; ++l) {
                long m = (long)start[b] + l;
                long s = slot_of(m, W);
                long src = (((long)b * Hkv + hk) * L + l) * D;
                long dst = (((long)b * Hkv + hk) * capacity + s) * D;
                memcpy(kc + dst, kr + src, sizeof(double) * D);
                memcpy(vc + dst, v + src, sizeof(double) * D);
                written[((long)b * Hkv + hk) * capacity + s] = m;
            }
}

/*
 * Single-token decode ([mojo] TransformerBlock.step: forward with L = 1 at
 * position cached_tokens). Row b's query is at p = cache_len[b] - 1 (the
 * length counts the token just appended) and reads cache positions
 * max(0, p - W + 1) .. p, each from its slot. qr [B, H, D] is rotated;
 * caches are [B, Hkv, capacity, D]; out [B, H, D].
 */
void orc_decode(const orc_cfg* c, const double* qr, const double* kc, const double* vc,
                const int* cache_len, int capacity, double* out)
{
    int B = c->B, H = c->H, Hkv = c->Hkv, D = c->D, W = c->window;
    int G = H / Hkv;
    long rows = (long)B * H;
    long maxn = 0;
    for (int b = 0; b < B; ++b) if (cache_len[b] > maxn) maxn = cache_len[b];
#pragma omp parallel
    {
        const double** kp = (const double**)malloc(sizeof(double*) * (maxn + 1));
        const double** vp = (const double**)malloc(sizeof(double*) * (maxn + 1));
        long* pos = (long*)malloc(sizeof(long) * (maxn + 1));
        double* scratch = (double*)malloc(sizeof(double) * (maxn + 1));
#pragma omp for schedule(dynamic, 1)
        for (long r = 0; r < rows; ++r) {
            int b = (int)(r / H), h = (int)(r % H), hk = h / G;
            long p = (long)cache_len[b] - 1;
            long first = (W > 0 && p - W + 1 > 0) ? p - W + 1 : 0;
            int n = 0;
            for (long m = first; m <= p; ++m, ++n) {
                long off = (((long)b * Hkv + hk) * capacity + slot_of(m, W)) * D;
                kp[n] = kc + off;
                vp[n] = vc + off;
                pos[n] = m;
            }
            attend(c, qr + r * D, kp, vp, pos, n, p, out + r * D, scratch);
        }
        free(kp); free(vp); free(pos); free(scratch);
    }
}
