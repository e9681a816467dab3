/*
 * pti_oracle.c -- plain fp64 CPU oracle for the Packed Twin Inference hot path.
 *
 * TEST INFRASTRUCTURE ONLY (see pti_oracle.h).  Written for clarity, not speed:
 * every result is the plain definition evaluated with straight loops in
 * double precision.  No blocking, no reordering, no fusion.
 */
#include "pti_oracle.h"

/* The row (and verify-step) loops carry "#pragma omp parallel for": built
 * with -fopenmp (the CPU-baseline timing of the benchmark) the rows are split
 * over the host's cores, each row still computed by the same loop; built
 * without it (the tests) the pragmas are ignored.  Rows are independent, so
 * the results are identical either way. */
#include <math.h>
#include <stddef.h>
#include <stdlib.h>

/* ---------------------------------------------------------------------------
 * IEEE-754 binary16 decode, written from the format definition: 1 sign bit,
 * 5 exponent bits (bias 15), 10 fraction bits; exponent 0 holds zero and the
 * subnormals (fraction * 2^-24), exponent 31 holds inf and NaN.
 * The pages store every block scale as "f16" ([PTI-forum] §"PTI的核心创新：
 * SSQ打包技术": "[scale_A f16][scale_B f16][32 × uint16]").
 * ------------------------------------------------------------------------- */
double pti_or_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int exponent = (h >> 10) & 0x1F;
    int fraction = h & 0x3FF;
    double magnitude;

    if (exponent == 0) {
        magnitude = ldexp((double)fraction, -24);
    } else if (exponent == 31) {
        magnitude = (fraction == 0) ? INFINITY : NAN;
    } else {
        magnitude = ldexp(1.0 + (double)fraction / 1024.0, exponent - 15);
    }
    return sign ? -magnitude : magnitude;
}

static uint16_t read_u16_le(const uint8_t *p)
{
    return (uint16_t)((uint16_t)p[0] | ((uint16_t)p[1] << 8));
}

static int as_int8(uint8_t byte)
{
    /* two's-complement reinterpretation without relying on char signedness */
    return byte < 128 ? (int)byte : (int)byte - 256;
}

/* ---------------------------------------------------------------------------
 * Q8 block: f16 scale followed by 32 int8 values; weight = scale * q.
 * The symmetric (zero-point 0) case of the affine quantisation in [CS336-L10]
 * §"7.1 量化的机制"; the 34-byte size is half of the 68-byte twin block, which
 * [PTI-forum] §"PTI的核心创新：SSQ打包技术" says holds the same bytes as two
 * independent Q8 blocks.
 * ------------------------------------------------------------------------- */
double pti_or_q8_weight(const uint8_t *w, int64_t cols, int64_t row, int64_t col)
{
    int64_t blocks_per_row = cols / PTI_OR_BLOCK_COLS;
    int64_t block = row * blocks_per_row + col / PTI_OR_BLOCK_COLS;
    const uint8_t *blk = w + block * PTI_OR_Q8_BLOCK_BYTES;
    double scale = pti_or_f16_to_f64(read_u16_le(blk));
    int i = (int)(col % PTI_OR_BLOCK_COLS);
    return scale * (double)as_int8(blk[2 + i]);
}

/* ---------------------------------------------------------------------------
 * Twin block: "[scale_A f16][scale_B f16][32 × uint16]" with model A in the
 * high byte and model B in the low byte of each uint16 ([PTI-forum]
 * §"PTI的核心创新：SSQ打包技术"); unpacked as wa = (int8)(pw >> 8),
 * wb = (int8)(pw & 0xFF), each multiplied by its own scale ([PTI-readme]
 * §"与 SSQ（Side-by-Side Quantization）的关系").
 * ------------------------------------------------------------------------- */
void pti_or_twin_weight(const uint8_t *w, int64_t cols, int64_t row, int64_t col,
                        double *wa, double *wb)
{
    int64_t blocks_per_row = cols / PTI_OR_BLOCK_COLS;
    int64_t block = row * blocks_per_row + col / PTI_OR_BLOCK_COLS;
    const uint8_t *blk = w + block * PTI_OR_TWIN_BLOCK_BYTES;
    double scale_a = pti_or_f16_to_f64(read_u16_le(blk));
    double scale_b = pti_or_f16_to_f64(read_u16_le(blk + 2));
    int i = (int)(col % PTI_OR_BLOCK_COLS);
    uint16_t pw = read_u16_le(blk + 4 + 2 * i);
    uint8_t hi = (uint8_t)(pw >> 8);
    uint8_t lo = (uint8_t)(pw & 0xFF);
    *wa = scale_a * (double)as_int8(hi);
    *wb = scale_b * (double)as_int8(lo);
}

/* ---------------------------------------------------------------------------
 * SSQ pack / unpack ([PTI-forum] §"技术实现架构": the ssq/ package packs,
 * unpacks and converts weights).  Pack puts model A's scale first, model B's
 * second, then for each of the 32 positions the uint16 (qA << 8) | qB.
 * ------------------------------------------------------------------------- */
int pti_or_twin_pack(const uint8_t *qa, const uint8_t *qb, int64_t n_blocks, uint8_t *twin)
{
    int64_t b;
    int i;
    if (qa == NULL || qb == NULL || twin == NULL || n_blocks < 0)
        return -1;
    for (b = 0; b < n_blocks; ++b) {
        const uint8_t *a = qa + b * PTI_OR_Q8_BLOCK_BYTES;
        const uint8_t *bb = qb + b * PTI_OR_Q8_BLOCK_BYTES;
        uint8_t *t = twin + b * PTI_OR_TWIN_BLOCK_BYTES;
        uint16_t scale_a = read_u16_le(a);
        uint16_t scale_b = read_u16_le(bb);
        t[0] = (uint8_t)(scale_a & 0xFF);
        t[1] = (uint8_t)(scale_a >> 8);
        t[2] = (uint8_t)(scale_b & 0xFF);
        t[3] = (uint8_t)(scale_b >> 8);
        for (i = 0; i < PTI_OR_BLOCK_COLS; ++i) {
            uint16_t pw = (uint16_t)(((uint16_t)a[2 + i] << 8) | (uint16_t)bb[2 + i]);
            t[4 + 2 * i] = (uint8_t)(pw & 0xFF);
            t[5 + 2 * i] = (uint8_t)(pw >> 8);
        }
    }
    return 0;
}

int pti_or_twin_unpack(const uint8_t *twin, int64_t n_blocks, uint8_t *qa, uint8_t *qb)
{
    int64_t b;
    int i;
    if (qa == NULL || qb == NULL || twin == NULL || n_blocks < 0)
        return -1;
    for (b = 0; b < n_blocks; ++b) {
        const uint8_t *t = twin + b * PTI_OR_TWIN_BLOCK_BYTES;
        uint8_t *a = qa + b * PTI_OR_Q8_BLOCK_BYTES;
        uint8_t *bb = qb + b * PTI_OR_Q8_BLOCK_BYTES;
        uint16_t scale_a = read_u16_le(t);
        uint16_t scale_b = read_u16_le(t + 2);
        a[0] = (uint8_t)(scale_a & 0xFF);
        a[1] = (uint8_t)(scale_a >> 8);
        bb[0] = (uint8_t)(scale_b & 0xFF);
        bb[1] = (uint8_t)(scale_b >> 8);
        for (i = 0; i < PTI_OR_BLOCK_COLS; ++i) {
            uint16_t pw = read_u16_le(t + 4 + 2 * i);
            a[2 + i] = (uint8_t)(pw >> 8);
            bb[2 + i] = (uint8_t)(pw & 0xFF);
        }
    }
    return 0;
}

static int shape_ok(int64_t rows, int64_t cols)
{
    return rows >= 1 && cols >= PTI_OR_BLOCK_COLS && cols % PTI_OR_BLOCK_COLS == 0;
}

/* ---------------------------------------------------------------------------
 * N-stream Q8 GEMV: y_s = W x_s for every stream s, one pass over W serving
 * all streams ([PTI-readme] §"带宽分析：为什么会有开销", the multi-stream kernel
 * that loads each weight group once and forms the N dot products together).
 * The oracle evaluates the definition row by row: dequantise each weight,
 * multiply by the activation, add, in double.
 * ------------------------------------------------------------------------- */
int pti_or_q8_gemv_rows(const uint8_t *w, int64_t rows, int64_t cols, int n,
                        const float *x, const int64_t *rows_idx, int64_t n_idx,
                        double *y, double *bound)
{
    int64_t j, k;
    int s;
    if (w == NULL || x == NULL || rows_idx == NULL || y == NULL || bound == NULL)
        return -1;
    if (!shape_ok(rows, cols) || n < 1 || n_idx < 0)
        return -1;
    for (j = 0; j < n_idx; ++j)
        if (rows_idx[j] < 0 || rows_idx[j] >= rows)
            return -1;

    for (s = 0; s < n; ++s) {
        const float *xs = x + (int64_t)s * cols;
#pragma omp parallel for private(k) schedule(static)
        for (j = 0; j < n_idx; ++j) {
            double acc = 0.0, mag = 0.0;
            for (k = 0; k < cols; ++k) {
                double term = pti_or_q8_weight(w, cols, rows_idx[j], k) * (double)xs[k];
                acc += term;
                mag += fabs(term);
            }
            y[(int64_t)s * n_idx + j] = acc;
            bound[(int64_t)s * n_idx + j] = mag;
        }
    }
    return 0;
}

/* ---------------------------------------------------------------------------
 * SSQ twin GEMV ([PTI-readme] §"与 SSQ（Side-by-Side Quantization）的关系";
 * [PTI-forum] §"PTI的核心创新：SSQ打包技术"): y_a[r] is the dot product of model
 * A's dequantised row (the upper bytes of the packed 16-bit elements times A's
 * block scales) with x_a, y_b[r] that of model B's row (the lower bytes times
 * B's scales) with x_b; both come from one read of the packed matrix.
 * ------------------------------------------------------------------------- */
int pti_or_twin_gemv_rows(const uint8_t *w, int64_t rows, int64_t cols,
                          const float *xa, const float *xb,
                          const int64_t *rows_idx, int64_t n_idx,
                          double *ya, double *yb, double *bound_a, double *bound_b)
{
    int64_t j, k;
    if (w == NULL || xa == NULL || xb == NULL || rows_idx == NULL || ya == NULL ||
        yb == NULL || bound_a == NULL || bound_b == NULL)
        return -1;
    if (!shape_ok(rows, cols) || n_idx < 0)
        return -1;
    for (j = 0; j < n_idx; ++j)
        if (rows_idx[j] < 0 || rows_idx[j] >= rows)
            return -1;

#pragma omp parallel for private(k) schedule(static)
    for (j = 0; j < n_idx; ++j) {
        double acc_a = 0.0, acc_b = 0.0, mag_a = 0.0, mag_b = 0.0;
        for (k = 0; k < cols; ++k) {
            double wa, wb, ta, tb;
            pti_or_twin_weight(w, cols, rows_idx[j], k, &wa, &wb);
            ta = wa * (double)xa[k];
            tb = wb * (double)xb[k];
            acc_a += ta;
            acc_b += tb;
            mag_a += fabs(ta);
            mag_b += fabs(tb);
        }
        ya[j] = acc_a;
        yb[j] = acc_b;
        bound_a[j] = mag_a;
        bound_b[j] = mag_b;
    }
    return 0;
}

/* ---------------------------------------------------------------------------
 * Greedy verify ([PTI-readme] §"接受机制如何工作"; [PTI-forum] §"技术实现架构",
 * step 3 "验证").  Stream 0 runs on the confirmed token, stream s on the guess
 * for position n+s.  Under greedy decoding the output of stream s is its
 * argmax; the guess fed to stream s+1 is accepted when it equals that argmax,
 * and acceptance stops at the first mismatch, so a step emits 1 + accept
 * tokens.  Ties in the argmax go to the lowest index (a strictly-greater scan
 * from index 0).
 * ------------------------------------------------------------------------- */
int pti_or_verify_greedy(const float *logits, const int32_t *guess, int64_t steps, int n,
                         int64_t vocab, int32_t *argmax, uint8_t *match, int32_t *accept)
{
    int64_t t, v;
    int s;
    if (logits == NULL || guess == NULL || argmax == NULL || accept == NULL)
        return -1;
    if (steps < 0 || n < 1 || vocab < 1 || (n > 1 && match == NULL))
        return -1;

#pragma omp parallel for private(s, v) schedule(static)
    for (t = 0; t < steps; ++t) {
        int run = 1;
        int32_t accepted = 0;
        for (s = 0; s < n; ++s) {
            const float *row = logits + (t * n + s) * vocab;
            int64_t best = 0;
            for (v = 1; v < vocab; ++v)
                if (row[v] > row[best])
                    best = v;
            argmax[t * n + s] = (int32_t)best;
        }
        for (s = 0; s + 1 < n; ++s) {
            uint8_t m = (uint8_t)(guess[t * n + s + 1] == argmax[t * n + s]);
            match[t * (n - 1) + s] = m;
            if (run && m)
                ++accepted;
            else
                run = 0;
        }
        accept[t] = accepted;
    }
    return 0;
}

/* ---------------------------------------------------------------------------
 * Sampling-mode verify ([PTI-readme] §"接受机制如何工作", the temperature > 0
 * case): at temperature T each stream's output distribution is
 * p(v) = exp(l_v / T) / sum_u exp(l_u / T); the stream draws its token from p,
 * and the guess fed to stream s+1 is accepted when it equals stream s's draw.
 * Two independent draws from the same p agree with probability sum_v p(v)^2,
 * the collision probability the pages give as the acceptance rate.
 *
 * The draw is the inverse-CDF one for the supplied uniform number u in
 * [0, 1): the smallest v with p(0) + ... + p(v) > u.  (The random numbers are
 * inputs, so the draw is a plain function of them.)  The exponentials are
 * taken after subtracting the row maximum, which changes no ratio.
 * margin[t][s] = min(u - CDF(v - 1), CDF(v) - u) for the drawn v: how far u
 * lies from the edges of the drawn token's interval.
 * ------------------------------------------------------------------------- */
int pti_or_verify_sample(const float *logits, const int32_t *guess, const float *uniform,
                         int64_t steps, int n, int64_t vocab, double temperature,
                         int32_t *token, uint8_t *match, int32_t *accept, double *collision,
                         double *margin)
{
    int64_t t, v;
    int s;
    double *e;
    if (logits == NULL || guess == NULL || uniform == NULL || token == NULL || accept == NULL)
        return -1;
    if (steps < 0 || n < 1 || vocab < 1 || (n > 1 && match == NULL))
        return -1;
    if (!(temperature > 0.0) || !isfinite(temperature))
        return -1;
    e = (double *)malloc((size_t)vocab * sizeof(double));
    if (e == NULL)
        return -1;

    for (t = 0; t < steps; ++t) {
        int run = 1;
        int32_t accepted = 0;
        for (s = 0; s < n; ++s) {
            const float *row = logits + (t * n + s) * vocab;
            const double u = (double)uniform[t * n + s];
            double top = (double)row[0], total = 0.0, squares = 0.0, cum = 0.0, below = 0.0;
            int64_t drawn = -1;
            for (v = 1; v < vocab; ++v)
                if ((double)row[v] > top)
                    top = (double)row[v];
            for (v = 0; v < vocab; ++v) {
                e[v] = exp(((double)row[v] - top) / temperature);
                total += e[v];
                squares += e[v] * e[v];
            }
            for (v = 0; v < vocab; ++v) {
                below = cum;
                cum += e[v] / total;
                if (cum > u) {
                    drawn = v;
                    break;
                }
            }
            if (drawn < 0) {  /* u at or above the last rounded CDF value: the last token with mass */
                for (v = vocab - 1; v > 0 && e[v] == 0.0; --v) {
                }
                drawn = v;
                below = cum - e[v] / total;
            }
            token[t * n + s] = (int32_t)drawn;
            if (collision != NULL)
                collision[t * n + s] = squares / (total * total);
            if (margin != NULL) {
                const double hi = below + e[drawn] / total;
                margin[t * n + s] = (u - below < hi - u) ? u - below : hi - u;
            }
        }
        for (s = 0; s + 1 < n; ++s) {
            uint8_t m = (uint8_t)(guess[t * n + s + 1] == token[t * n + s]);
            match[t * (n - 1) + s] = m;
            if (run && m)
                ++accepted;
            else
                run = 0;
        }
        accept[t] = accepted;
    }
    free(e);
    return 0;
}

/* ---------------------------------------------------------------------------
 * One gated-MLP layer of the multi-stream decode weight pass.  The pages'
 * step loads every weight once for N tokens ([PTI-readme] §"工作原理");
 * the gated MLP (W_up, W_gate, W_down) is the one of [CS336-L10] §"2.4 MLP 层
 * 的算术强度".  The pages name no activation and no normalisation: this oracle
 * uses SiLU(g) * u and an RMS rescale v / sqrt(mean(v^2) + eps) after h and
 * after the down projection.
 * ------------------------------------------------------------------------- */
static void q8_matvec_f64(const uint8_t *w, int64_t rows, int64_t cols, const double *x, double *y)
{
    int64_t r, k;
#pragma omp parallel for private(k) schedule(static)
    for (r = 0; r < rows; ++r) {
        double acc = 0.0;
        for (k = 0; k < cols; ++k)
            acc += pti_or_q8_weight(w, cols, r, k) * x[k];
        y[r] = acc;
    }
}

static void rms_rescale_f64(double *v, int64_t len, double eps)
{
    int64_t i;
    double sum_sq = 0.0, inv;
    for (i = 0; i < len; ++i)
        sum_sq += v[i] * v[i];
    inv = 1.0 / sqrt(sum_sq / (double)len + eps);
    for (i = 0; i < len; ++i)
        v[i] *= inv;
}

int pti_or_mlp_layer(const uint8_t *wg, const uint8_t *wu, const uint8_t *wd,
                     int64_t hidden, int64_t ffn, int n, double eps,
                     const double *x_in, double *x_out, double *h_out)
{
    double *g, *u, *h;
    int64_t i;
    int s;
    if (wg == NULL || wu == NULL || wd == NULL || x_in == NULL || x_out == NULL)
        return -1;
    if (!shape_ok(ffn, hidden) || !shape_ok(hidden, ffn) || n < 1 || !(eps >= 0.0))
        return -1;

    g = (double *)malloc((size_t)ffn * sizeof(double));
    u = (double *)malloc((size_t)ffn * sizeof(double));
    h = (double *)malloc((size_t)ffn * sizeof(double));
    if (g == NULL || u == NULL || h == NULL) {
        free(g);
        free(u);
        free(h);
        return -1;
    }
    for (s = 0; s < n; ++s) {
        const double *xs = x_in + (int64_t)s * hidden;
        double *xo = x_out + (int64_t)s * hidden;
        q8_matvec_f64(wg, ffn, hidden, xs, g);
        q8_matvec_f64(wu, ffn, hidden, xs, u);
        for (i = 0; i < ffn; ++i)
            h[i] = g[i] / (1.0 + exp(-g[i])) * u[i];
        rms_rescale_f64(h, ffn, eps);
        if (h_out != NULL)
            for (i = 0; i < ffn; ++i)
                h_out[(int64_t)s * ffn + i] = h[i];
        q8_matvec_f64(wd, hidden, ffn, h, xo);
        rms_rescale_f64(xo, hidden, eps);
    }
    free(g);
    free(u);
    free(h);
    return 0;
}

/* ---------------------------------------------------------------------------
 * Greedy self-speculative decoding, [PTI-readme] §"接受机制如何工作" with the
 * state handling of [PTI-forum] §"技术实现架构" (see pti_oracle.h for the
 * reading).  The model is given by its greedy next-token table; one step is
 * one pass of every stream through the model.
 * ------------------------------------------------------------------------- */
int pti_or_selfspec_greedy(const int32_t *next, int64_t vocab, int n, int32_t first, int64_t steps,
                           int32_t *tokens, int64_t cap, int64_t *count, int32_t *accept)
{
    int32_t win[4], a[4];
    int64_t t, v, c = 0;
    int i, L;
    if (next == NULL || count == NULL || n < 1 || n > 4 || vocab < 1 || steps < 0 || cap < 0)
        return -1;
    if ((cap > 0 && tokens == NULL) || first < 0 || first >= vocab)
        return -1;
    for (v = 0; v < vocab; ++v)
        if (next[v] < 0 || next[v] >= vocab)
            return -1;
    for (i = 0; i < n; ++i)
        win[i] = first;
    for (t = 0; t < steps; ++t) {
        /* every stream runs the model on its window token */
        for (i = 0; i < n; ++i)
            a[i] = next[win[i]];
        /* stream i+1's input was a guess of what stream i produces */
        L = 0;
        while (L < n - 1 && win[L + 1] == a[L])
            ++L;
        /* a[0 .. L] are confirmed */
        for (i = 0; i <= L; ++i) {
            if (c < cap)
                tokens[c] = a[i];
            ++c;
        }
        if (accept != NULL)
            accept[t] = L;
        /* the next window starts at the newest confirmed token */
        for (i = 0; i < n; ++i)
            win[i] = a[(L + i < n) ? (L + i) : (n - 1)];
    }
    *count = c;
    return 0;
}
