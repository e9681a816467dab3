/*
 * pti_oracle.h -- plain, slow CPU oracle for the Packed Twin Inference hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link or
 * call this library: only the test suite, the smoke check of the build entry
 * point and the CPU-baseline leg of the benchmark use it.  It shares no source
 * with the CUDA library (its own structs, its own binary16 decoder, its own
 * loops) and it never reads anything produced by the CUDA kernels.
 *
 * Arithmetic: every floating-point result is accumulated in double (fp64).
 * Each function states the passage of the source pages it follows; the pages
 * are cited by title and section:
 *
 *   [PTI-forum]  "Packed Twin Inference：无需草稿模型的推测解码新方案，实现2倍吞吐量提升"
 *   [PTI-readme] "打包双子推理（PTI）" (translation of the packed-twin-inference README)
 *   [CS336-L10]  "推理（Inference）" (CS336 lecture 10 notes)
 *
 * Data layouts (byte offsets, all little-endian):
 *
 *   Q8 block, 34 bytes, covers 32 consecutive columns of one row:
 *     [0..1]   scale d, IEEE-754 binary16
 *     [2..33]  q[0..31], two's-complement int8; weight(col 32b+i) = d * q[i]
 *
 *   SSQ "mode 16" twin block, 68 bytes, covers the same 32 columns of two
 *   models A and B ([PTI-forum] §"PTI的核心创新：SSQ打包技术"):
 *     [0..1]   scale_A (binary16)     [2..3]  scale_B (binary16)
 *     [4+2i .. 5+2i]  uint16 pw[i], i = 0..31, stored little-endian, with
 *              model A's int8 in the high byte and model B's int8 in the low
 *              byte ([PTI-readme] §"与 SSQ（Side-by-Side Quantization）的关系"):
 *              so qB[i] is byte 4+2i and qA[i] is byte 5+2i.
 *
 *   A matrix of R rows and K columns (K a multiple of 32) is R consecutive
 *   rows, each K/32 consecutive blocks in column order.
 *
 * Parity pins: every function here is pinned by CPU tests against closed
 * forms, library routines on special cases, invariants fixed by the pages and
 * brute force on tiny inputs (tests/test_oracle_pins.py).
 */
#ifndef PTI_ORACLE_H
#define PTI_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PTI_OR_Q8_BLOCK_BYTES 34
#define PTI_OR_TWIN_BLOCK_BYTES 68
#define PTI_OR_BLOCK_COLS 32

/* IEEE-754 binary16 bit pattern -> exact double (sign, 5-bit exponent with
 * bias 15, 10-bit fraction, subnormals).  Inf and NaN decode to the double
 * inf/NaN of the same sign. */
double pti_or_f16_to_f64(uint16_t h);

/* The weight at (row, col) of a Q8 matrix, as an exact double d*q. */
double pti_or_q8_weight(const uint8_t *w, int64_t cols, int64_t row, int64_t col);

/* The weights at (row, col) of both models of a twin matrix. */
void pti_or_twin_weight(const uint8_t *w, int64_t cols, int64_t row, int64_t col,
                        double *wa, double *wb);

/* SSQ pack: two Q8 block streams of the same shape (n_blocks blocks each) ->
 * one twin block stream.  Returns 0, or -1 if a pointer is NULL. */
int pti_or_twin_pack(const uint8_t *qa, const uint8_t *qb, int64_t n_blocks, uint8_t *twin);

/* SSQ unpack: the inverse of pti_or_twin_pack. */
int pti_or_twin_unpack(const uint8_t *twin, int64_t n_blocks, uint8_t *qa, uint8_t *qb);

/* N-stream Q8 GEMV on selected rows.
 *   w      [rows][cols/32] Q8 blocks
 *   x      [n][cols] float activations, stream-major
 *   rows_idx[n_idx] the rows to evaluate (each in [0, rows))
 *   y      [n][n_idx]  y[s][j] = sum_k W[rows_idx[j]][k] * x[s][k]      (fp64)
 *   bound  [n][n_idx]  sum_k |W[rows_idx[j]][k] * x[s][k]|                (fp64)
 * Returns 0, or -1 on a bad argument. */
int pti_or_q8_gemv_rows(const uint8_t *w, int64_t rows, int64_t cols, int n,
                        const float *x, const int64_t *rows_idx, int64_t n_idx,
                        double *y, double *bound);

/* SSQ twin GEMV on selected rows: y_A = W_A x_A and y_B = W_B x_B, with the
 * same bounds as above.  Returns 0, or -1 on a bad argument. */
int pti_or_twin_gemv_rows(const uint8_t *w, int64_t rows, int64_t cols,
                          const float *xa, const float *xb,
                          const int64_t *rows_idx, int64_t n_idx,
                          double *ya, double *yb, double *bound_a, double *bound_b);

/* Greedy verify ([PTI-readme] §"接受机制如何工作").
 *   logits [steps][n][vocab]; guess [steps][n] (guess[t][0] is not read)
 *   argmax [steps][n]     smallest v with logits[t][s][v] >= every other entry
 *   match  [steps][n-1]   match[t][s] = (guess[t][s+1] == argmax[t][s])   (may be NULL if n == 1)
 *   accept [steps]        number of leading 1s in match[t][.]
 * Returns 0, or -1 on a bad argument. */
int pti_or_verify_greedy(const float *logits, const int32_t *guess, int64_t steps, int n,
                         int64_t vocab, int32_t *argmax, uint8_t *match, int32_t *accept);

/* Sampling-mode verify at temperature > 0 ([PTI-readme] §"接受机制如何工作").
 *   logits [steps][n][vocab]; guess [steps][n] (guess[t][0] is not read);
 *   uniform [steps][n] in [0, 1): the random number of each stream's draw.
 *   token [steps][n]      inverse-CDF draw from p = softmax(logits / temperature):
 *                         the smallest v with p(0) + ... + p(v) > u
 *   match [steps][n-1], accept [steps]  as for the greedy verify, on the draws
 *   collision [steps][n]  sum_v p(v)^2 (may be NULL)
 *   margin [steps][n]     distance of u from the edges of the drawn token's
 *                         CDF interval (may be NULL)
 * Returns 0, or -1 on a bad argument (temperature must be finite and > 0). */
int pti_or_verify_sample(const float *logits, const int32_t *guess, const float *uniform,
                         int64_t steps, int n, int64_t vocab, double temperature,
                         int32_t *token, uint8_t *match, int32_t *accept, double *collision,
                         double *margin);

/* One layer of the multi-stream decode weight pass (gated MLP, RMS rescale):
 *   g = Wg x, u = Wu x            (Wg, Wu: [ffn][hidden] Q8)
 *   h = SiLU(g) * u, SiLU(v) = v / (1 + exp(-v))
 *   h <- h / sqrt(mean(h^2) + eps)
 *   x' = Wd h                     (Wd: [hidden][ffn] Q8)
 *   x_out = x' / sqrt(mean(x'^2) + eps)
 * per stream, all in fp64.  x_in, x_out: [n][hidden]; h_out (may be NULL):
 * [n][ffn], the normalised h.  Returns 0, or -1 on a bad argument. */
int pti_or_mlp_layer(const uint8_t *wg, const uint8_t *wu, const uint8_t *wd,
                     int64_t hidden, int64_t ffn, int n, double eps,
                     const double *x_in, double *x_out, double *h_out);

/* Greedy self-speculative decoding of a model whose next token depends on the
 * input token only ([PTI-readme] §"接受机制如何工作": stream 0 runs the model
 * on the last confirmed token, stream i on a guess for position n + i taken
 * from the previous step; [PTI-forum] §"技术实现架构", steps 2-4: compare the
 * streams' outputs, extend the confirmed text with the accepted guesses,
 * restart the rejected streams), read as a window updated in place:
 *   a[i] = next[win[i]]                    (the greedy output of stream i)
 *   L    = number of leading i < n-1 with win[i+1] == a[i]
 *   confirmed text += a[0], ..., a[L]
 *   win[0] = a[L]; win[j] = a[L+j] if L+j < n, else a[n-1]
 * starting from win[i] = first for every stream.
 *   next [vocab]     the model's greedy next token of each token
 *   tokens [cap]     confirmed tokens after `first` (those past cap are counted,
 *                    not stored); count: their number; accept [steps]: L
 * Returns 0, or -1 on a bad argument (n in 1..4, next[] in [0, vocab)). */
int pti_or_selfspec_greedy(const int32_t *next, int64_t vocab, int n, int32_t first, int64_t steps,
                           int32_t *tokens, int64_t cap, int64_t *count, int32_t *accept);

#ifdef __cplusplus
}
#endif

#endif /* PTI_ORACLE_H */
