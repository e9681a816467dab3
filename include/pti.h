/*
 * pti.h -- C ABI of the Packed Twin Inference hot path on NVIDIA GB300 (sm_103a).
 *
 * Packed Twin Inference is self-speculative decoding in which one weight load
 * from HBM serves several token streams.  This library holds its hot path:
 *
 *   pti_q8_gemv_nstream   N-stream Q8 GEMV: one pass over a Q8 matrix computes
 *                         y_s = W x_s for 1..4 activation vectors x_s.
 *   pti_ssq_twin_gemv     SSQ "mode 16" twin GEMV: one pass over a packed twin
 *                         matrix computes y_A = W_A x_A and y_B = W_B x_B.
 *   pti_verify_sample     sampling-mode verify: per-stream inverse-CDF draw from
 *                         softmax(logits / T), acceptance and sum p^2.
 *   pti_verify_greedy     greedy verify: per-stream argmax, guess == actual and
 *                         the accepted-prefix length of every step.
 *   pti_mlp_decode_pass   a chained decode pass: n_layers gated-MLP layers
 *                         (gate, up, SiLU, RMS, down, RMS) over 1..4 streams,
 *                         one pass over the weights for all streams.
 *   pti_selfspec_greedy   greedy self-speculative decoding of a toy model on
 *                         1..4 streams, device-resident (window update on the
 *                         GPU, no host synchronisation per step).
 *
 * Sources are cited by page title and section:
 *   [PTI-forum]  "Packed Twin Inference：无需草稿模型的推测解码新方案，实现2倍吞吐量提升"
 *   [PTI-readme] "打包双子推理（PTI）"
 *   [CS336-L10]  "推理（Inference）" (CS336 lecture 10 notes)
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Memory.  Every data pointer is DEVICE memory owned by the caller; the
 *   library never frees or retains it.  No entry point allocates memory.  The
 *   library keeps no per-call state; a device-side error word (see
 *   pti_device_error) is the only global state.
 * Streams.  `stream` is a cudaStream_t (NULL = the legacy default stream).
 *   Every call only validates its arguments and enqueues work: PTI_OK means
 *   "validated and launched", the results are ready when the stream reaches
 *   that point.  Inputs are never modified.
 * Errors.  Arguments are validated on the host before anything is enqueued;
 *   a failed validation enqueues nothing.  A launch failure reported by the
 *   CUDA runtime returns PTI_ERR_CUDA.  Kernels never trap or assert: a
 *   pipeline wait that exceeds its time limit (which only a hardware fault can
 *   cause) makes the kernel record a code in the device error word, skip its
 *   remaining work and return.
 * Layouts.  Little-endian byte layouts, matrices row-major:
 *   Q8 block (34 bytes, 32 columns): [0..1] scale d as IEEE binary16,
 *     [2..33] q[0..31] int8; weight = d * q.
 *   SSQ twin block (68 bytes, 32 columns of two models A and B):
 *     [0..1] scale_A binary16, [2..3] scale_B binary16, then 32 uint16 pw[i]
 *     (bytes 4+2i, 5+2i) with model A's int8 in the high byte and model B's
 *     int8 in the low byte ([PTI-forum] §"PTI的核心创新：SSQ打包技术").
 *   A rows x cols matrix is rows consecutive rows of cols/32 blocks.
 *   Activations and outputs are fp32, stream-major: x[s][k], y[s][r].
 * Arithmetic.  fp32 with exact dequantisation (scale * q is formed exactly),
 *   accumulation order fixed (results are bit-reproducible run to run); each
 *   output stays within 1e-5 * sum_k |w_k x_k| of the exact value.
 */
#ifndef PTI_H
#define PTI_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st *pti_stream_t; /* identical to cudaStream_t */

typedef enum pti_status {
    PTI_OK = 0,
    PTI_ERR_NULL = 1,      /* a required pointer is NULL */
    PTI_ERR_SHAPE = 2,     /* rows < 1, cols < 32, cols % 32 != 0, steps < 0, vocab < 1, layers < 1, too large */
    PTI_ERR_NSTREAMS = 3,  /* n_streams outside [1, 4] */
    PTI_ERR_ALIGN = 4,     /* a pointer is not aligned as documented */
    PTI_ERR_ALIAS = 5,     /* an output overlaps an input or another output */
    PTI_ERR_CUDA = 6,      /* the CUDA runtime reported an error (no device, launch failure) */
    PTI_ERR_WORKSPACE = 7, /* workspace missing or smaller than required */
    PTI_ERR_VALUE = 8      /* a scalar argument outside its documented range (eps, flags) */
} pti_status;

/* Human-readable name of a status code (static storage, never NULL). */
const char *pti_status_string(pti_status status);

/*
 * N-stream Q8 GEMV.
 *   [PTI-readme] §"带宽分析：为什么会有开销": one kernel loads each weight
 *   group once and forms the N dot products together, reading the N
 *   activation vectors side by side and reducing all N streams in one pass.
 *
 *   w_q8       [rows][cols/32] Q8 blocks, 16-byte aligned.
 *   rows, cols rows >= 1, cols >= 32, cols % 32 == 0, rows * cols < 2^40.
 *   n_streams  1..4.
 *   x          [n_streams][cols] fp32, 4-byte aligned.
 *   y          [n_streams][rows] fp32 out, 4-byte aligned, overlapping neither
 *              w_q8 nor x.
 *   workspace  device scratch of at least pti_q8_gemv_workspace_bytes(rows,
 *              cols, n_streams) bytes (at most 1,310,720 bytes: it depends only
 *              on n_streams), 256-byte aligned; its contents need no
 *              initialisation and are undefined afterwards, so one workspace
 *              serves calls of any shape and stream count; may be NULL when
 *              that size is 0.  Calls that share a workspace must be ordered
 *              (same stream or synchronised).
 * Fast path when cols % 256 == 0 and x is 16-byte aligned: TMA-streamed,
 * persistent, one pass over the weights, followed by a small kernel that
 * adds the partial sums of the row tiles several CTAs shared (launched with
 * programmatic dependent launch, so it waits for the GEMV without a launch
 * gap); other calls use a plain per-row kernel with the same bound on the
 * error (a different rounding order).  The fast path forms the products on
 * the CUDA cores (exact dequantisation, fp32 FMAs); with PTI_FLAG_TENSOR_CORES
 * (the _ex variant) on the tensor core instead (tcgen05.mma on binary16
 * operands that hold every weight exactly and every fp32 activation as three
 * pieces, with fp32 accumulation), measured no faster on GB300.  That path's
 * pieces are scaled per 32-column block and stream, and an activation 2^15
 * or more below its block's largest loses bits: its error bound adds at most
 * 2^-39 * sum_k |w_k| * (largest |x| in k's block) to the bar above (nothing
 * for blocks whose values lie within a factor 2^15 of each other).  A
 * non-finite activation gives non-finite outputs on both paths (NaN on the
 * tensor core where the CUDA cores may give an infinity).
 */
size_t pti_q8_gemv_workspace_bytes(int64_t rows, int64_t cols, int n_streams);

pti_status pti_q8_gemv_nstream(const void *w_q8, int64_t rows, int64_t cols, int n_streams,
                               const float *x, float *y,
                               void *workspace, size_t workspace_bytes,
                               pti_stream_t stream);

/*
 * Launch flags of the _ex variants below (0 = the plain entry point's
 * behaviour).
 *   PTI_FLAG_PDL  programmatic dependent launch: the GEMV may start while the
 *                 kernel before it in `stream` is still running.  Until that
 *                 kernel has completed, the GEMV only reads the weight matrix
 *                 (it fetches its first weight tiles early); it reads x and
 *                 writes y and the workspace only afterwards.  So the caller
 *                 promises that the preceding work in the stream does not write
 *                 the weights.  This hides most of the launch and ramp-up time
 *                 of a GEMV that follows another kernel (a decode step's chain
 *                 of GEMVs).
 *   PTI_FLAG_CUDA_CORES, PTI_FLAG_TENSOR_CORES  (Q8 GEMV only) the fast
 *                 path's products on the CUDA cores (the default) or on the
 *                 tensor core; both at once return PTI_ERR_VALUE, and so does
 *                 either one on the twin GEMVs.
 * Other flag bits return PTI_ERR_VALUE.
 */
#define PTI_FLAG_PDL 0x1u
#define PTI_FLAG_CUDA_CORES 0x2u
#define PTI_FLAG_TENSOR_CORES 0x4u

pti_status pti_q8_gemv_nstream_ex(const void *w_q8, int64_t rows, int64_t cols, int n_streams,
                                  const float *x, float *y,
                                  void *workspace, size_t workspace_bytes,
                                  pti_stream_t stream, uint32_t flags);

/*
 * Allocation-free N-stream Q8 GEMV.  The pages have no counterpart: this is a
 * library convenience for callers that cannot allocate device memory, such as
 * a plug-in running inside a host runtime that owns every device allocation
 * through its own pool, or a decode loop that must not call the CUDA allocator
 * once it runs (freeing device memory synchronises the whole device).
 *
 * Same arguments, results and checks as pti_q8_gemv_nstream, without the
 * workspace: the scratch it needs lives in a 2 MiB array inside this library
 * (pti_q8_gemv_noalloc_max_scratch_bytes()), held by every GPU that loads the
 * library until the process exits.  Every valid shape fits (the scratch
 * depends only on n_streams, at most 1.31 MB); a request for more would return
 * PTI_ERR_WORKSPACE before anything is enqueued.  The call allocates nothing.
 *
 * The first call on a device looks up the array's device address (so make
 * that first call before any stream capture) and keeps it for the life of the
 * process: do not use this entry point across a cudaDeviceReset of that
 * device.  All calls on a device share the one array: calls that overlap on
 * the GPU race, so order them (one stream, or synchronise).
 */
size_t pti_q8_gemv_noalloc_max_scratch_bytes(void);

pti_status pti_q8_gemv_nstream_noalloc(const void *w_q8, int64_t rows, int64_t cols, int n_streams,
                                       const float *x, float *y, pti_stream_t stream);

/*
 * SSQ mode-16 twin GEMV.
 *   [PTI-readme] §"与 SSQ（Side-by-Side Quantization）的关系" and [PTI-forum]
 *   §"PTI的核心创新：SSQ打包技术": a twin block packs the same 32 columns of
 *   two models.  It starts with model A's binary16 scale and then model B's,
 *   followed by 32 little-endian 16-bit elements; element i holds column i
 *   of model A as a signed byte in its upper 8 bits and column i of model B
 *   in its lower 8 bits.  One read of the packed matrix gives both products,
 *   y_a = W_A x_a and y_b = W_B x_b.
 *
 *   w_twin     [rows][cols/32] twin blocks (68 bytes each), 16-byte aligned.
 *   rows, cols as for the Q8 GEMV.
 *   x_a, x_b   [cols] fp32 (A's and B's activations; may be the same pointer).
 *   y_a, y_b   [rows] fp32 out; distinct, overlapping no input.
 *   workspace  as for the Q8 GEMV (scratch, no initialisation), sized by
 *              pti_ssq_twin_gemv_workspace_bytes.
 * Fast path when cols % 128 == 0 and x_a, x_b are 16-byte aligned.
 */
size_t pti_ssq_twin_gemv_workspace_bytes(int64_t rows, int64_t cols);

pti_status pti_ssq_twin_gemv(const void *w_twin, int64_t rows, int64_t cols,
                             const float *x_a, const float *x_b, float *y_a, float *y_b,
                             void *workspace, size_t workspace_bytes,
                             pti_stream_t stream);

/*
 * Twin GEMV with several streams per model: one pass over the packed twin
 * matrix serves n_streams activation vectors of model A and n_streams of
 * model B, y_A[s] = W_A x_A[s] and y_B[s] = W_B x_B[s].  With n_streams = 2,
 * one weight load serves four tokens ([PTI-forum] §"未来发展方向": the PTI +
 * MTP plan of four tokens per weight load; here the two extra tokens come
 * from a second stream per twin, e.g. two speculative positions).
 *
 *   n_streams  1 or 2 per model (n_streams = 1 is pti_ssq_twin_gemv_ex).
 *   x_a, x_b   [n_streams][cols] fp32 each, stream-major.
 *   y_a, y_b   [n_streams][rows] fp32 out each; distinct, overlapping no input.
 *   workspace  pti_ssq_twin_gemv_nstream_workspace_bytes(rows, cols, n_streams)
 *              bytes of scratch (as for the other GEMVs).
 *   flags      PTI_FLAG_PDL or 0.
 * Other arguments, the fast-path condition and the error bound as for
 * pti_ssq_twin_gemv.  A caller with an unequal number of streams per model
 * passes a copy of one vector twice.
 */
size_t pti_ssq_twin_gemv_nstream_workspace_bytes(int64_t rows, int64_t cols, int n_streams);

pti_status pti_ssq_twin_gemv_nstream(const void *w_twin, int64_t rows, int64_t cols, int n_streams,
                                     const float *x_a, const float *x_b, float *y_a, float *y_b,
                                     void *workspace, size_t workspace_bytes,
                                     pti_stream_t stream, uint32_t flags);

/* pti_ssq_twin_gemv with launch flags (PTI_FLAG_PDL, see above). */
pti_status pti_ssq_twin_gemv_ex(const void *w_twin, int64_t rows, int64_t cols,
                                const float *x_a, const float *x_b, float *y_a, float *y_b,
                                void *workspace, size_t workspace_bytes,
                                pti_stream_t stream, uint32_t flags);

/*
 * Greedy verify.
 *   [PTI-readme] §"接受机制如何工作": stream 0 runs the model on the confirmed
 *   token, stream s on the guess for position n+s; under greedy decoding the
 *   guess fed to stream s+1 is accepted when it equals stream s's argmax, and
 *   acceptance stops at the first mismatch (each step emits 1 + accept_len
 *   tokens).  [PTI-forum] §"技术实现架构", step 3.
 *
 *   logits      [steps][n_streams][vocab] fp32, 4-byte aligned (16-byte
 *               aligned rows take the vector path).  Precondition: no NaN.
 *   guess       [steps][n_streams] int32; guess[t][0] is not read.
 *   steps >= 0, n_streams in [1, 4], vocab in [1, 2^31 - 1].
 *   argmax_out  [steps][n_streams] int32 out: the smallest index holding the
 *               row's maximum (-0.0 and +0.0 compare equal).
 *   match_out   [steps][n_streams-1] uint8 out, 1 when guess[t][s+1] ==
 *               argmax[t][s]; may be NULL when n_streams == 1.
 *   accept_len_out [steps] int32 out, the number of leading 1s of match, in
 *               [0, n_streams - 1].
 * steps == 0 enqueues nothing and returns PTI_OK (the pointers are not
 * checked, since nothing is read or written).
 */
pti_status pti_verify_greedy(const float *logits, const int32_t *guess,
                             int64_t steps, int n_streams, int64_t vocab,
                             int32_t *argmax_out, uint8_t *match_out, int32_t *accept_len_out,
                             pti_stream_t stream);

/*
 * Sampling-mode verify.
 *   [PTI-readme] §"接受机制如何工作", the temperature > 0 case: stream s's
 *   output token is a draw from p_s = softmax(logits[t][s] / T); the guess fed
 *   to stream s+1 is accepted when it equals stream s's draw, and acceptance
 *   stops at the first mismatch.  A guess drawn independently from the same
 *   distribution matches with probability sum_v p(v)^2 (the collision
 *   probability), returned per stream.
 *
 *   logits      [steps][n_streams][vocab] fp32, 4-byte aligned (16-byte
 *               aligned rows take the vector path).  -inf marks a token with
 *               no mass; each row needs at least one finite logit, and NaN or
 *               +inf give unspecified (but in-range) tokens.
 *   guess       [steps][n_streams] int32; guess[t][0] is not read.
 *   uniform     [steps][n_streams] fp32 in [0, 1): the random number of each
 *               draw (supplied by the caller, so the draw is a plain function
 *               of the inputs).  Other values give unspecified in-range tokens.
 *   temperature T > 0, finite, with log2(e) / T finite in fp32 (else
 *               PTI_ERR_VALUE).
 *   token_out   [steps][n_streams] int32 out: the inverse-CDF draw, the
 *               smallest v with p(0) + ... + p(v) > u, computed in fp32; when
 *               u lies within fp32 rounding of an interval edge either
 *               neighbouring token may be returned (always one with p > 0).
 *               Results are deterministic.
 *   match_out   [steps][n_streams-1] uint8 out, 1 when guess[t][s+1] ==
 *               token[t][s]; may be NULL when n_streams == 1.
 *   accept_len_out [steps] int32 out, the number of leading 1s of match.
 *   collision_out  [steps][n_streams] fp32 out, sum_v p(v)^2, or NULL.
 * steps == 0 enqueues nothing and returns PTI_OK once the scalars are valid.
 * One CTA handles one step; each row is read once from HBM plus about a
 * sixteenth of it again from L2.
 */
pti_status pti_verify_sample(const float *logits, const int32_t *guess, const float *uniform,
                             int64_t steps, int n_streams, int64_t vocab, float temperature,
                             int32_t *token_out, uint8_t *match_out, int32_t *accept_len_out,
                             float *collision_out, pti_stream_t stream);

/*
 * Chained decode pass over n_layers gated-MLP layers.
 *   A decode step of the N streams is one pass over all the weights for all N
 *   streams ([PTI-readme] §"带宽分析：为什么会有开销"; [PTI-forum] §"技术实现架构",
 *   step 2).  The layer is the gated MLP (W_gate, W_up, W_down) of [CS336-L10]
 *   §"2.4 MLP 层的算术强度"; the pages name no nonlinearity or normalisation,
 *   so this library takes SiLU and an RMS rescale after h and after the layer:
 *     g = W_gate x,  u = W_up x                 (ffn rows, hidden columns)
 *     h = rms(SiLU(g) * u)                      rms(v) = v / sqrt(mean(v^2) + eps)
 *     x <- rms(W_down h)                        (hidden rows, ffn columns)
 *   for every stream s independently.
 *
 *   w_gate, w_up, w_down  HOST arrays of n_layers DEVICE pointers: layer l
 *              reads w_gate[l] and w_up[l] ([ffn][hidden/32] Q8 blocks) and
 *              w_down[l] ([hidden][ffn/32] Q8 blocks), each 16-byte aligned.
 *              The arrays are read during the call only; layers may share
 *              matrices.
 *   n_layers   1 .. 4096.
 *   hidden, ffn  multiples of 256, hidden * ffn < 2^40.
 *   n_streams  1..4.
 *   eps        finite, >= 0 (else PTI_ERR_VALUE).
 *   x_in       [n_streams][hidden] fp32, 16-byte aligned; read by the first
 *              layer only.
 *   x_out      [n_streams][hidden] fp32 out, 4-byte aligned, overlapping no
 *              weight matrix; may be x_in (in place).
 *   workspace  at least pti_mlp_decode_pass_workspace_bytes(hidden, ffn,
 *              n_streams) bytes, 256-byte aligned, overlapping no argument;
 *              scratch (h, each layer's raw output, per-tile sums of squares,
 *              partial sums): no initialisation needed, contents undefined
 *              afterwards.  One workspace may serve this call and the GEMVs
 *              above, ordered in one stream.
 * Work per layer: a gate/up step streams W_gate and W_up together (64 gate
 * rows and their 64 up rows per tile) and writes SiLU(g) * u; a down step
 * streams W_down and applies h's RMS scale to its output; each writes per-tile
 * sums of squares of its output, from which the next step takes the RMS scale
 * of its input (W (c v) = c (W v), so no separate normalisation pass over the
 * vectors is needed).  A last kernel applies the final RMS scale.  Each
 * gate/up and down step is its own launch (with a small kernel behind it that
 * combines the row tiles several CTAs shared), all chained by programmatic
 * dependent launch: a step streams its first weight tiles while the previous
 * one finishes.  The first launch waits for all earlier work in the stream.
 * Arithmetic: GEMVs as in the conventions, SiLU with expf, RMS scales from
 * fp32 per-tile sums of squares summed exactly enough (float-float, about
 * 1e-15 relative) and a float reciprocal square root refined in double;
 * bit-reproducible run to run.
 */
size_t pti_mlp_decode_pass_workspace_bytes(int64_t hidden, int64_t ffn, int n_streams);

pti_status pti_mlp_decode_pass(const void *const *w_gate, const void *const *w_up, const void *const *w_down,
                               int n_layers, int64_t hidden, int64_t ffn, int n_streams, double eps,
                               const float *x_in, float *x_out,
                               void *workspace, size_t workspace_bytes,
                               pti_stream_t stream);

/*
 * Greedy self-speculative decoding of a toy model, on the device.
 *   [PTI-readme] §"接受机制如何工作": in each step stream 0 runs the model on
 *   the last confirmed token (position n) and stream i >= 1 on a guess for
 *   position n + i taken from the previous step; one weight pass serves all
 *   streams ([PTI-forum] §"技术实现架构", steps 2-4: the streams' outputs are
 *   compared, the confirmed text is extended by the accepted guesses, the
 *   streams past the first rejection restart).  The pages give the loop only
 *   in outline; this library reads it as a window of n_streams positions
 *   updated in place (Jacobi iteration):
 *     a[i]  = argmax (lowest index on ties) of the model's logits for token
 *             win[i], i.e. the model's next token after win[i];
 *     L     = the number of leading i < n_streams - 1 with win[i+1] == a[i]
 *             (pti_verify_greedy's rule with guess = win; argmax ties go to
 *             the lowest index, -0.0 ties +0.0);
 *     a[0 .. L] are appended to the confirmed text (each is the model's
 *     greedy continuation of a confirmed token, so the text is exactly the
 *     model's greedy rollout from first_token: no quality loss);
 *     win'[0] = a[L]; win'[j] = a[L + j] while L + j < n_streams, else
 *     a[n_streams - 1] (the streams past the rejection restart from the
 *     newest outputs).
 *   The initial window is first_token in every stream.
 * The toy model has no state beyond the input token (its logits depend on
 * that token only), so a stream's "KV state" is its window token:
 *     x = embedding[token]; x = one decode layer (pti_mlp_decode_pass);
 *     logits = W_head x  (pti_q8_gemv_nstream, vocab rows, hidden columns).
 *
 *   model      HOST struct, read during the call: embedding [vocab][hidden]
 *              fp32 (16-byte aligned), the layer's w_gate, w_up ([ffn]
 *              [hidden/32] Q8 blocks), w_down ([hidden][ffn/32]) and w_head
 *              ([vocab][hidden/32]), all DEVICE pointers, 16-byte aligned;
 *              vocab 2 .. 2^24, hidden and ffn as pti_mlp_decode_pass,
 *              eps finite >= 0.
 *   n_streams  1..4 (1: plain greedy decoding, one token per step).
 *   first_token  in [0, vocab).
 *   steps      0 .. 2^28 decode steps, each one pass over the weights for all
 *              streams; enqueued as 10 launches per step (embedding gather,
 *              the decode layer's 5, the LM head and its tile combine, a
 *              vocabulary-parallel argmax, the verify rule and window
 *              update), no host synchronisation.
 *   tokens_out DEVICE [tokens_capacity] int32: the confirmed tokens after
 *              first_token, in order; tokens past the capacity are counted
 *              but not stored.
 *   count_out  DEVICE int32: the number of confirmed tokens (sum over steps
 *              of 1 + accept_out[step]).
 *   accept_out DEVICE [steps] int32 (may be NULL): L of each step.
 *   workspace  at least pti_selfspec_greedy_workspace_bytes(vocab, hidden,
 *              ffn, n_streams) bytes, 256-byte aligned, scratch.
 * Errors: invalid arguments return a status and enqueue nothing; the embedding
 * and the tokens are checked only on the host side (pointers, alignment);
 * a token is used as an index only after clamping to [0, vocab).  As for
 * pti_verify_greedy the logits must be finite (a NaN logit makes the argmax
 * unspecified).
 */
typedef struct pti_toy_model {
    const float *embedding;
    const void *w_gate, *w_up, *w_down, *w_head;
    int64_t vocab, hidden, ffn;
    double eps;
} pti_toy_model;

size_t pti_selfspec_greedy_workspace_bytes(int64_t vocab, int64_t hidden, int64_t ffn, int n_streams);

pti_status pti_selfspec_greedy(const pti_toy_model *model, int n_streams, int32_t first_token, int steps,
                               int32_t *tokens_out, int64_t tokens_capacity, int32_t *count_out,
                               int32_t *accept_out, void *workspace, size_t workspace_bytes,
                               pti_stream_t stream);

/*
 * Testing hook for the pipeline's bounded waits; the pages have no
 * counterpart.  It is the fast-path pti_q8_gemv_nstream (cols % 256 == 0, x
 * 16-byte aligned, workspace given) with two changes that make one wait run
 * out without harming the GPU:
 *   - the copy producer of the first CTA issues no copy from its unit
 *     `stall_unit` on, as if that copy never arrived;
 *   - every pipeline wait gives up after `wait_ns` nanoseconds instead of
 *     2 seconds.
 * The consumer warps waiting for the missing tile then give up, record
 * PTI_DEVERR_FULL_TIMEOUT in the device error word (pti_device_error), and
 * skip their remaining waits; every copy that was issued has landed before the
 * kernel exits (else PTI_DEVERR_DRAIN_TIMEOUT is recorded too), so the
 * device, the stream and the library stay usable.  y is undefined afterwards.
 *   stall_unit  at least 6 (the ring depth) and below the first CTA's unit
 *               count (units / grid, units = (rows/128 rounded up) (cols/256),
 *               grid = min(SM count, units, 320)); else PTI_ERR_VALUE.
 *   wait_ns     1000 .. 2e9; else PTI_ERR_VALUE.
 *   flags       0, PTI_FLAG_CUDA_CORES or PTI_FLAG_TENSOR_CORES (which
 *               consumer runs, as for pti_q8_gemv_nstream_ex).
 * Other arguments and checks as pti_q8_gemv_nstream.
 */
pti_status pti_test_q8_gemv_stall(const void *w_q8, int64_t rows, int64_t cols, int n_streams,
                                  const float *x, float *y, void *workspace, size_t workspace_bytes,
                                  pti_stream_t stream, int64_t stall_unit, uint64_t wait_ns, uint32_t flags);

/*
 * Reads and clears the device error word of the current device (a blocking
 * call: it synchronises the device).  0 means no kernel of this library has
 * recorded an error since the last call; otherwise a bit set of
 * PTI_DEVERR_* codes.  Returns PTI_OK or PTI_ERR_CUDA.
 */
#define PTI_DEVERR_FULL_TIMEOUT 0x1u  /* a consumer waited too long for a weight tile */
#define PTI_DEVERR_EMPTY_TIMEOUT 0x2u /* the producer waited too long for a free slot */
#define PTI_DEVERR_DRAIN_TIMEOUT 0x4u /* copies still in flight at exit after an error */
pti_status pti_device_error(uint32_t *code_out);

#ifdef __cplusplus
}
#endif

#endif /* PTI_H */
