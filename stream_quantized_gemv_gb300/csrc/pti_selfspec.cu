// pti_selfspec.cu -- device-resident greedy self-speculative decoding of a toy
// model: the loop of [PTI-readme] "打包双子推理（PTI）" §"接受机制如何工作" and
// [PTI-forum] "Packed Twin Inference：无需草稿模型的推测解码新方案，实现2倍吞吐量提升"
// §"技术实现架构" (one weight pass for every stream, compare the streams'
// outputs, extend the confirmed text with the accepted guesses, restart the
// rejected streams), read as a window of positions updated in place.
//
// One step is, in one CUDA stream: the embedding gather, the decode layer
// (two GEMVs with their tile combines and the final RMS kernel,
// pti_mlp_decode_pass), the LM-head GEMV (pti_q8_gemv_nstream, with its tile
// combine), the greedy verify of the step and the window update below.  The
// verify is split in two: a vocabulary-parallel argmax (a single step's
// 4 x vocab logits are too few rows for pti_verify_greedy's one CTA per step
// to stream them fast) and the match / accepted-length rule in the update
// kernel, with pti_verify_greedy's semantics.  The window and the confirmed
// text stay in device memory, so steps are enqueued back to back without a
// host round trip.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "pti.h"
#include "pti_host.h"

namespace pti {
namespace {

constexpr int kGatherThreads = 256;
constexpr int kArgmaxThreads = 256;
constexpr int kArgmaxChunk = 4096;  // logits of one stream per argmax CTA

// Orderable 64-bit key of (value, index): the float's bits mapped to an
// unsigned integer with the same order (-0.0 folded onto +0.0, so the two
// tie), above the complement of the index, so the maximum key is the largest
// value and, among equal values, the lowest index.  The maximum of keys does
// not depend on the order they are combined in.
__device__ __forceinline__ unsigned long long argmax_key(float v, uint32_t idx) {
  uint32_t u = __float_as_uint(v == 0.0f ? 0.0f : v);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return (static_cast<unsigned long long>(u) << 32) | (0xFFFFFFFFu - idx);
}

// keys[s] = max over v of argmax_key(logits[s][v], v); keys start at 0 (below
// every key), reset by the gather kernel of the step.
__global__ void __launch_bounds__(kArgmaxThreads) argmax_split_kernel(const float *__restrict__ logits,
                                                                      int64_t vocab,
                                                                      unsigned long long *__restrict__ keys) {
  const int s = static_cast<int>(blockIdx.y);
  const int64_t v0 = static_cast<int64_t>(blockIdx.x) * kArgmaxChunk;
  const int64_t v1 = v0 + kArgmaxChunk < vocab ? v0 + kArgmaxChunk : vocab;
  const float *row = logits + static_cast<int64_t>(s) * vocab;
  unsigned long long best = 0ull;
  for (int64_t v = v0 + threadIdx.x; v < v1; v += kArgmaxThreads) {
    const unsigned long long k = argmax_key(__ldcs(row + v), static_cast<uint32_t>(v));
    best = k > best ? k : best;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long k = __shfl_xor_sync(0xFFFFFFFFu, best, o);
    best = k > best ? k : best;
  }
  __shared__ unsigned long long warp_best[kArgmaxThreads / 32];
  if ((threadIdx.x & 31u) == 0) warp_best[threadIdx.x >> 5] = best;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kArgmaxThreads / 32; ++w) best = warp_best[w] > best ? warp_best[w] : best;
    atomicMax(keys + s, best);
  }
}

// x[s][:] = embedding[win[s]][:] for the n streams (the token clamped to
// [0, vocab), so a corrupt window cannot index outside the table); also
// resets the step's argmax keys.
__global__ void __launch_bounds__(kGatherThreads) embed_gather_kernel(const float *__restrict__ emb,
                                                                      const int32_t *__restrict__ win, int n,
                                                                      int64_t vocab, int64_t hidden,
                                                                      float *__restrict__ x,
                                                                      unsigned long long *__restrict__ keys) {
  const int s = static_cast<int>(blockIdx.y);
  if (s >= n) return;
  if (blockIdx.x == 0 && threadIdx.x == 0) keys[s] = 0ull;
  int64_t t = win[s];
  t = t < 0 ? 0 : (t >= vocab ? vocab - 1 : t);
  const float4 *src = reinterpret_cast<const float4 *>(emb + t * hidden);
  float4 *dst = reinterpret_cast<float4 *>(x + static_cast<int64_t>(s) * hidden);
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kGatherThreads + threadIdx.x; i < hidden / 4;
       i += static_cast<int64_t>(gridDim.x) * kGatherThreads)
    dst[i] = src[i];
}

// The verify rule and the window update: a[s] = the argmax of stream s (from
// its key), L = the number of leading s < n - 1 with win[s + 1] == a[s] (the
// guess fed to stream s + 1 is what stream s produced: pti_verify_greedy's
// accepted length), then the confirmed tokens a[0 .. L] and the next window
// win[0] = a[L], win[j] = a[L + j] (or a[n - 1] past the end).
struct UpdateArgs {
  int32_t *win;                   // [n] the window (stream inputs)
  const unsigned long long *keys; // [n] argmax keys of the step
  int32_t *tokens;                // [capacity] confirmed text
  int64_t capacity;
  int32_t *count;            // [1] confirmed tokens so far
  int32_t *accept_log;       // [steps] or null
  int step, n;
};

__global__ void __launch_bounds__(32) window_update_kernel(const UpdateArgs u) {
  if (threadIdx.x != 0) return;
  int32_t a[4];
  for (int i = 0; i < u.n; ++i) a[i] = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(u.keys[i]));
  int L = 0;
  while (L < u.n - 1 && u.win[L + 1] == a[L]) ++L;
  const int32_t c = u.count[0];
  for (int i = 0; i <= L; ++i)
    if (static_cast<int64_t>(c) + i < u.capacity) u.tokens[c + i] = a[i];
  u.count[0] = c + L + 1;
  if (u.accept_log != nullptr) u.accept_log[u.step] = L;
  for (int j = 0; j < u.n; ++j) u.win[j] = a[(L + j < u.n) ? (L + j) : (u.n - 1)];
}

__global__ void __launch_bounds__(32) window_init_kernel(int32_t *win, int n, int32_t first, int32_t *count) {
  if (threadIdx.x < static_cast<unsigned>(n)) win[threadIdx.x] = first;
  if (threadIdx.x == 0) count[0] = 0;
}

size_t round256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

// Workspace: window, argmax keys, x, y, logits, then the decode pass's and
// the LM-head GEMV's own workspaces.
struct SelfspecLayout {
  size_t win = 0, keys = 0, x = 0, y = 0, logits = 0, decode = 0, gemv = 0, total = 0;
  size_t decode_bytes = 0, gemv_bytes = 0;
};

SelfspecLayout selfspec_layout(int64_t vocab, int64_t hidden, int64_t ffn, int n) {
  SelfspecLayout d;
  size_t off = 0;
  d.win = off;
  off = round256(off + 4 * sizeof(int32_t));
  d.keys = off;
  off = round256(off + 4 * sizeof(unsigned long long));
  d.x = off;
  off = round256(off + static_cast<size_t>(n) * hidden * sizeof(float));
  d.y = off;
  off = round256(off + static_cast<size_t>(n) * hidden * sizeof(float));
  d.logits = off;
  off = round256(off + static_cast<size_t>(n) * vocab * sizeof(float));
  d.decode_bytes = pti_mlp_decode_pass_workspace_bytes(hidden, ffn, n);
  d.decode = off;
  off = round256(off + d.decode_bytes);
  d.gemv_bytes = pti_q8_gemv_workspace_bytes(vocab, hidden, n);
  d.gemv = off;
  off = round256(off + d.gemv_bytes);
  d.total = off;
  return d;
}

// vocab in [2, 2^24]; hidden and ffn as the decode pass requires (then the
// LM head, vocab rows by hidden columns, takes the GEMV's fast path).
bool valid_model(const pti_toy_model *m) {
  return m->vocab >= 2 && m->vocab <= (int64_t{1} << 24) &&
         pti_mlp_decode_pass_workspace_bytes(m->hidden, m->ffn, 1) != 0;
}

}  // namespace
}  // namespace pti

using namespace pti;

extern "C" size_t pti_selfspec_greedy_workspace_bytes(int64_t vocab, int64_t hidden, int64_t ffn, int n_streams) {
  if (n_streams < 1 || n_streams > 4 || vocab < 2 || vocab > (int64_t{1} << 24)) return 0;
  if (pti_mlp_decode_pass_workspace_bytes(hidden, ffn, n_streams) == 0) return 0;
  return selfspec_layout(vocab, hidden, ffn, n_streams).total;
}

extern "C" pti_status pti_selfspec_greedy(const pti_toy_model *model, int n_streams, int32_t first_token,
                                          int steps, int32_t *tokens_out, int64_t tokens_capacity,
                                          int32_t *count_out, int32_t *accept_out, void *workspace,
                                          size_t workspace_bytes, pti_stream_t stream) {
  if (model == nullptr || count_out == nullptr || workspace == nullptr) return PTI_ERR_NULL;
  if (model->embedding == nullptr || model->w_gate == nullptr || model->w_up == nullptr ||
      model->w_down == nullptr || model->w_head == nullptr)
    return PTI_ERR_NULL;
  if (n_streams < 1 || n_streams > 4) return PTI_ERR_NSTREAMS;
  // steps * n_streams confirmed tokens must fit the int32 count
  if (steps < 0 || steps > (1 << 28) || tokens_capacity < 0 || !valid_model(model)) return PTI_ERR_SHAPE;
  if (tokens_capacity > 0 && tokens_out == nullptr) return PTI_ERR_NULL;
  if (first_token < 0 || first_token >= model->vocab) return PTI_ERR_VALUE;
  if (!std::isfinite(model->eps) || model->eps < 0.0) return PTI_ERR_VALUE;
  if (!aligned(model->embedding, 16) || !aligned(model->w_gate, 16) || !aligned(model->w_up, 16) ||
      !aligned(model->w_down, 16) || !aligned(model->w_head, 16) || !aligned(workspace, 256) ||
      !aligned(count_out, 4) || (tokens_out != nullptr && !aligned(tokens_out, 4)) ||
      (accept_out != nullptr && !aligned(accept_out, 4)))
    return PTI_ERR_ALIGN;
  const size_t need = pti_selfspec_greedy_workspace_bytes(model->vocab, model->hidden, model->ffn, n_streams);
  if (need == 0) return PTI_ERR_SHAPE;
  if (workspace_bytes < need) return PTI_ERR_WORKSPACE;
  // Nothing written (the workspace, the outputs) may overlap anything read
  // (the embedding, the weights): checked here, so that no launch of the
  // loop can fail validation once the first has been enqueued.
  const uint64_t emb_bytes = static_cast<uint64_t>(model->vocab) * model->hidden * 4;
  const uint64_t gu_bytes = static_cast<uint64_t>(model->ffn) * (model->hidden / 32) * 34;
  const uint64_t dn_bytes = static_cast<uint64_t>(model->hidden) * (model->ffn / 32) * 34;
  const uint64_t hd_bytes = static_cast<uint64_t>(model->vocab) * (model->hidden / 32) * 34;
  const void *const outs[4] = {workspace, tokens_out, count_out, accept_out};
  const uint64_t out_bytes[4] = {workspace_bytes, static_cast<uint64_t>(tokens_capacity) * 4, 4,
                                 static_cast<uint64_t>(steps) * 4};
  for (int k = 0; k < 4; ++k)
    if (overlaps(outs[k], out_bytes[k], model->embedding, emb_bytes) ||
        overlaps(outs[k], out_bytes[k], model->w_gate, gu_bytes) ||
        overlaps(outs[k], out_bytes[k], model->w_up, gu_bytes) ||
        overlaps(outs[k], out_bytes[k], model->w_down, dn_bytes) ||
        overlaps(outs[k], out_bytes[k], model->w_head, hd_bytes))
      return PTI_ERR_ALIAS;
  if (overlaps(workspace, workspace_bytes, tokens_out, static_cast<uint64_t>(tokens_capacity) * 4) ||
      overlaps(workspace, workspace_bytes, count_out, 4) ||
      overlaps(workspace, workspace_bytes, accept_out, static_cast<uint64_t>(steps) * 4) ||
      overlaps(tokens_out, static_cast<uint64_t>(tokens_capacity) * 4, count_out, 4) ||
      overlaps(accept_out, static_cast<uint64_t>(steps) * 4, count_out, 4) ||
      overlaps(accept_out, static_cast<uint64_t>(steps) * 4, tokens_out, static_cast<uint64_t>(tokens_capacity) * 4))
    return PTI_ERR_ALIAS;

  const SelfspecLayout d = selfspec_layout(model->vocab, model->hidden, model->ffn, n_streams);
  uint8_t *const ws = static_cast<uint8_t *>(workspace);
  int32_t *const win = reinterpret_cast<int32_t *>(ws + d.win);
  unsigned long long *const keys = reinterpret_cast<unsigned long long *>(ws + d.keys);
  float *const x = reinterpret_cast<float *>(ws + d.x);
  float *const y = reinterpret_cast<float *>(ws + d.y);
  float *const logits = reinterpret_cast<float *>(ws + d.logits);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

  window_init_kernel<<<1, 32, 0, st>>>(win, n_streams, first_token, count_out);
  if (cudaGetLastError() != cudaSuccess) return PTI_ERR_CUDA;
  const int64_t chunks = model->hidden / 4;
  const unsigned gx = static_cast<unsigned>((chunks + kGatherThreads - 1) / kGatherThreads);
  const unsigned ax = static_cast<unsigned>((model->vocab + kArgmaxChunk - 1) / kArgmaxChunk);
  const void *const wg[1] = {model->w_gate};
  const void *const wu[1] = {model->w_up};
  const void *const wd[1] = {model->w_down};
  for (int step = 0; step < steps; ++step) {
    embed_gather_kernel<<<dim3(gx, static_cast<unsigned>(n_streams)), kGatherThreads, 0, st>>>(
        model->embedding, win, n_streams, model->vocab, model->hidden, x, keys);
    if (cudaGetLastError() != cudaSuccess) return PTI_ERR_CUDA;
    if (const pti_status s = pti_mlp_decode_pass(wg, wu, wd, 1, model->hidden, model->ffn, n_streams, model->eps,
                                                 x, y, ws + d.decode, d.decode_bytes, stream);
        s != PTI_OK)
      return s;
    if (const pti_status s = pti_q8_gemv_nstream(model->w_head, model->vocab, model->hidden, n_streams, y, logits,
                                                 ws + d.gemv, d.gemv_bytes, stream);
        s != PTI_OK)
      return s;
    argmax_split_kernel<<<dim3(ax, static_cast<unsigned>(n_streams)), kArgmaxThreads, 0, st>>>(logits, model->vocab,
                                                                                              keys);
    if (cudaGetLastError() != cudaSuccess) return PTI_ERR_CUDA;
    UpdateArgs u{win, keys, tokens_out, tokens_capacity, count_out, accept_out, step, n_streams};
    window_update_kernel<<<1, 32, 0, st>>>(u);
    if (cudaGetLastError() != cudaSuccess) return PTI_ERR_CUDA;
  }
  return PTI_OK;
}
