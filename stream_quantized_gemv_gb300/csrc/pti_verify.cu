// pti_verify.cu -- greedy verify of self-speculative decoding on sm_103a.
//
// [PTI-readme] "打包双子推理（PTI）" §"接受机制如何工作": at each step stream 0
// runs on the confirmed token and stream s on the guess for position n+s.  Under
// greedy decoding stream s's output is the argmax of its logits row; the guess
// fed to stream s+1 is accepted when it equals that argmax, and acceptance
// stops at the first mismatch.  ([PTI-forum] §"技术实现架构", step 3 "验证".)
//
// One CTA handles one step (its n_streams logits rows), so the match flags and
// the accepted-prefix length need no cross-CTA communication.  Rows are
// streamed with 16-byte evict-first loads, several in flight per thread; the
// (value, index) maximum is reduced with the order "larger value, then smaller
// index", a total order on non-NaN values, so the result is the smallest index
// holding the row maximum whatever the reduction order.
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cstdint>

#include "pti.h"
#include "pti_host.h"

namespace pti {
namespace {

constexpr int kVerifyThreads = 512;
constexpr int kVerifyWarps = kVerifyThreads / 32;

__device__ __forceinline__ void take_better(float &bv, int &bi, float v, int i) {
  if (v > bv || (v == bv && i < bi)) {
    bv = v;
    bi = i;
  }
}

__device__ __forceinline__ void take4(float &bv, int &bi, const float4 &f, int i0) {
  take_better(bv, bi, f.x, i0);
  take_better(bv, bi, f.y, i0 + 1);
  take_better(bv, bi, f.z, i0 + 2);
  take_better(bv, bi, f.w, i0 + 3);
}

template <bool kVec>
__global__ void __launch_bounds__(kVerifyThreads)
    verify_greedy_kernel(const float *__restrict__ logits, const int32_t *__restrict__ guess, int64_t steps,
                         int n, int64_t vocab, int32_t *__restrict__ argmax_out, uint8_t *__restrict__ match_out,
                         int32_t *__restrict__ accept_out) {
  __shared__ float s_val[kVerifyWarps];
  __shared__ int s_idx[kVerifyWarps];
  __shared__ int s_arg[4];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int64_t t = blockIdx.x; t < steps; t += gridDim.x) {
    for (int s = 0; s < n; ++s) {
      const float *row = logits + (t * n + s) * vocab;
      float bv = -INFINITY;
      int bi = INT_MAX;
      if constexpr (kVec) {
        const float4 *row4 = reinterpret_cast<const float4 *>(row);
        const int64_t nv = vocab >> 2;
        int64_t v = tid;
        for (; v + 3 * kVerifyThreads < nv; v += 4 * kVerifyThreads) {
          const float4 a0 = __ldcs(row4 + v);
          const float4 a1 = __ldcs(row4 + v + kVerifyThreads);
          const float4 a2 = __ldcs(row4 + v + 2 * kVerifyThreads);
          const float4 a3 = __ldcs(row4 + v + 3 * kVerifyThreads);
          take4(bv, bi, a0, static_cast<int>(4 * v));
          take4(bv, bi, a1, static_cast<int>(4 * (v + kVerifyThreads)));
          take4(bv, bi, a2, static_cast<int>(4 * (v + 2 * kVerifyThreads)));
          take4(bv, bi, a3, static_cast<int>(4 * (v + 3 * kVerifyThreads)));
        }
        for (; v < nv; v += kVerifyThreads) take4(bv, bi, __ldcs(row4 + v), static_cast<int>(4 * v));
        for (int64_t e = 4 * nv + tid; e < vocab; e += kVerifyThreads)
          take_better(bv, bi, __ldcs(row + e), static_cast<int>(e));
      } else {
        for (int64_t e = tid; e < vocab; e += kVerifyThreads) take_better(bv, bi, __ldcs(row + e), static_cast<int>(e));
      }
      for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, o);
        const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, o);
        take_better(bv, bi, ov, oi);
      }
      if (lane == 0) {
        s_val[warp] = bv;
        s_idx[warp] = bi;
      }
      __syncthreads();
      if (warp == 0) {
        bv = lane < kVerifyWarps ? s_val[lane] : -INFINITY;
        bi = lane < kVerifyWarps ? s_idx[lane] : INT_MAX;
        for (int o = 16; o > 0; o >>= 1) {
          const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, o);
          const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, o);
          take_better(bv, bi, ov, oi);
        }
        if (lane == 0) {
          s_arg[s] = bi;
          argmax_out[t * n + s] = bi;
        }
      }
      __syncthreads();
    }
    if (tid == 0) {
      int32_t accepted = 0;
      bool run = true;
      for (int s = 0; s + 1 < n; ++s) {
        const bool m = guess[t * n + s + 1] == s_arg[s];
        match_out[t * (n - 1) + s] = m ? 1 : 0;
        if (run && m) ++accepted;
        else run = false;
      }
      accept_out[t] = accepted;
    }
    __syncthreads();
  }
}

}  // namespace
}  // namespace pti

using namespace pti;

extern "C" pti_status pti_verify_greedy(const float *logits, const int32_t *guess, int64_t steps, int n_streams,
                                        int64_t vocab, int32_t *argmax_out, uint8_t *match_out,
                                        int32_t *accept_len_out, pti_stream_t stream) {
  if (n_streams < 1 || n_streams > 4) return PTI_ERR_NSTREAMS;
  if (steps < 0 || vocab < 1 || vocab > INT_MAX) return PTI_ERR_SHAPE;
  if (steps > (int64_t{1} << 40) / (static_cast<int64_t>(n_streams) * vocab)) return PTI_ERR_SHAPE;
  if (steps == 0) return PTI_OK;  // nothing is read or written: pointers may be NULL
  if (logits == nullptr || guess == nullptr || argmax_out == nullptr || accept_len_out == nullptr ||
      (n_streams > 1 && match_out == nullptr))
    return PTI_ERR_NULL;
  if (!aligned(logits, 4) || !aligned(guess, 4) || !aligned(argmax_out, 4) || !aligned(accept_len_out, 4))
    return PTI_ERR_ALIGN;
  const uint64_t l_bytes = static_cast<uint64_t>(steps) * n_streams * vocab * 4;
  const uint64_t g_bytes = static_cast<uint64_t>(steps) * n_streams * 4;
  const uint64_t a_bytes = g_bytes;
  const uint64_t m_bytes = n_streams > 1 ? static_cast<uint64_t>(steps) * (n_streams - 1) : 0;
  const uint64_t c_bytes = static_cast<uint64_t>(steps) * 4;
  const void *outs[3] = {argmax_out, match_out, accept_len_out};
  const uint64_t out_bytes[3] = {a_bytes, m_bytes, c_bytes};
  for (int i = 0; i < 3; ++i) {
    if (overlaps(outs[i], out_bytes[i], logits, l_bytes) || overlaps(outs[i], out_bytes[i], guess, g_bytes))
      return PTI_ERR_ALIAS;
    for (int j = i + 1; j < 3; ++j)
      if (overlaps(outs[i], out_bytes[i], outs[j], out_bytes[j])) return PTI_ERR_ALIAS;
  }
  const int sms = current_device_sms();
  if (sms <= 0) return PTI_ERR_CUDA;
  const unsigned grid = static_cast<unsigned>(std::min<int64_t>(steps, static_cast<int64_t>(sms) * 4));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (aligned(logits, 16) && vocab % 4 == 0)
    verify_greedy_kernel<true><<<grid, kVerifyThreads, 0, st>>>(logits, guess, steps, n_streams, vocab, argmax_out,
                                                                 match_out, accept_len_out);
  else
    verify_greedy_kernel<false><<<grid, kVerifyThreads, 0, st>>>(logits, guess, steps, n_streams, vocab,
                                                                  argmax_out, match_out, accept_len_out);
  return launch_status();
}
