// pti_verify.cu -- greedy and sampling-mode verify of self-speculative
// decoding on sm_103a.
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
#include <cmath>
#include <cstdint>

#include "pti.h"
#include "pti_device.cuh"
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

// ---------------------------------------------------------------------------
// Sampling-mode verify ([PTI-readme] §"接受机制如何工作", temperature > 0): each
// stream draws its token from p = softmax(logits / T) by inverse CDF with the
// supplied uniform u (the smallest v with p(0) + ... + p(v) > u); the guess
// fed to stream s+1 is accepted when it equals stream s's draw; the collision
// probability sum p^2 (the pages' acceptance rate) is returned per stream.
//
// One CTA per step.  Per row, warp w owns the contiguous segment
// [w L, (w+1) L) of the vocabulary (L a multiple of 4, so segments start on
// 16-byte boundaries).  Pass 1 streams the row once from HBM, four 16-byte
// loads in flight per lane, keeping per lane an online maximum m with the sums
// of 2^((x-m)c) and of its square (c = log2(e) / T, rescaled when m grows).
// The warps' results give the row maximum M, the normaliser Z, sum e^2 / Z^2
// and the segment masses.  The draw lies in the first segment whose running
// mass exceeds u Z; pass 2 reads only that segment again (from L2) with the
// whole block, each thread summing one contiguous run of it, then a
// block-wide inclusive prefix sum over the runs.  The first thread whose
// prefix exceeds the threshold walks its run again to the token.  (Float
// rounding can make two warps claim when the threshold sits on a run edge;
// the smaller token wins, so the result is deterministic.)
// Logits may hold -inf (masked tokens, mass 0); each row needs one finite
// logit.
// ---------------------------------------------------------------------------
constexpr int kSampleThreads = 512;
constexpr int kSampleWarps = kSampleThreads / 32;
constexpr int kSampleDepth = 4;  // 16-byte loads in flight per lane in pass 1
constexpr int kSampleBlocksPerSM = 3;  // resident CTAs per SM (40 registers a thread)

struct OnlineSums {
  float m, s, q;  // maximum, sum of 2^((x-m)c), sum of its square
};

// 2^x by the PTX ISA's ex2.approx.ftz.f32 instruction (a few ulp of relative
// error).  A result below 2^-126 flushes to zero, which drops only tokens
// whose probability is below 1e-38 of the most likely one.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// The unnormalised weights e = 2^((x - m) c) of four logits, as two packed
// pairs; x - m and the product by c are rounded like the scalar operations.
__device__ __forceinline__ void weights4(const float4 &v, uint64_t neg_m2, uint64_t c2, uint64_t &e01,
                                         uint64_t &e23) {
  const float2 a = unpack2(fmul2(fadd2(pack2(v.x, v.y), neg_m2), c2));
  const float2 b = unpack2(fmul2(fadd2(pack2(v.z, v.w), neg_m2), c2));
  e01 = pack2(ex2(a.x), ex2(a.y));
  e23 = pack2(ex2(b.x), ex2(b.y));
}

// One lane's running sums over its share of a segment, two packed lanes each.
struct LaneSums {
  float m;          // running maximum
  uint64_t neg_m2;  // (-m, -m)
  uint64_t s2, q2;  // sums of e and of e^2, relative to m
};

__device__ __forceinline__ void lane_add4(LaneSums &a, const float4 &v, uint64_t c2, float c) {
  const float mx = fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w));
  if (!(mx > -INFINITY)) return;  // four masked tokens (or padding): no mass
  if (mx > a.m) {
    const float r = ex2((a.m - mx) * c);  // a.m = -inf gives r = 0
    a.s2 = fmul2(a.s2, pack2(r, r));
    a.q2 = fmul2(a.q2, pack2(r * r, r * r));
    a.m = mx;
    a.neg_m2 = pack2(-mx, -mx);
  }
  uint64_t e01, e23;
  weights4(v, a.neg_m2, c2, e01, e23);
  a.s2 = fadd2(a.s2, e01);
  a.s2 = fadd2(a.s2, e23);
  a.q2 = ffma2(e01, e01, a.q2);
  a.q2 = ffma2(e23, e23, a.q2);
}

__device__ __forceinline__ OnlineSums online_merge(OnlineSums a, OnlineSums b, float c) {
  if (b.m > a.m) {
    const OnlineSums t = a;
    a = b;
    b = t;
  }
  if (!(b.m > -INFINITY)) return a;
  const float r = ex2((b.m - a.m) * c);
  a.s += b.s * r;
  a.q += b.q * (r * r);
  return a;
}

// Four logits from i on; positions at or past `end` read as -inf.  kVec: the
// row base is 16-byte aligned and i is a multiple of 4.
template <bool kVec>
__device__ __forceinline__ float4 load4(const float *row, int64_t i, int64_t end) {
  if (kVec && i + 3 < end) return __ldcg(reinterpret_cast<const float4 *>(row + i));
  float4 v;
  v.x = (i + 0 < end) ? __ldcg(row + i + 0) : -INFINITY;
  v.y = (i + 1 < end) ? __ldcg(row + i + 1) : -INFINITY;
  v.z = (i + 2 < end) ? __ldcg(row + i + 2) : -INFINITY;
  v.w = (i + 3 < end) ? __ldcg(row + i + 3) : -INFINITY;
  return v;
}

template <bool kVec>
__global__ void __launch_bounds__(kSampleThreads, kSampleBlocksPerSM)
    verify_sample_kernel(const float *__restrict__ logits, const int32_t *__restrict__ guess,
                         const float *__restrict__ uniform, int64_t steps, int n, int64_t vocab, float c,
                         int32_t *__restrict__ token_out, uint8_t *__restrict__ match_out,
                         int32_t *__restrict__ accept_out, float *__restrict__ collision_out) {
  __shared__ OnlineSums s_warp[kSampleWarps];
  __shared__ float s_scan[kSampleWarps];
  __shared__ int s_last[kSampleWarps];
  __shared__ int s_tok[4];
  __shared__ int s_seg;
  __shared__ float s_theta, s_max;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint64_t c2 = pack2(c, c);
  const int64_t seg = ((vocab + 4 * kSampleWarps - 1) / (4 * kSampleWarps)) * 4;
  const int64_t run_len = ((seg + 4 * kSampleThreads - 1) / (4 * kSampleThreads)) * 4;
  for (int64_t t = blockIdx.x; t < steps; t += gridDim.x) {
    for (int s = 0; s < n; ++s) {
      const float *row = logits + (t * n + s) * vocab;
      // ---- pass 1: this warp's segment, online maximum and sums
      const int64_t lo = warp * seg, hi = min(lo + seg, vocab);
      LaneSums ls{-INFINITY, pack2(INFINITY, INFINITY), 0, 0};
      // kSampleDepth loads in flight per lane, also in the segment's last
      // round (positions past its end read as -inf)
      for (int64_t i = lo + 4 * lane; i < hi; i += 32 * 4 * kSampleDepth) {
        float4 v[kSampleDepth];
#pragma unroll
        for (int d = 0; d < kSampleDepth; ++d) v[d] = load4<kVec>(row, i + 128 * d, hi);
#pragma unroll
        for (int d = 0; d < kSampleDepth; ++d) lane_add4(ls, v[d], c2, c);
      }
      const float2 s_pair = unpack2(ls.s2), q_pair = unpack2(ls.q2);
      OnlineSums a{ls.m, s_pair.x + s_pair.y, q_pair.x + q_pair.y};
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        OnlineSums b;
        b.m = __shfl_xor_sync(0xFFFFFFFFu, a.m, o);
        b.s = __shfl_xor_sync(0xFFFFFFFFu, a.s, o);
        b.q = __shfl_xor_sync(0xFFFFFFFFu, a.q, o);
        a = online_merge(a, b, c);
      }
      if (lane == 0) s_warp[warp] = a;
      __syncthreads();
      // ---- row maximum, normaliser, collision; the segment holding the draw
      if (warp == 0) {
        const OnlineSums w_sums = lane < kSampleWarps ? s_warp[lane] : OnlineSums{-INFINITY, 0.0f, 0.0f};
        float m = w_sums.m;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        const float r = (w_sums.m > -INFINITY) ? ex2((w_sums.m - m) * c) : 0.0f;
        float q = w_sums.q * (r * r);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) q += __shfl_xor_sync(0xFFFFFFFFu, q, o);
        if (lane < kSampleWarps) s_scan[lane] = w_sums.s * r;  // segment masses
        __syncwarp();
        if (lane == 0) {
          float z = 0.0f;
          int last_w = 0;
          for (int w = 0; w < kSampleWarps; ++w) {
            z += s_scan[w];
            if (s_scan[w] > 0.0f) last_w = w;
          }
          if (collision_out != nullptr) collision_out[t * n + s] = q / (z * z);
          const float theta = uniform[t * n + s] * z;
          // the first segment whose running mass passes theta (the running sum
          // repeats the one above term by term)
          float cum = 0.0f, below = 0.0f;
          int w = 0;
          for (; w < kSampleWarps; ++w) {
            below = cum;
            cum += s_scan[w];
            if (cum > theta) break;
          }
          s_seg = w < kSampleWarps ? w : last_w;
          // mass left to pass within the segment (>= 0); when u Z lies at the
          // end of the row within rounding, no run may claim and the draw is
          // the last token with mass
          s_theta = w < kSampleWarps ? theta - below : INFINITY;
          s_max = m;
          s_tok[s] = INT_MAX;
        }
      }
      __syncthreads();
      // ---- pass 2: the draw's segment again, thread k taking the k-th run of
      // cl tokens; a block-wide prefix sum finds the run holding the draw, and
      // that thread walks its run once more
      const int64_t slo = s_seg * seg, shi = min(slo + seg, vocab);
      const int64_t jlo = slo + tid * run_len, jhi = min(jlo + run_len, shi);
      const float theta = s_theta;
      const uint64_t neg_m2 = pack2(-s_max, -s_max);
      float own = 0.0f;
      int last = -1;  // last token of the run with mass (the rounding fallback)
      for (int64_t j0 = jlo; j0 < jhi; j0 += 4 * kSampleDepth) {
        float4 v[kSampleDepth];
#pragma unroll
        for (int d = 0; d < kSampleDepth; ++d) v[d] = load4<kVec>(row, j0 + 4 * d, jhi);
#pragma unroll
        for (int d = 0; d < kSampleDepth; ++d) {
          const int64_t j = j0 + 4 * d;
          uint64_t e01, e23;
          weights4(v[d], neg_m2, c2, e01, e23);
          const float2 a01 = unpack2(e01), a23 = unpack2(e23);
          own += (a01.x + a01.y) + (a23.x + a23.y);
          if (a23.y > 0.0f) last = static_cast<int>(j + 3);
          else if (a23.x > 0.0f) last = static_cast<int>(j + 2);
          else if (a01.y > 0.0f) last = static_cast<int>(j + 1);
          else if (a01.x > 0.0f) last = static_cast<int>(j);
        }
      }
      float incl = own;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += y;
      }
      float prev = __shfl_up_sync(0xFFFFFFFFu, incl, 1);
      if (lane == 0) prev = 0.0f;
      if (lane == 31) s_scan[warp] = incl;
      int lw = last;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) lw = max(lw, __shfl_xor_sync(0xFFFFFFFFu, lw, o));
      if (lane == 0) s_last[warp] = lw;
      __syncthreads();
      float before = 0.0f, total = 0.0f;
      for (int w = 0; w < kSampleWarps; ++w) {
        if (w == warp) before = total;
        total += s_scan[w];
      }
      const bool over = before + incl > theta;
      const unsigned ballot = __ballot_sync(0xFFFFFFFFu, over);
      if (over && !(before > theta) && lane == __ffs(ballot) - 1) {
        // the first thread of its warp whose prefix passes theta, in a warp whose
        // predecessors' total does not: its run holds the draw
        float cum = before + prev;
        int k = -1;
        for (int64_t j = jlo; j < jhi && k < 0; j += 4) {
          uint64_t e01, e23;
          weights4(load4<kVec>(row, j, jhi), neg_m2, c2, e01, e23);
          const float2 a01 = unpack2(e01), a23 = unpack2(e23);
          const float e[4] = {a01.x, a01.y, a23.x, a23.y};
          for (int d = 0; d < 4 && k < 0; ++d) {
            cum += e[d];
            if (cum > theta && e[d] > 0.0f) k = static_cast<int>(j + d);
          }
        }
        const int cand = k >= 0 ? k : last;
        if (cand >= 0) atomicMin(&s_tok[s], cand);
      }
      __syncthreads();
      if (tid == 0 && s_tok[s] == INT_MAX) {  // u Z at the segment's end within rounding
        int best = -1;
        for (int w = 0; w < kSampleWarps; ++w) best = max(best, s_last[w]);
        s_tok[s] = best >= 0 ? best : static_cast<int>(slo);
      }
      __syncthreads();
      if (tid == 0) token_out[t * n + s] = s_tok[s];
    }
    if (tid == 0) {
      int32_t accepted = 0;
      bool run = true;
      for (int s = 0; s + 1 < n; ++s) {
        const bool mtc = guess[t * n + s + 1] == s_tok[s];
        match_out[t * (n - 1) + s] = mtc ? 1 : 0;
        if (run && mtc) ++accepted;
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

extern "C" pti_status pti_verify_sample(const float *logits, const int32_t *guess, const float *uniform,
                                        int64_t steps, int n_streams, int64_t vocab, float temperature,
                                        int32_t *token_out, uint8_t *match_out, int32_t *accept_len_out,
                                        float *collision_out, pti_stream_t stream) {
  if (n_streams < 1 || n_streams > 4) return PTI_ERR_NSTREAMS;
  if (steps < 0 || vocab < 1 || vocab > INT_MAX) return PTI_ERR_SHAPE;
  if (steps > (int64_t{1} << 40) / (static_cast<int64_t>(n_streams) * vocab)) return PTI_ERR_SHAPE;
  if (!(temperature > 0.0f) || !std::isfinite(temperature)) return PTI_ERR_VALUE;
  const float c = static_cast<float>(1.4426950408889634 / static_cast<double>(temperature));  // log2(e) / T
  if (!std::isfinite(c)) return PTI_ERR_VALUE;
  if (steps == 0) return PTI_OK;
  if (logits == nullptr || guess == nullptr || uniform == nullptr || token_out == nullptr ||
      accept_len_out == nullptr || (n_streams > 1 && match_out == nullptr))
    return PTI_ERR_NULL;
  if (!aligned(logits, 4) || !aligned(guess, 4) || !aligned(uniform, 4) || !aligned(token_out, 4) ||
      !aligned(accept_len_out, 4) || !aligned(collision_out, 4))
    return PTI_ERR_ALIGN;
  const uint64_t l_bytes = static_cast<uint64_t>(steps) * n_streams * vocab * 4;
  const uint64_t g_bytes = static_cast<uint64_t>(steps) * n_streams * 4;
  const void *ins[3] = {logits, guess, uniform};
  const uint64_t in_bytes[3] = {l_bytes, g_bytes, g_bytes};
  void *outs[4] = {token_out, match_out, accept_len_out, collision_out};
  const uint64_t out_bytes[4] = {g_bytes, n_streams > 1 ? static_cast<uint64_t>(steps) * (n_streams - 1) : 0,
                                 static_cast<uint64_t>(steps) * 4, collision_out ? g_bytes : 0};
  for (int i = 0; i < 4; ++i) {
    for (int j = 0; j < 3; ++j)
      if (overlaps(outs[i], out_bytes[i], ins[j], in_bytes[j])) return PTI_ERR_ALIAS;
    for (int j = i + 1; j < 4; ++j)
      if (overlaps(outs[i], out_bytes[i], outs[j], out_bytes[j])) return PTI_ERR_ALIAS;
  }
  const int sms = current_device_sms();
  if (sms <= 0) return PTI_ERR_CUDA;
  const bool vec = aligned(logits, 16) && vocab % 4 == 0;
  auto kernel = vec ? verify_sample_kernel<true> : verify_sample_kernel<false>;
  // one wave of resident CTAs, each taking every grid-th step
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kSampleThreads, 0) != cudaSuccess || per_sm < 1)
    return PTI_ERR_CUDA;
  const unsigned grid = static_cast<unsigned>(std::min<int64_t>(steps, static_cast<int64_t>(sms) * per_sm));
  kernel<<<grid, kSampleThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      logits, guess, uniform, steps, n_streams, vocab, c, token_out, match_out, accept_len_out, collision_out);
  return launch_status();
}
