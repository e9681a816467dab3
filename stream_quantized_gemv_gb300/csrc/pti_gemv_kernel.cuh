// pti_gemv_kernel.cuh -- the persistent TMA GEMV kernel (N-stream Q8 and SSQ
// "mode 16" twin) and its host-side launch helpers, shared by the plain GEMV
// entry points (pti_gemv.cu) and the chained decode pass (pti_decode.cu).
//
// Both GEMVs stream each weight byte from HBM exactly once and use it for every
// activation stream it serves: the N streams of the Q8 kernel ([PTI-readme]
// "打包双子推理（PTI）" §"带宽分析：为什么会有开销", a kernel that loads each
// weight group once and forms N dot products together) or the two models packed
// in one uint16 of the twin kernel ([PTI-readme] §"与 SSQ（Side-by-Side
// Quantization）的关系"; [PTI-forum] "Packed Twin Inference：无需草稿模型的推测解码
// 新方案，实现2倍吞吐量提升" §"PTI的核心创新：SSQ打包技术").
//
// Fast-path design (cols % 256 == 0 for Q8, cols % 128 == 0 for twin):
//  * A row is a sequence of 272-byte super-blocks (8 Q8 blocks = 256 columns,
//    or 4 twin blocks = 128 columns), i.e. 17 aligned 16-byte chunks.  Work is
//    cut into units of (128-row tile, super-block); one TMA 2-D tile copy
//    (box 34 x 8 bytes by 128 rows) brings a unit into shared memory.
//  * Persistent grid, one CTA per SM, stream-K split: CTA c owns the units
//    [c U / G, (c+1) U / G) in row-major order, so every SM streams the same
//    number of bytes.  Row tiles shared by several CTAs are combined by a
//    small kernel launched right behind the GEMV (partials in a
//    caller-supplied workspace, summed in a fixed CTA order).
//  * Lane 0 of the producer warp issues the copies into a ring of up to 6
//    stages guarded by mbarriers (it refills a slot once every consumer warp
//    has released it).
//  * Q8 (16 consumer warps): warp w always computes block w % 8 of each unit
//    for 64 rows (two per lane), reading each row's 40-byte window around
//    the block with five aligned 8-byte loads; the four warps of a scheduler
//    share one code body.
//  * Twin (16 consumer warps): warp w computes half of block w % 4 (16
//    columns of both models) of each unit for 64 rows, two per lane; the
//    block is fixed per scheduler, so its byte offsets are compile-time.
//  * Each stage also holds the unit's slice of the activations (N x 1 KB,
//    stream-major), fetched by one bulk copy per stream next to the weight
//    tile, so activation traffic is one slice per unit and does not grow
//    with the number of rows (the L2 thrash the pages diagnose for the
//    per-row-block design comes from re-reading x once per row block).
//  * Dequantisation is exact (see pti_device.cuh); products use packed
//    f32x2 FMAs.  A lane's products of one block and unit are summed into a
//    fresh partial (16 Q8 or 8 twin products per half of the f32x2 pair),
//    which is then added to the running accumulator once per unit, so an
//    output's longest chain of dependent roundings is about K/256 (Q8) or
//    K/128 (twin) plus a few dozen.
//  * Programmatic dependent launch: the producer fetches its first weight
//    tiles before waiting for the previous kernel in the stream, and only then
//    fetches activations; nothing is written before that wait.
//  * On request (PTI_FLAG_TENSOR_CORES) the Q8 kernel's products run on the
//    tensor core instead: gemv_tc_kernel in pti_gemv_tc.cuh, the same ring,
//    producer and tile finishing with a converter/MMA consumer side.
//  * Epilogue modes (template parameter Epi) fuse the decode pass's glue into
//    the tile epilogue: Plain writes y; GateUp reads 64 gate rows and the 64
//    matching up rows into one tile and writes h = SiLU(b g) * (b u); Down
//    writes a x' = a (W_down h).  b and a are the RMS scales of the input
//    vectors, computed from per-tile sums of squares that the previous kernel
//    wrote, and each mode writes the per-tile sums of squares of its own output.
// Other shapes use a plain per-row kernel (pti_gemv.cu).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "pti.h"
#include "pti_device.cuh"
#include "pti_host.h"

namespace pti {
namespace {

constexpr int kSBBytes = 272;                          // super-block bytes (17 chunks of 16)
constexpr int kRowsPerTile = 128;                      // rows per unit
constexpr int kMaxStages = 6;
constexpr int kStageBytes = kRowsPerTile * kSBBytes;   // 34816
constexpr int kMaxGrid = 320;
constexpr int kSmemOptin = 232448;                     // 227 KB per CTA
constexpr uint32_t kBarConsumers = 1;                  // named barrier of the consumer warps
constexpr int kRedWarps = 8;                           // warps whose sums make up one output element

__device__ unsigned int g_device_error = 0;

enum class Fmt : int { Q8 = 0, Twin = 1 };

// Tile epilogue: plain GEMV output, or one of the decode pass's fused glue
// steps (see the file comment).
enum class Epi : int { Plain = 0, GateUp = 1, Down = 2 };

// Shared memory of the fused epilogues: the tile's sums [kOut][128], the RMS
// scale of each input vector, and one partial sum of squares per warp.
constexpr int kEpiBytes = (4 * kRowsPerTile + 4 + 16) * 4;

template <Fmt F, int N>
struct Traits;
template <int N>
struct Traits<Fmt::Q8, N> {
  static constexpr int kOut = N;                   // output vectors
  static constexpr int kWarps = 16;                // four per scheduler
  static constexpr int kColsPerSB = 256;
  static constexpr int kXStreams = N;
  static constexpr int kBlockBytes = 34;
};
// Twin: N activation streams per model (model A's streams first, then B's).
template <int N>
struct Traits<Fmt::Twin, N> {
  static constexpr int kOut = 2 * N;
  static constexpr int kWarps = 16;                // four per scheduler
  static constexpr int kColsPerSB = 128;
  static constexpr int kXStreams = 2 * N;
  static constexpr int kBlockBytes = 68;
};

// One pipeline stage: the 128 x 272-byte weight tile followed by the unit's
// activations, stream-major (kXStreams rows of kColsPerSB floats).  kRedBytes:
// the parked sums of two row tiles, kRedWarps per output element.
template <Fmt F, int N>
struct Stage {
  static constexpr int kXStreamBytes = Traits<F, N>::kColsPerSB * 4;
  static constexpr int kXBytes = Traits<F, N>::kXStreams * kXStreamBytes;
  static constexpr int kBytes = ((kStageBytes + kXBytes) + 1023) / 1024 * 1024;
  static constexpr int kRedBytes = 2 * kRedWarps * Traits<F, N>::kOut * kRowsPerTile * 4;
};

struct GemvArgs {
  const float *x0;  // Q8: x [N][cols]; twin: x_a [N][cols]
  const float *x1;  // twin: x_b [N][cols]
  float *y0;        // Q8: y [N][rows]; twin: y_a [N][rows]
  float *y1;        // twin: y_b [N][rows]
  float *part;      // workspace: [grid][2 slots][kOut][128] partial sums
  int64_t rows, cols, units;  // GateUp: rows = gate rows = up rows = outputs per stream
  int32_t n_sb, n_rb, grid, stages;
  // Fused epilogues only (Epi::GateUp, Epi::Down):
  const float *sq_in;  // [n_sq_in][kOut] per-tile sums of squares of the input vectors; null: scale 1
  float *sq_out;       // [n_rb][kOut] per-tile sums of squares of the output vectors
  double inv_len_in;   // 1 / length of each input vector
  double eps;          // added to the mean square before the square root
  int32_t n_sq_in;
  // Fused epilogues of the chained pass: the input scales the GEMV derived, for
  // its tile-combine kernel ([kOut] floats, written by CTA 0).
  float *scale_out;
  int32_t prefetch_all;  // 1: fetch every initial stage's weights before waiting for the previous kernel
  // Pipeline waits give up after this many ns (0: kWaitTimeoutNs).
  uint64_t wait_ns = 0;
  // Testing only: the producer of CTA 0 issues no copy from its unit
  // `stall_unit` on (-1: never; must be at least the ring depth), as if the
  // copy never arrived; the consumers' wait for it then runs out after
  // wait_ns.
  int64_t stall_unit = -1;
};

__device__ __forceinline__ uint64_t wait_limit(const GemvArgs &a) {
  return a.wait_ns != 0 ? a.wait_ns : kWaitTimeoutNs;
}

// ---------------------------------------------------------------------------
// Q8 consumer (16 warps).  Warp w computes block B = w % 8 of every unit
// (columns 32B .. 32B+31, the block's 34 bytes at row byte 34B = 32B + 2B)
// for the 64 rows of half hf = w / 8, two rows per lane (64 hf + l and
// 64 hf + 32 + l).  With B = 2c + e, the 40-byte window that starts at byte
// 32B + 8 [c >= 2] of the row (five aligned 8-byte loads; B is fixed per
// warp, so the offset is loop-invariant) holds the block from word c % 2 on,
// at half-word e: the scale is half-word e of that word, weight pair j
// (columns 32B+2j, 32B+2j+1) is at byte 2e+2+2j.  The warps of a scheduler
// (w % 4) share c % 2 and e (template parameters E and CLO), so they run one
// code body.  (Five 8-byte loads replace three 16-byte loads and ten selects:
// measured 5% faster at N = 4, 7% at N = 1.)
//
// Activations are warp-broadcast 16-byte loads (two weight pairs of one
// stream) reused across the lane's two rows; each weight pair is dequantised
// to q d exactly (dequant2) and its products with the N activation pairs go
// to a fresh partial (16 dependent FMAs per half of the pair), which is added
// to the row's accumulator once per unit.
// ---------------------------------------------------------------------------
template <int N, int E, int CLO>
struct Q8Pair {
  static constexpr int kSlots = 2;
  uint64_t acc[kSlots][N];
  uint32_t lane, half, blk;

  __device__ __forceinline__ void init(uint32_t warp, uint32_t lane_) {
    lane = lane_;
    half = warp >> 3;
    blk = warp & 7u;
  }

  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int r = 0; r < kSlots; ++r)
#pragma unroll
      for (int s = 0; s < N; ++s) acc[r][s] = 0ull;
  }

  template <int kXS>
  __device__ __forceinline__ void unit(const uint8_t *tile, const uint8_t *xsb) {
    const uint8_t *xblk = xsb + 128u * blk;  // block B's 32 activations of stream 0
    const uint32_t win_off = 32u * blk + ((blk & 4u) != 0u ? 8u : 0u);
    uint32_t w[kSlots][9];
    ScalePair sc[kSlots];
#pragma unroll
    for (int r = 0; r < kSlots; ++r) {
      const uint8_t *win = tile + (half * 64 + r * 32 + lane) * kSBBytes + win_off;
      uint32_t t1[10];
#pragma unroll
      for (int k = 0; k < 5; ++k) {
        const uint2 v = *reinterpret_cast<const uint2 *>(win + 8 * k);
        t1[2 * k] = v.x;
        t1[2 * k + 1] = v.y;
      }
#pragma unroll
      for (int k = 0; k < 9; ++k) w[r][k] = t1[k + CLO];
      sc[r] = make_scale(E ? (w[r][0] >> 16) : (w[r][0] & 0xFFFFu));
#pragma unroll
      for (int k = 0; k < 9; ++k) w[r][k] ^= 0x80808080u;
    }
    uint64_t p[kSlots][N];
    static_for<0, 8>([&](auto jc) {  // two weight pairs per step: one 16-byte x load per stream
      constexpr int j0 = 2 * decltype(jc)::value;
      ulonglong2 xv[N];
#pragma unroll
      for (int st = 0; st < N; ++st) xv[st] = *reinterpret_cast<const ulonglong2 *>(xblk + st * kXS + j0 * 8);
      static_for<0, 2>([&](auto jj_) {
        constexpr int j = j0 + decltype(jj_)::value;
        constexpr int t = 2 * E + 2 + 2 * j;  // byte of the pair's first weight in the aligned words
#pragma unroll
        for (int r = 0; r < kSlots; ++r) {
          const uint64_t wq = dequant2(w[r][t / 4], t % 4, w[r][t / 4], t % 4 + 1, sc[r]);
#pragma unroll
          for (int st = 0; st < N; ++st) {
            const uint64_t xs = (j & 1) ? xv[st].y : xv[st].x;
            if constexpr (j == 0) p[r][st] = fmul2(wq, xs);
            else p[r][st] = ffma2(wq, xs, p[r][st]);
          }
        }
      });
    });
#pragma unroll
    for (int r = 0; r < kSlots; ++r)
#pragma unroll
      for (int st = 0; st < N; ++st) acc[r][st] = fadd2(acc[r][st], p[r][st]);
  }

  // End of a row tile: red[sl][warp][s][row of the half] (64 rows per warp).
  template <int kOut>
  __device__ __forceinline__ void park(float *red, int sl, uint32_t warp) const {
#pragma unroll
    for (int r = 0; r < kSlots; ++r)
#pragma unroll
      for (int s = 0; s < kOut; ++s) {
        const float2 v = unpack2(acc[r][s]);
        red[((sl * 16 + static_cast<int>(warp)) * kOut + s) * 64 + r * 32 + static_cast<int>(lane)] = v.x + v.y;
      }
  }
};

// ---------------------------------------------------------------------------
// Twin consumer.  Warp w computes columns 16ch .. 16ch+15 (ch = w / 8) of
// block B = w % 4 of the super-block, both models, for the 64 rows of half
// hf = (w / 4) % 2, two rows per lane (64 hf + l and 64 hf + 32 + l).  The
// block's scale word (binary16 scale of A, then of B) is at byte 68B; payload
// word k (columns 2k, 2k+1) at 68B + 4 + 4k holds the bytes
// [B(2k), A(2k), B(2k+1), A(2k+1)] (each uint16 is A << 8 | B, stored
// little-endian).  The warp's eight payload words start (68B + 4) % 16 bytes
// past a 16-byte boundary: two or three aligned 16-byte loads, with B (= the
// warp's scheduler) a compile-time constant, plus one 4-byte load of the
// scales.  Products go to fresh partials per unit (8 dependent FMAs per half
// of the pair), added to the accumulators once per unit.
// ---------------------------------------------------------------------------
template <int N, int B>
struct TwinSlab {
  static constexpr int kSlots = 2;
  uint64_t acc[kSlots][2 * N];
  uint32_t lane, half, ch;

  __device__ __forceinline__ void init(uint32_t warp, uint32_t lane_) {
    lane = lane_;
    half = (warp >> 2) & 1u;
    ch = warp >> 3;
  }

  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int r = 0; r < kSlots; ++r)
#pragma unroll
      for (int s = 0; s < 2 * N; ++s) acc[r][s] = 0ull;
  }

  template <int kXS>
  __device__ __forceinline__ void unit(const uint8_t *tile, const uint8_t *xsb) {
    constexpr int kP = (68 * B + 4) % 16;         // payload offset past the 16-byte boundary
    constexpr int kChunks = (kP + 32 + 15) / 16;  // 16-byte loads covering the 32 payload bytes
    uint32_t w[kSlots][8];
    ScalePair sa[kSlots], sb[kSlots];
#pragma unroll
    for (int r = 0; r < kSlots; ++r) {
      const uint8_t *row = tile + (half * 64 + r * 32 + lane) * kSBBytes;
      const uint32_t scales = *reinterpret_cast<const uint32_t *>(row + 68 * B);
      const uint8_t *pl = row + (68 * B + 4 - kP) + 32 * ch;
      uint32_t words[4 * kChunks];
#pragma unroll
      for (int c = 0; c < kChunks; ++c) {
        const uint4 v = *reinterpret_cast<const uint4 *>(pl + 16 * c);
        words[4 * c] = v.x;
        words[4 * c + 1] = v.y;
        words[4 * c + 2] = v.z;
        words[4 * c + 3] = v.w;
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) w[r][k] = words[kP / 4 + k] ^ 0x80808080u;
      sa[r] = make_scale(scales & 0xFFFFu);
      sb[r] = make_scale(scales >> 16);
    }
    const uint8_t *xcol = xsb + (32 * B) * 4 + ch * 64;  // column 32B + 16ch of stream 0
    uint64_t pa[kSlots][N], pb[kSlots][N];
    static_for<0, 4>([&](auto jc) {  // two payload words (four columns) per step
      constexpr int k0 = 2 * decltype(jc)::value;
      ulonglong2 xa[N], xb[N];
#pragma unroll
      for (int s = 0; s < N; ++s) {
        xa[s] = *reinterpret_cast<const ulonglong2 *>(xcol + s * kXS + k0 * 8);
        xb[s] = *reinterpret_cast<const ulonglong2 *>(xcol + (N + s) * kXS + k0 * 8);
      }
      static_for<0, 2>([&](auto kk_) {
        constexpr int kk = decltype(kk_)::value;
        constexpr int k = k0 + kk;
#pragma unroll
        for (int r = 0; r < kSlots; ++r) {
          // bytes 1 and 3 of a payload word are model A's weights, 0 and 2 model B's
          const uint64_t wa = dequant2(w[r][k], 1, w[r][k], 3, sa[r]);
          const uint64_t wb = dequant2(w[r][k], 0, w[r][k], 2, sb[r]);
#pragma unroll
          for (int s = 0; s < N; ++s) {
            const uint64_t x_a = kk ? xa[s].y : xa[s].x;
            const uint64_t x_b = kk ? xb[s].y : xb[s].x;
            if constexpr (k == 0) {
              pa[r][s] = fmul2(wa, x_a);
              pb[r][s] = fmul2(wb, x_b);
            } else {
              pa[r][s] = ffma2(wa, x_a, pa[r][s]);
              pb[r][s] = ffma2(wb, x_b, pb[r][s]);
            }
          }
        }
      });
    });
#pragma unroll
    for (int r = 0; r < kSlots; ++r)
#pragma unroll
      for (int s = 0; s < N; ++s) {
        acc[r][s] = fadd2(acc[r][s], pa[r][s]);
        acc[r][N + s] = fadd2(acc[r][N + s], pb[r][s]);
      }
  }

  // End of a row tile: red[sl][warp][s][row of the half] (64 rows per warp).
  template <int kOut>
  __device__ __forceinline__ void park(float *red, int sl, uint32_t warp) const {
#pragma unroll
    for (int r = 0; r < kSlots; ++r)
#pragma unroll
      for (int s = 0; s < kOut; ++s) {
        const float2 v = unpack2(acc[r][s]);
        red[((sl * 16 + static_cast<int>(warp)) * kOut + s) * 64 + r * 32 + static_cast<int>(lane)] = v.x + v.y;
      }
  }
};

__device__ __forceinline__ int32_t cta_of_unit(int64_t u, int64_t units, int32_t grid) {
  return static_cast<int32_t>(((u + 1) * grid - 1) / units);
}

__device__ __forceinline__ int32_t first_tile_of_cta(int32_t c, int64_t units, int32_t grid, int32_t n_sb) {
  return static_cast<int32_t>((static_cast<int64_t>(c) * units / grid) / n_sb);
}

// Pairwise (tree) sum of K values in a fixed order.
template <int K>
__device__ __forceinline__ float tree_sum(float (&t)[K]) {
#pragma unroll
  for (int n = K; n > 1; n = (n + 1) / 2) {
#pragma unroll
    for (int i = 0; i < n / 2; ++i) t[i] = t[2 * i] + t[2 * i + 1];
    if (n % 2) t[n / 2] = t[n - 1];
  }
  return t[0];
}

// Sum of v over the warp, in a fixed butterfly order (the result of lane 0 is
// the same wherever the same values are summed).
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

// RMS scale 1 / sqrt(mean + eps) of a vector whose sum of squares is s2 (in
// double), rounded to float.  A float reciprocal square root (relative error
// below 2^-21) refined by one Newton step in double leaves a relative error
// near 1e-13 before the final rounding, so the float result is the correctly
// rounded scale except for values within that distance of a rounding
// boundary (then it is one ulp away).  This replaces a double square root and
// division: this GPU's double-precision unit is slow, and the scale sits on
// the path from one decode step to the next.  A zero or non-finite argument
// takes the plain formula.
__device__ __forceinline__ float rms_inv_scale(double s2, double inv_len, double eps) {
  const double m = s2 * inv_len + eps;
  const float r0 = rsqrtf(static_cast<float>(m));
  if (!(r0 > 0.0f) || !isfinite(r0) || !(m > 0.0)) return static_cast<float>(1.0 / sqrt(m));
  const double r = static_cast<double>(r0);
  return static_cast<float>(r * fma(-0.5 * m * r, r, 1.5));
}

// Staging of the fused epilogues' input sums: the per-tile sums of squares of
// the previous kernel's output ([n_sq_in][kOut] floats) are bulk-copied into
// a kSqStageBytes buffer of shared memory right after the wait on that
// kernel.  The copy is rounded up to 16 bytes; the workspace pads every such
// array to 256 bytes, so the few bytes past its end are still workspace.
// Returns 0 when there is nothing to stage (no input sums, or more than the
// buffer holds: then the sums are read from global memory).
constexpr int kSqStageBytes = 4608;  // 288 tiles of 4 streams

template <int kOut>
__device__ __forceinline__ uint32_t staged_sum_bytes(const GemvArgs &a) {
  if (a.sq_in == nullptr) return 0u;
  const uint32_t bytes = (static_cast<uint32_t>(a.n_sq_in) * kOut * 4u + 15u) & ~15u;
  return bytes <= static_cast<uint32_t>(kSqStageBytes) ? bytes : 0u;
}

// Float-float accumulator: the pair (hi, lo) holds the value hi + lo exactly
// as long as no term is lost (Knuth's TwoSum makes each addition error-free;
// the error terms are gathered in lo), which keeps the sum of a few hundred
// positive floats to within a few 1e-15 relative (checked against exact
// rational sums), on the single-precision pipe.
struct F2Sum {
  float hi, lo;
};

__device__ __forceinline__ F2Sum f2_add(F2Sum x, float h2, float l2) {
  const float s = x.hi + h2;
  const float bb = s - x.hi;
  const float e = (x.hi - (s - bb)) + (h2 - bb);  // x.hi + h2 == s + e exactly
  const float t = e + (x.lo + l2);
  const float hi = s + t;
  return F2Sum{hi, t - (hi - s)};
}

// RMS scale of input vector s, 1 / sqrt(mean(v^2) + eps), from the previous
// kernel's per-tile sums of squares (staged in shared memory at `stage`, or
// read from global memory when stage == 0), computed by one warp in a fixed
// order, so every CTA derives the same scale; 1 when there are none.  Lane l
// accumulates tiles l, l + 32, ... in a float-float sum, a fixed butterfly
// combines the lanes, and the mean and scale are formed in double.  (This
// GPU's double-precision pipe is slow, in latency and in throughput; the sum
// runs on the single-precision pipe instead.)  Lane 0 writes scale[s].
template <int kOut>
__device__ __noinline__ void input_scale_of_stream(const GemvArgs &a, uint32_t stage, uint32_t s, uint32_t lane,
                                                   float *scale) {
  F2Sum acc{0.0f, 0.0f};
  if (a.sq_in != nullptr) {
    if (stage != 0u) {
      for (int32_t t = static_cast<int32_t>(lane); t < a.n_sq_in; t += 32)
        acc = f2_add(acc, __uint_as_float(lds32(stage + (static_cast<uint32_t>(t) * kOut + s) * 4u)), 0.0f);
    } else {
      for (int32_t t = static_cast<int32_t>(lane); t < a.n_sq_in; t += 32)
        acc = f2_add(acc, __ldcg(a.sq_in + static_cast<int64_t>(t) * kOut + s), 0.0f);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float h2 = __shfl_xor_sync(0xFFFFFFFFu, acc.hi, o);
    const float l2 = __shfl_xor_sync(0xFFFFFFFFu, acc.lo, o);
    acc = f2_add(acc, h2, l2);
  }
  if (lane == 0) {
    const double s2 = static_cast<double>(acc.hi) + static_cast<double>(acc.lo);
    scale[s] = a.sq_in != nullptr ? rms_inv_scale(s2, a.inv_len_in, a.eps) : 1.0f;
  }
}

// Decode-pass epilogue of gate/up tile rb: the tile's rows 0..63 are gate rows
// 64 rb + p, rows 64..127 the matching up rows.  With b the input's RMS scale,
// h = SiLU(b g) (b u) (W (b x) = b (W x)); writes h [kOut][rows] and the
// tile's sum of h^2 per vector.
template <int kOut>
__device__ __forceinline__ void gateup_epilogue(const GemvArgs &a, const float *tile_out, const float *scale,
                                                float *wsum, int32_t rb, uint32_t tid, uint32_t consumer_threads) {
  float h = 0.0f;
  if (tid < static_cast<uint32_t>(kOut * 64)) {
    const int s = static_cast<int>(tid >> 6), p = static_cast<int>(tid & 63u);
    const int64_t row = static_cast<int64_t>(rb) * 64 + p;
    if (row < a.rows) {
      const float g = tile_out[s * kRowsPerTile + p] * scale[s];
      const float u = tile_out[s * kRowsPerTile + 64 + p] * scale[s];
      h = g / (1.0f + expf(-g)) * u;
      a.y0[s * a.rows + row] = h;
    }
  }
  const uint32_t warp = tid >> 5;
  if (warp < static_cast<uint32_t>(2 * kOut)) {
    const float v = warp_sum(h * h);
    if ((tid & 31u) == 0) wsum[warp] = v;
  }
  named_barrier(kBarConsumers, consumer_threads);
  if (tid < static_cast<uint32_t>(kOut)) a.sq_out[static_cast<int64_t>(rb) * kOut + tid] = wsum[2 * tid] + wsum[2 * tid + 1];
}

// Decode-pass epilogue of down tile rb: x' = a (W h) with a the RMS scale of
// h; writes x' [kOut][rows] and the tile's sum of x'^2 per vector.  Element
// e = (s, r) = (e / 128, e % 128) is handled by thread e % threads; the sums
// of squares are formed per group of 32 elements (a warp's share) and then
// over the 4 groups of a vector, in the same order for any thread count.
template <int kOut>
__device__ __forceinline__ void down_epilogue(const GemvArgs &a, const float *tile_out, const float *scale,
                                              float *wsum, int32_t rb, uint32_t tid, uint32_t consumer_threads) {
  for (uint32_t e0 = 0; e0 < static_cast<uint32_t>(kOut * kRowsPerTile); e0 += consumer_threads) {
    const uint32_t e = e0 + tid;
    float v = 0.0f;
    if (e < static_cast<uint32_t>(kOut * kRowsPerTile)) {
      const int s = static_cast<int>(e >> 7), r = static_cast<int>(e & 127u);
      const int64_t row = static_cast<int64_t>(rb) * kRowsPerTile + r;
      if (row < a.rows) {
        v = tile_out[s * kRowsPerTile + r] * scale[s];
        a.y0[s * a.rows + row] = v;
      }
    }
    if ((e0 >> 5) + (tid >> 5) < static_cast<uint32_t>(4 * kOut)) {
      const float q = warp_sum(v * v);
      if ((tid & 31u) == 0) wsum[e >> 5] = q;
    }
  }
  named_barrier(kBarConsumers, consumer_threads);
  if (tid < static_cast<uint32_t>(kOut))
    a.sq_out[static_cast<int64_t>(rb) * kOut + tid] =
        (wsum[4 * tid] + wsum[4 * tid + 1]) + (wsum[4 * tid + 2] + wsum[4 * tid + 3]);
}

// Sum over the kRedWarps warps that computed element (s, row) of the parked
// tile in slot sl (red[sl][warp][s][row % 64]), as a fixed tree.  Q8: warp
// w computed block w % 8 for the rows of half w / 8.  Twin: warp w computed
// columns 16 (w / 8) .. 16 (w / 8) + 15 of block w % 4 for the rows of half
// (w / 4) % 2.
template <Fmt F, int kOut>
__device__ __forceinline__ float warp_total(const float *red, int sl, int s, int row) {
  float v[kRedWarps];
#pragma unroll
  for (int q = 0; q < kRedWarps; ++q) {
    const int w = F == Fmt::Q8 ? 8 * (row >> 6) + q : (q >> 2) * 8 + (row >> 6) * 4 + (q & 3);
    v[q] = red[((sl * 16 + w) * kOut + s) * 64 + (row & 63)];
  }
  return tree_sum(v);
}

// Totals policy of the CUDA-core consumers: kRedWarps parked warp sums per
// element, 16 consumer warps.
template <Fmt F>
struct WarpTotals {
  static constexpr int kThreads = 16 * 32;
  template <int kOut>
  __device__ __forceinline__ static float total(const float *red, int sl, int s, int row) {
    return warp_total<F, kOut>(red, sl, s, row);
  }
};

// Total of element (s, row) of shared tile rb: the partials of its CTAs
// c_lo .. c_hi added in CTA order, so the result does not depend on which CTA
// or kernel adds them.  Each CTA's partial sits in slot 0 if rb is its first
// tile, else slot 1: the CTAs after c_lo start inside tile rb, so only c_lo
// can hold it in slot 1 (`lo_slot`).  The loads of up to kPartialBatch
// contributors are issued together.
constexpr int kPartialBatch = 8;

template <int kOut>
__device__ __forceinline__ float sum_partials(const GemvArgs &a, int32_t c_lo, int32_t c_hi, int lo_slot, int s,
                                              int row) {
  float total = 0.0f;
  for (int32_t c0 = c_lo; c0 <= c_hi; c0 += kPartialBatch) {
    float v[kPartialBatch];
#pragma unroll
    for (int k = 0; k < kPartialBatch; ++k) {
      const int32_t c = c0 + k;
      const int cs = c == c_lo ? lo_slot : 0;
      v[k] = c <= c_hi ? __ldcg(&a.part[((static_cast<int64_t>(c) * 2 + cs) * kOut + s) * kRowsPerTile + row]) : 0.0f;
    }
#pragma unroll
    for (int k = 0; k < kPartialBatch; ++k)
      if (c0 + k <= c_hi) total = (c0 + k == c_lo) ? v[k] : total + v[k];
  }
  return total;
}

__device__ __forceinline__ int partial_slot_of_first(int32_t rb, int32_t c_lo, const GemvArgs &a) {
  return rb == first_tile_of_cta(c_lo, a.units, a.grid, a.n_sb) ? 0 : 1;
}

// Writes element (s, row) of tile rb: y for Plain, else the epilogue's tile
// buffer.
template <Fmt F, int N, Epi E>
__device__ __forceinline__ void deliver(const GemvArgs &a, float *tile_out, int32_t rb, int s, int row, float total) {
  if constexpr (E == Epi::Plain) {
    const int64_t row_g = static_cast<int64_t>(rb) * kRowsPerTile + row;
    if (row_g < a.rows) {
      if constexpr (F == Fmt::Q8) a.y0[s * a.rows + row_g] = total;
      else if (s < N) a.y0[s * a.rows + row_g] = total;  // model A's streams, then B's
      else a.y1[(s - N) * a.rows + row_g] = total;
    }
  } else {
    tile_out[s * kRowsPerTile + row] = total;
  }
}

template <int kOut, Epi E>
__device__ __forceinline__ void run_epilogue(const GemvArgs &a, float *epi, int32_t rb, uint32_t tid,
                                             uint32_t threads) {
  float *const scale = epi + 4 * kRowsPerTile;
  if constexpr (E == Epi::GateUp) gateup_epilogue<kOut>(a, epi, scale, scale + 4, rb, tid, threads);
  else if constexpr (E == Epi::Down) down_epilogue<kOut>(a, epi, scale, scale + 4, rb, tid, threads);
}

// Finishes one or two row tiles of the CTA: tile k (row tile rb[k], parked
// sums in red slot sl[k]).  Each element's total is formed from its parked
// sums by the consumer's totals policy Tot (Tot::kThreads consumer threads).  A tile no other CTA shares is written out directly
// (Plain) or through the fused epilogue.  A shared tile's totals go to this
// CTA's partial slot in the workspace, and a separate kernel
// (combine_tiles_kernel) adds the partials of every shared tile once the GEMV
// has completed, so a CTA leaves the SM right after its last tile.  Not
// inlined: it runs a few times per CTA, and one shared copy keeps the consumer
// loops' instruction footprint small.
template <Fmt F, int N, Epi E, class Tot>
__device__ __noinline__ void finish_tiles(const GemvArgs &a, const float *red, int count, int32_t rb0, int sl0,
                                          int32_t rb1, int sl1, uint32_t tid, float *epi) {
  using T = Traits<F, N>;
  constexpr int kOut = T::kOut;
  constexpr int kConsumerThreads = Tot::kThreads;
  const int32_t rbs[2] = {rb0, rb1};
  const int sls[2] = {sl0, sl1};
  bool epilogue_ran = false;
  for (int k = 0; k < count; ++k) {
    const int32_t clo = cta_of_unit(static_cast<int64_t>(rbs[k]) * a.n_sb, a.units, a.grid);
    const int32_t chi = cta_of_unit(static_cast<int64_t>(rbs[k] + 1) * a.n_sb - 1, a.units, a.grid);
    if (chi > clo) {  // shared tile: publish this CTA's partials
      for (int t = tid; t < kOut * kRowsPerTile; t += kConsumerThreads) {
        const int s = t / kRowsPerTile, row = t - s * kRowsPerTile;
        a.part[((static_cast<int64_t>(blockIdx.x) * 2 + sls[k]) * kOut + s) * kRowsPerTile + row] =
            Tot::template total<kOut>(red, sls[k], s, row);
      }
      continue;
    }
    if constexpr (E != Epi::Plain)
      if (epilogue_ran) named_barrier(kBarConsumers, kConsumerThreads);  // tile_out and wsum are reused
    for (int t = tid; t < kOut * kRowsPerTile; t += kConsumerThreads) {
      const int s = t / kRowsPerTile, row = t - s * kRowsPerTile;
      deliver<F, N, E>(a, epi, rbs[k], s, row, Tot::template total<kOut>(red, sls[k], s, row));
    }
    if constexpr (E != Epi::Plain) {
      named_barrier(kBarConsumers, kConsumerThreads);
      run_epilogue<kOut, E>(a, epi, rbs[k], tid, kConsumerThreads);
      epilogue_ran = true;
    }
  }
}

// Adds the partials of the shared row tiles of a GEMV launch (one CTA per
// row tile; tiles a single CTA computed were written by the GEMV) and runs
// the fused epilogue on them.  Launched right after the GEMV with
// programmatic dependent launch: it is resident early, works out which CTAs
// share its tile (CTAs of unshared tiles exit at once) and only then waits
// for the GEMV; after the wait every load it needs (the partials, the input
// scales the GEMV derived) is issued before the first is used.
constexpr int kCombineThreads = 512;

template <Fmt F, int N, Epi E>
__global__ void __launch_bounds__(kCombineThreads) combine_tiles_kernel(const __grid_constant__ GemvArgs a) {
  constexpr int kOut = Traits<F, N>::kOut;
  static_assert(kOut * kRowsPerTile <= kCombineThreads, "one element per thread");
  __shared__ float epi[kEpiBytes / 4];
  const uint32_t tid = threadIdx.x;
  pdl_launch_dependents();
  const int32_t rb = static_cast<int32_t>(blockIdx.x);
  const int32_t c_lo = cta_of_unit(static_cast<int64_t>(rb) * a.n_sb, a.units, a.grid);
  const int32_t c_hi = cta_of_unit(static_cast<int64_t>(rb + 1) * a.n_sb - 1, a.units, a.grid);
  if (c_hi == c_lo) return;  // written by the GEMV
  const int lo_slot = partial_slot_of_first(rb, c_lo, a);
  const int t = static_cast<int>(tid);
  const int s = t / kRowsPerTile, row = t - s * kRowsPerTile;
  pdl_wait_primary();
  float total = 0.0f;
  if (t < kOut * kRowsPerTile) total = sum_partials<kOut>(a, c_lo, c_hi, lo_slot, s, row);
  if constexpr (E != Epi::Plain)
    if (tid < static_cast<uint32_t>(kOut)) epi[4 * kRowsPerTile + tid] = __ldcg(a.scale_out + tid);
  if (t < kOut * kRowsPerTile) deliver<F, N, E>(a, epi, rb, s, row, total);
  if constexpr (E != Epi::Plain) {
    named_barrier(kBarConsumers, kCombineThreads);
    run_epilogue<kOut, E>(a, epi, rb, tid, kCombineThreads);
  }
}

// Shared-memory layout and identity of a consumer thread.
struct ConsumerCtx {
  uint8_t *base_ptr;        // ring of stages
  float *red;               // [2 slots] parked warp sums (Stage::kRedBytes)
  float *epi;               // fused-epilogue scratch
  volatile uint32_t *flag;  // [0] abort
  uint32_t bars, flags;     // shared addresses of the barriers and flags
  uint32_t sq_bar;          // fused epilogues: completes when the input's per-tile sums are staged
  uint32_t sq_stage;        // shared address of the staged sums
  int stages;
  uint32_t tid, warp, lane;
  int64_t u0, u1;           // this CTA's unit range
};

// Fused epilogues: consumer warp s < kOut derives the RMS scale of input
// vector s from the per-tile sums of squares that the producer staged in
// shared memory (or, when they were too many to stage, from global memory
// after the wait on the previous kernel); CTA 0 also hands the scales to the
// tile-combine kernel.
template <int kOut>
__device__ __forceinline__ void derive_input_scale(const GemvArgs &a, const ConsumerCtx &c, uint64_t limit) {
  const bool staged = staged_sum_bytes<kOut>(a) != 0u;
  if (staged && !mbar_try_wait(c.sq_bar, 0) && !mbar_wait_bounded(c.sq_bar, 0, c.flags, limit)) {
    if (c.flag[0] == 0) atomicOr(&g_device_error, PTI_DEVERR_FULL_TIMEOUT);
    c.flag[0] = 1;
    return;
  }
  if (!staged && a.sq_in != nullptr) pdl_wait_primary();  // the sums come from the previous kernel
  float *const scale = c.epi + 4 * kRowsPerTile;
  input_scale_of_stream<kOut>(a, staged ? c.sq_stage : 0u, c.warp, c.lane, scale);
  if (c.lane == 0 && blockIdx.x == 0 && a.scale_out != nullptr) a.scale_out[c.warp] = scale[c.warp];
}

// The consumer warps' walk over the CTA's units: wait for each stage, run the
// consumer `cons` on it (the warp's share of the unit), release the stage; at
// the end of each row tile park the warp's sums, and finish the tiles.
template <Fmt F, int N, Epi E, class Cons>
__device__ __forceinline__ void consumer_loop(const GemvArgs &a, const ConsumerCtx &c, Cons &cons) {
  using T = Traits<F, N>;
  using S = Stage<F, N>;
  constexpr int kOut = T::kOut;
  constexpr int kConsumerThreads = T::kWarps * 32;
  const uint64_t limit = wait_limit(a);
  uint32_t st = 0, ph = 0;  // ring slot and phase parity of the current unit
  // The fused epilogues need the input scales.  The producer stages the
  // input's per-tile sums in shared memory right after its wait on the
  // previous kernel; warp s < kOut derives scale s from them when the first
  // tile is finished (a few shared loads; deriving them earlier, in the
  // stream, measured slower: the deriving warps fall behind and hold ring
  // slots).  The consumer barrier before finish_tiles publishes the scales;
  // CTA 0 also hands them to the tile-combine kernel.
  bool scales_ready = (E == Epi::Plain) || c.warp >= static_cast<uint32_t>(kOut);
  auto wait_scales = [&]() {
    if (scales_ready) return;
    scales_ready = true;
    derive_input_scale<kOut>(a, c, limit);
  };
  const int32_t rb_first = static_cast<int32_t>(c.u0 / a.n_sb);
  const int32_t rb_last = static_cast<int32_t>((c.u1 - 1) / a.n_sb);
  for (int32_t rb = rb_first; rb <= rb_last; ++rb) {
    const int32_t sb_begin = (rb == rb_first) ? static_cast<int32_t>(c.u0 - static_cast<int64_t>(rb) * a.n_sb) : 0;
    const int32_t sb_end = (rb == rb_last) ? static_cast<int32_t>(c.u1 - static_cast<int64_t>(rb) * a.n_sb) : a.n_sb;
    cons.reset();
    for (int32_t sb = sb_begin; sb < sb_end; ++sb) {
      const uint32_t full = c.bars + 8 * st;
      bool ok = mbar_test_wait(full, ph);
      if (!ok) {
        ok = c.flag[0] == 0 && mbar_wait_bounded(full, ph, c.flags, limit);
        if (!ok && c.flag[0] == 0) {
          atomicOr(&g_device_error, PTI_DEVERR_FULL_TIMEOUT);
          c.flag[0] = 1;
        }
      }
      if (ok) {
        const uint8_t *tile = c.base_ptr + st * S::kBytes;
        cons.template unit<S::kXStreamBytes>(tile, tile + kStageBytes);
      }
      __syncwarp();
      if (c.lane == 0) mbar_arrive(c.bars + 8 * (c.stages + st));
      if (++st == static_cast<uint32_t>(c.stages)) {
        st = 0;
        ph ^= 1u;
      }
    }

    // ---- park this warp's sums for the tile: slot 0 = first tile of the CTA,
    //      slot 1 = any later one (only the last can be shared with another CTA)
    const int sl = (rb == rb_first) ? 0 : 1;
    cons.template park<kOut>(c.red, sl, c.warp);
    if (rb != rb_first && rb != rb_last) {
      // a tile wholly inside this CTA's range: finish it now (when a CTA
      // spans more than two row tiles, as most gate/up CTAs of the decode
      // pass do: 20 units per tile, about 36 per CTA)
      wait_scales();
      named_barrier(kBarConsumers, kConsumerThreads);
      finish_tiles<F, N, E, WarpTotals<F>>(a, c.red, 1, rb, 1, 0, 0, c.tid, c.epi);
      named_barrier(kBarConsumers, kConsumerThreads);
    }
  }
  wait_scales();
  named_barrier(kBarConsumers, kConsumerThreads);
  finish_tiles<F, N, E, WarpTotals<F>>(a, c.red, rb_last != rb_first ? 2 : 1, rb_first, 0, rb_last, 1, c.tid,
                                       c.epi);
}

// The copy side of the ring, run by lane 0 of the producer warp: it fills the
// first stages at start and refills each slot as soon as every consumer warp
// has released it.  (Folding this into a consumer warp frees a warp and
// raises the register budget from 96 to 128 per thread, but the consumer that
// refills then waits for the slowest warp on every unit; measured slower.)
template <Fmt F, int N, Epi E>
struct Producer {
  using T = Traits<F, N>;
  using S = Stage<F, N>;
  const CUtensorMap *tmap, *tmap2;
  const GemvArgs *a;
  uint32_t base, bars, flags;
  volatile uint32_t *flag;
  int stages;
  int64_t u0, nu, issued;
  uint64_t pol;
  uint32_t sq_bar, sq_stage;  // fused epilogues: barrier and buffer of the staged input sums
  int32_t ramp;               // initial stages in flight before the next waits for its predecessor
  // Row tile and super-block of the next unit whose weights (w) and
  // activations (x) are to be fetched.  Copies are issued in unit order, so
  // both cursors only step forward (no division per unit: the producer warp
  // shares a scheduler with four consumer warps and every instruction it
  // issues is taken from them).
  int32_t w_rb, w_sb, x_sb;

  __device__ __forceinline__ void init_cursors() {
    w_rb = static_cast<int32_t>(u0 / a->n_sb);
    w_sb = static_cast<int32_t>(u0 - static_cast<int64_t>(w_rb) * a->n_sb);
    x_sb = w_sb;
  }
  __device__ __forceinline__ void load_w(uint32_t slot) {
    const uint32_t dst = base + slot * S::kBytes, bar = bars + 8 * slot;
    if constexpr (E == Epi::GateUp) {
      tma_load_2d(dst, tmap, 34 * w_sb, w_rb * 64, bar, pol);
      tma_load_2d(dst + 64 * kSBBytes, tmap2, 34 * w_sb, w_rb * 64, bar, pol);
    } else {
      tma_load_2d(dst, tmap, 34 * w_sb, w_rb * kRowsPerTile, bar, pol);
    }
    if (++w_sb == a->n_sb) {
      w_sb = 0;
      ++w_rb;
    }
  }
  __device__ __forceinline__ void load_x(uint32_t slot) {
    const uint32_t xdst = base + slot * S::kBytes + kStageBytes, bar = bars + 8 * slot;
    const int64_t col = static_cast<int64_t>(x_sb) * T::kColsPerSB;
    if constexpr (F == Fmt::Q8) {
#pragma unroll
      for (int st = 0; st < N; ++st)
        bulk_load(xdst + st * S::kXStreamBytes, a->x0 + static_cast<int64_t>(st) * a->cols + col, S::kXStreamBytes,
                  bar);
    } else {
#pragma unroll
      for (int st = 0; st < N; ++st) {
        bulk_load(xdst + st * S::kXStreamBytes, a->x0 + static_cast<int64_t>(st) * a->cols + col, S::kXStreamBytes,
                  bar);
        bulk_load(xdst + (N + st) * S::kXStreamBytes, a->x1 + static_cast<int64_t>(st) * a->cols + col,
                  S::kXStreamBytes, bar);
      }
    }
    if (++x_sb == a->n_sb) x_sb = 0;
  }
  // Weights do not depend on the previous kernel in the stream: fetch the
  // first tiles before waiting for it, then their activations.  When the
  // consumers are the slower side (the CUDA-core Q8 consumer with N >= 2),
  // the kernel sets `ramp` to 2: only that many stages go out at once and
  // each further initial stage waits until the one `ramp` before it has
  // landed; with every SM requesting its whole ring at the same moment the
  // first stage would otherwise land only after most of the burst (measured:
  // about 4 us), and compute could not start before.  Chained decode-pass
  // launches (prefetch_all) fetch every initial stage before the wait: the
  // previous kernel's tile combine leaves time for all of them.
  __device__ __forceinline__ void start() {
    prefetch_tmap(tmap);
    if constexpr (E == Epi::GateUp) prefetch_tmap(tmap2);
    init_cursors();
    const int64_t pre = nu < stages ? nu : stages;
    const int64_t first = pre < ramp ? pre : ramp;
    for (int64_t i = 0; i < first; ++i) {
      mbar_expect_tx(bars + 8 * i, kStageBytes);
      load_w(static_cast<uint32_t>(i));
    }
    pdl_wait_primary();
    if constexpr (E != Epi::Plain) {
      // The input's per-tile sums of squares, for the consumers' scales.
      const uint32_t bytes = staged_sum_bytes<T::kOut>(*a);
      if (bytes != 0u) {
        mbar_arrive_expect_tx(sq_bar, bytes);
        bulk_load(sq_stage, a->sq_in, bytes, sq_bar);
      }
    }
    for (int64_t i = 0; i < first; ++i) {
      mbar_arrive_expect_tx(bars + 8 * i, S::kXBytes);
      load_x(static_cast<uint32_t>(i));
    }
    issued = first;
    for (int64_t i = first; i < pre; ++i) {
      const uint32_t landed = bars + 8 * static_cast<uint32_t>(i - ramp);
      if (!mbar_try_wait(landed, 0) && !mbar_wait_bounded(landed, 0, flags, wait_limit(*a))) {
        if (flag[0] == 0) atomicOr(&g_device_error, PTI_DEVERR_FULL_TIMEOUT);
        flag[0] = 1;
        return;
      }
      mbar_arrive_expect_tx(bars + 8 * i, kStageBytes + S::kXBytes);
      load_w(static_cast<uint32_t>(i));
      load_x(static_cast<uint32_t>(i));
      issued = i + 1;
    }
  }
  // Once every consumer warp has released unit i (ring slot st, phase parity
  // ph), fetch unit i + stages into the slot.  (Testing: CTA 0 issues nothing
  // from unit a->stall_unit on.)
  __device__ __forceinline__ void refill(int64_t i, uint32_t st, uint32_t ph) {
    const int64_t j = i + stages;
    if (j >= nu || flag[0] != 0) return;
    if (a->stall_unit >= 0 && j >= a->stall_unit && blockIdx.x == 0) return;
    const uint32_t empty = bars + 8 * (stages + st);
    if (!mbar_try_wait(empty, ph) && !mbar_wait_bounded(empty, ph, flags, wait_limit(*a), kProducerBackoffNs)) {
      if (flag[0] == 0) atomicOr(&g_device_error, PTI_DEVERR_EMPTY_TIMEOUT);
      flag[0] = 1;
      return;
    }
    mbar_arrive_expect_tx(bars + 8 * st, kStageBytes + S::kXBytes);
    load_w(st);
    load_x(st);
    issued = j + 1;
  }
  // Stay until every copy issued into this CTA's shared memory has landed
  // (they all have unless a wait gave up).
  __device__ __forceinline__ void drain() const {
    for (int64_t i = (issued > stages ? issued - stages : 0); i < issued; ++i)
      if (!mbar_wait_bounded(bars + 8 * (i % stages), static_cast<uint32_t>((i / stages) & 1), 0))
        atomicOr(&g_device_error, PTI_DEVERR_DRAIN_TIMEOUT);
  }
};

// tmap: the weight matrix (box 34 x 8 bytes by 128 rows); GateUp: the gate
// matrix and tmap2 the up matrix (boxes of 64 rows each).
template <Fmt F, int N, Epi E>
__global__ void __launch_bounds__(Traits<F, N>::kWarps * 32 + 32, 1)
    gemv_tma_kernel(const __grid_constant__ CUtensorMap tmap, const __grid_constant__ CUtensorMap tmap2,
                    const __grid_constant__ GemvArgs a) {
  using T = Traits<F, N>;
  using S = Stage<F, N>;
  constexpr int kConsumerWarps = T::kWarps;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *const base_ptr = smem_raw + (base - raw);
  const int stages = a.stages;
  float *const red = reinterpret_cast<float *>(base_ptr + stages * S::kBytes);  // parked warp sums
  const uint32_t bars = base + stages * S::kBytes + S::kRedBytes;             // full[stages], empty[stages]
  const uint32_t flags = bars + 2 * stages * 8;  // abort flag, a spare word; then the barrier of the staged sums
  const uint32_t sq_bar = flags + 8;
  volatile uint32_t *const flag = reinterpret_cast<volatile uint32_t *>(base_ptr + (flags - base));
  float *const epi = reinterpret_cast<float *>(base_ptr + (flags - base) + 16);  // kEpiBytes (fused epilogues)
  const uint32_t sq_stage = flags + 16 + kEpiBytes;  // fused epilogues: kSqStageBytes of staged input sums

  const uint32_t tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t u0 = static_cast<int64_t>(blockIdx.x) * a.units / a.grid;
  const int64_t u1 = static_cast<int64_t>(blockIdx.x + 1) * a.units / a.grid;

  if (tid == 0) {
    for (int i = 0; i < stages; ++i) {
      mbar_init(bars + 8 * i, 1);
      mbar_init(bars + 8 * (stages + i), kConsumerWarps);
    }
    mbar_init(sq_bar, 1);
    flag[0] = 0;
    flag[1] = 0;
    mbar_init_fence();
  }
  __syncthreads();
  if (tid == 0) pdl_launch_dependents();

  if (warp == kConsumerWarps) {
    // ---------------- producer: one lane issues every copy --------------------
    if (lane == 0) {
      const int32_t ramp = (F == Fmt::Q8 && N >= 2 && !a.prefetch_all) ? 2 : kMaxStages;
      Producer<F, N, E> prod{&tmap, &tmap2, &a, base, bars, flags, flag, stages, u0, u1 - u0, 0,
                             l2_policy_evict_first(), sq_bar, sq_stage, ramp, 0, 0, 0};
      prod.start();
      uint32_t st = 0, ph = 0;
      for (int64_t i = 0; i + stages < prod.nu && flag[0] == 0; ++i) {
        prod.refill(i, st, ph);
        if (++st == static_cast<uint32_t>(stages)) {
          st = 0;
          ph ^= 1u;
        }
      }
      prod.drain();
    }
    return;
  }

  // ---------------- consumers ----------------------------------------------
  const ConsumerCtx cx{base_ptr, red, epi, flag, bars, flags, sq_bar, sq_stage, stages, tid, warp, lane, u0, u1};
  auto run = [&](auto cons) {
    cons.init(warp, lane);
    consumer_loop<F, N, E>(a, cx, cons);
  };
  if constexpr (F == Fmt::Q8) {
    // Warp w computes block w % 8; the warps of a scheduler (w % 4) share the
    // parity of the block and so run one code body.
    switch (warp & 3u) {  // block b = 2c + e: (e, c % 2)
      case 0: run(Q8Pair<N, 0, 0>{}); break;
      case 1: run(Q8Pair<N, 1, 0>{}); break;
      case 2: run(Q8Pair<N, 0, 1>{}); break;
      default: run(Q8Pair<N, 1, 1>{}); break;
    }
  } else {
    // Twin: warp w computes block w % 4 (its scheduler, so one code body per
    // scheduler).
    switch (warp & 3u) {
      case 0: run(TwinSlab<N, 0>{}); break;
      case 1: run(TwinSlab<N, 1>{}); break;
      case 2: run(TwinSlab<N, 2>{}); break;
      default: run(TwinSlab<N, 3>{}); break;
    }
  }
}

// The tensor-core consumer of the Q8 kernel (gemv_tc_kernel).
#include "pti_gemv_tc.cuh"

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    else
      cudaGetLastError();
  });
  return fn;
}

struct TilePlan {
  int64_t n_sb = 0, n_rb = 0, units = 0;
  int32_t grid = 0, stages = 0;
  size_t smem = 0;
};

// Rows of the output vectors per tile: 128, or 64 (gate, up) pairs for GateUp.
template <Epi E>
constexpr int64_t out_rows_per_tile() {
  return E == Epi::GateUp ? 64 : kRowsPerTile;
}

template <Fmt F, int N, Epi E>
TilePlan plan_tiles(int64_t rows, int64_t cols, int sms) {
  using T = Traits<F, N>;
  using S = Stage<F, N>;
  TilePlan p;
  p.n_sb = cols / T::kColsPerSB;
  p.n_rb = (rows + out_rows_per_tile<E>() - 1) / out_rows_per_tile<E>();
  p.units = p.n_sb * p.n_rb;
  p.grid = static_cast<int32_t>(std::min<int64_t>({static_cast<int64_t>(sms), p.units, kMaxGrid}));
  const int64_t fixed = 1024 + S::kRedBytes + 16 * kMaxStages + 16 + (E == Epi::Plain ? 0 : kEpiBytes + kSqStageBytes);
  p.stages = static_cast<int32_t>(std::min<int64_t>(kMaxStages, (kSmemOptin - fixed) / S::kBytes));
  p.smem = static_cast<size_t>(fixed) + static_cast<size_t>(p.stages) * S::kBytes;
  return p;
}

// The same tiling for the tensor-core kernel, with its shared-memory layout.
template <int N, Epi E>
TilePlan plan_tiles_tc(int64_t rows, int64_t cols, int sms) {
  using S = Stage<Fmt::Q8, N>;
  TilePlan p = plan_tiles<Fmt::Q8, N, E>(rows, cols, sms);
  const int64_t fixed = 1024 + 2 * kTcBBytes + TcLayout<N>::kXinvBytes + TcLayout<N>::kRedBytes +
                        8 * (2 * kMaxStages + 4) + 16 + (E == Epi::Plain ? 0 : kEpiBytes + kSqStageBytes);
  p.stages = static_cast<int32_t>(std::min<int64_t>(kMaxStages, (kSmemOptin - fixed) / S::kBytes));
  p.smem = static_cast<size_t>(fixed) + static_cast<size_t>(p.stages) * S::kBytes;
  return p;
}

// Which consumer a Q8 launch uses: the CUDA-core one (the default: it
// measured at least as fast at every stream count) or, on request, the
// tensor-core one.
enum class Cores : int { Auto = 0, Cuda = 1, Tensor = 2 };

template <Fmt F, int N, Epi E>
constexpr bool use_tensor_cores(Cores c) {
  return F == Fmt::Q8 && E == Epi::Plain && c == Cores::Tensor;
}

// Stream-K partials of one call: [kMaxGrid][2 slots][kout][128] floats.
inline size_t partial_bytes(int kout) {
  return static_cast<size_t>(kMaxGrid) * 2 * kout * kRowsPerTile * sizeof(float);
}

// Workspace of the fast GEMV paths: the partials of shared tiles only (no
// counters, so it needs no initialisation).
inline size_t fast_workspace_bytes(int kout) {
  return (partial_bytes(kout) + 255) & ~static_cast<size_t>(255);
}

// Encodes the 2-D tensor map of a row-major matrix of `rows` rows of
// (cols / 32) blocks, in 8-byte units, with a box of one super-block by
// `box_rows` rows.  No L2 promotion: a box row is 272 bytes at any offset
// mod 128, and promoting its requests to 256-byte L2 fetches read 1.5 times
// its sectors; the neighbouring unit uses most of the extra, but not at row
// ends, where the surplus came back from DRAM (about 1.4% more DRAM reads
// per launch, 3.3% in the gate/up step; no difference in time).
template <Fmt F>
bool encode_weight_map(CUtensorMap *tmap, const void *w, int64_t rows, int64_t cols, uint32_t box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (encode == nullptr) return false;
  const uint64_t row_bytes = static_cast<uint64_t>(cols / 32) * Traits<F, 1>::kBlockBytes;
  std::memset(tmap, 0, sizeof(*tmap));
  const cuuint64_t gdim[2] = {row_bytes / 8, static_cast<cuuint64_t>(rows)};
  const cuuint64_t gstride[1] = {row_bytes};
  const cuuint32_t box[2] = {kSBBytes / 8, box_rows};
  const cuuint32_t estride[2] = {1, 1};
  return encode(tmap, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<void *>(w), gdim, gstride, box, estride,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Launches the persistent kernel.  `a` carries the operands (x0, x1, y0, y1,
// part, rows, cols and the epilogue fields); the tiling fields are
// filled in here.  w2 is the up matrix of a GateUp launch.  With `pdl` the
// launch may start while the previous kernel in the stream is still running
// (programmatic dependent launch); the kernel reads only weights before it
// waits for that kernel to complete.
template <Fmt F, int N, Epi E = Epi::Plain>
pti_status launch_gemv(const void *w, const void *w2, GemvArgs a, cudaStream_t stream, bool pdl,
                       Cores cores = Cores::Auto) {
  using T = Traits<F, N>;
  constexpr bool kTcCapable = F == Fmt::Q8 && E == Epi::Plain;  // the decode pass runs on the CUDA cores
  const bool tc = use_tensor_cores<F, N, E>(cores);
  int dev = 0;
  const int sms = current_device_sms(&dev);
  if (sms <= 0) return PTI_ERR_CUDA;
  TilePlan p;
  if constexpr (kTcCapable) p = tc ? plan_tiles_tc<N, E>(a.rows, a.cols, sms) : plan_tiles<F, N, E>(a.rows, a.cols, sms);
  else p = plan_tiles<F, N, E>(a.rows, a.cols, sms);
  if (p.stages < 2 || p.smem > static_cast<size_t>(kSmemOptin)) return PTI_ERR_SHAPE;

  static std::mutex mu;
  static bool attr_done[2][128] = {};
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!attr_done[tc][dev]) {
      cudaError_t e = cudaSuccess;
      if constexpr (kTcCapable) {
        if (tc) e = cudaFuncSetAttribute(gemv_tc_kernel<N, E>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemOptin);
      }
      if (!tc) e = cudaFuncSetAttribute(gemv_tma_kernel<F, N, E>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemOptin);
      if (e != cudaSuccess) return launch_status();
      attr_done[tc][dev] = true;
    }
  }

  CUtensorMap tmap, tmap2;
  const uint32_t box_rows = static_cast<uint32_t>(E == Epi::GateUp ? 64 : kRowsPerTile);
  if (!encode_weight_map<F>(&tmap, w, a.rows, a.cols, box_rows)) return PTI_ERR_CUDA;
  if constexpr (E == Epi::GateUp) {
    if (!encode_weight_map<F>(&tmap2, w2, a.rows, a.cols, box_rows)) return PTI_ERR_CUDA;
  } else {
    tmap2 = tmap;
  }

  a.units = p.units;
  a.n_sb = static_cast<int32_t>(p.n_sb);
  a.n_rb = static_cast<int32_t>(p.n_rb);
  a.grid = p.grid;
  a.stages = p.stages;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.grid));
  cfg.blockDim = dim3(tc ? kTcThreads + 64 : T::kWarps * 32 + 32);
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  cudaError_t le = cudaSuccess;
  if constexpr (kTcCapable) {
    if (tc) le = cudaLaunchKernelEx(&cfg, gemv_tc_kernel<N, E>, tmap, tmap2, a);
  }
  if (!tc) le = cudaLaunchKernelEx(&cfg, gemv_tma_kernel<F, N, E>, tmap, tmap2, a);
  if (le != cudaSuccess) return launch_status();
  // the shared tiles' partials, once the GEMV has completed (only if a tile
  // spans several CTAs: never when every CTA owns whole tiles)
  if (p.grid > 1) {
    cudaLaunchConfig_t cc = {};
    cc.gridDim = dim3(static_cast<unsigned>(p.n_rb));
    cc.blockDim = dim3(kCombineThreads);
    cc.stream = stream;
    cc.attrs = attr;
    cc.numAttrs = 1;
    if (cudaLaunchKernelEx(&cc, combine_tiles_kernel<F, N, E>, a) != cudaSuccess) return launch_status();
  }
  return launch_status();
}

// The plain GEMV: the workspace holds the shared tiles' partials.
template <Fmt F, int N>
pti_status launch_fast(const void *w, int64_t rows, int64_t cols, const float *x0, const float *x1,
                       float *y0, float *y1, void *workspace, cudaStream_t stream, bool pdl = false,
                       Cores cores = Cores::Auto, uint64_t wait_ns = 0, int64_t stall_unit = -1) {
  GemvArgs a = {};
  a.wait_ns = wait_ns;
  a.stall_unit = stall_unit;
  a.x0 = x0;
  a.x1 = x1;
  a.y0 = y0;
  a.y1 = y1;
  a.part = static_cast<float *>(workspace);
  a.rows = rows;
  a.cols = cols;
  return launch_gemv<F, N, Epi::Plain>(w, nullptr, a, stream, pdl, cores);
}

pti_status check_gemv_shape(int64_t rows, int64_t cols) {
  if (rows < 1 || cols < 32 || cols % 32 != 0) return PTI_ERR_SHAPE;
  if (rows > (int64_t{1} << 31) || cols > (int64_t{1} << 31) || rows * cols >= (int64_t{1} << 40))
    return PTI_ERR_SHAPE;
  return PTI_OK;
}

}  // namespace
}  // namespace pti
