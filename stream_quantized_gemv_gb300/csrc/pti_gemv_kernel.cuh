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
//    number of bytes.  Row tiles shared by several CTAs are combined by the
//    last CTA to finish them (an atomic ticket per tile, partials in a
//    caller-supplied workspace, summed in a fixed CTA order).
//  * One producer warp issues the copies into a ring of up to 6 stages guarded
//    by mbarriers; 16 consumer warps compute.  Lane l of a consumer task owns
//    two rows of the tile and reads its 16-byte chunk of each with one aligned,
//    bank-conflict-free shared load.  The 17 chunk positions fall into a few
//    structural classes (where the block scale sits in the chunk), one code
//    body per class; scheduler k owns chunks k, k+4, k+8, k+12 (chunk 16
//    rotates over the schedulers from unit to unit) and its four warps split
//    each owned chunk into two 64-row halves.
//  * Each stage also holds the unit's slice of the activations (N x 1 KB,
//    stream-major), fetched by one bulk copy per stream next to the weight
//    tile.  Every warp reads them with broadcast loads and reuses them for its
//    64 rows, so activation traffic is one slice per unit and does not grow
//    with the number of rows (the L2 thrash the pages diagnose for the
//    per-row-block design comes from re-reading x once per row block).
//  * Dequantisation is exact (see pti_device.cuh); products use packed
//    f32x2 FMAs.  Each chunk's products are summed into a fresh partial, which
//    is then added to the running accumulator, so no fp32 chain is longer than
//    a few dozen dependent roundings per output.
//  * Programmatic dependent launch: the producer fetches its first weight
//    tiles before waiting for the previous kernel in the stream, and only then
//    fetches activations; nothing is written before that wait.
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
constexpr int kWarpCount = 16;  // consumer warps, 4 per scheduler
constexpr int kStageBytes = kRowsPerTile * kSBBytes;   // 34816
constexpr int kMaxGrid = 320;
constexpr int kSmemOptin = 232448;                     // 227 KB per CTA
constexpr uint32_t kBarConsumers = 1;                  // named barrier of the consumer warps

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
  static constexpr int kWarps = kWarpCount;
  static constexpr int kColsPerSB = 256;
  static constexpr int kXStreams = N;
  static constexpr int kBlockBytes = 34;
};
template <int N>
struct Traits<Fmt::Twin, N> {
  static constexpr int kOut = 2;
  static constexpr int kWarps = kWarpCount;
  static constexpr int kColsPerSB = 128;
  static constexpr int kXStreams = 2;
  static constexpr int kBlockBytes = 68;
};

// One pipeline stage: the 128 x 272-byte weight tile followed by the unit's
// activations, stream-major (kXStreams rows of kColsPerSB floats).
template <Fmt F, int N>
struct Stage {
  static constexpr int kXStreamBytes = Traits<F, N>::kColsPerSB * 4;
  static constexpr int kXBytes = Traits<F, N>::kXStreams * kXStreamBytes;
  static constexpr int kBytes = ((kStageBytes + kXBytes) + 1023) / 1024 * 1024;
  static constexpr int kRedBytes = 2 * Traits<F, N>::kWarps * Traits<F, N>::kOut * 64 * 4;
};

struct GemvArgs {
  const float *x0;  // Q8: x [N][cols]; twin: x_a
  const float *x1;  // twin: x_b
  float *y0;        // Q8: y [N][rows]; twin: y_a
  float *y1;        // twin: y_b
  float *part;      // workspace: [grid][2 slots][kOut][128] partial sums
  unsigned int *tickets;  // workspace: [n_rb] arrival counters (zero between calls)
  int64_t rows, cols, units;  // GateUp: rows = gate rows = up rows = outputs per stream
  int32_t n_sb, n_rb, grid, stages;
  // Fused epilogues only (Epi::GateUp, Epi::Down):
  const float *sq_in;  // [n_sq_in][kOut] per-tile sums of squares of the input vectors; null: scale 1
  float *sq_out;       // [n_rb][kOut] per-tile sums of squares of the output vectors
  double inv_len_in;   // 1 / length of each input vector
  double eps;          // added to the mean square before the square root
  int32_t n_sq_in;
};

// Rows handled by one warp task: lane l owns rows 64h + l and 64h + 32 + l of
// the tile (h = the task's half).  (Four rows per lane halves the activation
// loads per weight but doubles the code of each chunk body; measured slower.)
constexpr int kTaskSlots = 2;

// Where a 16-byte chunk's weights sit.  Chunks come in a few structural
// classes: `cls` = -1 when the chunk holds no scale (all its bytes are weights
// of block b0), else the index of the byte pair holding the next block's scale
// (Q8: 0..7; twin: the word index 0..3).  The generic parameters are the byte
// offset of the chunk, the offset of block b0's scale in the row, and the
// column pair of the chunk's first weight pair (`cpbase`).
struct ChunkParams {
  int cls;
  uint32_t choff;     // 16 * c
  uint32_t scale_off; // byte offset of block b0's scale within the super-block row
  uint32_t cpbase;    // column pair (within the super-block) of pair 0
};

__device__ __forceinline__ ChunkParams q8_chunk_params(int c) {
  ChunkParams p;
  p.choff = 16u * c;
  if (c <= 14 && (c & 1) == 0) {  // the scale of block c/2 sits at pair (16c - 34(c/2)) / 2 = c/2
    p.cls = c / 2;
    const int b0 = c / 2 > 0 ? c / 2 - 1 : 0;
    p.scale_off = 34u * b0;
    p.cpbase = 15u * (c / 2);
  } else {
    const int b0 = (16 * c) / 34;
    p.cls = -1;
    p.scale_off = 34u * b0;
    p.cpbase = static_cast<uint32_t>((32 * b0 + (16 * c) % 34 - 2) / 2);
  }
  return p;
}

__device__ __forceinline__ ChunkParams twin_chunk_params(int c) {
  ChunkParams p;
  p.choff = 16u * c;
  if ((c & 3) == 0 && c <= 12) {  // chunk c holds the scale word of block c/4 at word c/4
    p.cls = c / 4;
    const int b0 = c / 4 > 0 ? c / 4 - 1 : 0;
    p.scale_off = 68u * b0;
    p.cpbase = 15u * (c / 4);
  } else {
    const int b0 = (4 * c) / 17;
    p.cls = -1;
    p.scale_off = 68u * b0;
    p.cpbase = static_cast<uint32_t>(16 * b0 + (4 * c) % 17 - 1);
  }
  return p;
}

template <int I>
__device__ __forceinline__ uint32_t word_at(const uint4 &w) {
  if constexpr (I == 0) return w.x;
  else if constexpr (I == 1) return w.y;
  else if constexpr (I == 2) return w.z;
  else return w.w;
}

// One Q8 chunk of class K for the lane's two rows of half h.  Byte pair m of
// the chunk holds weight columns cpbase + m (pairs before the scale) or
// cpbase + m - 1 (pairs after it).
template <int N, int K>
__device__ __forceinline__ void q8_body(const uint8_t *tile, const ChunkParams &cp, const uint8_t *xsb,
                                        uint32_t lane, uint32_t half, uint64_t (&acc)[kTaskSlots][N]) {
  constexpr int M0 = (K == 0) ? 1 : 0;  // first weight pair
  uint32_t wx[kTaskSlots][4];
  ScalePair s_lo[kTaskSlots], s_hi[kTaskSlots];
#pragma unroll
  for (int r = 0; r < kTaskSlots; ++r) {
    const uint8_t *row = tile + (half * 64 + r * 32 + lane) * kSBBytes;
    const uint4 w = *reinterpret_cast<const uint4 *>(row + cp.choff);
    if constexpr (K != 0) s_lo[r] = make_scale(*reinterpret_cast<const uint16_t *>(row + cp.scale_off));
    if constexpr (K >= 0) {
      const uint32_t wd = word_at<K / 2>(w);
      s_hi[r] = make_scale((K & 1) ? (wd >> 16) : (wd & 0xFFFFu));
    }
    wx[r][0] = w.x ^ 0x80808080u;
    wx[r][1] = w.y ^ 0x80808080u;
    wx[r][2] = w.z ^ 0x80808080u;
    wx[r][3] = w.w ^ 0x80808080u;
  }
  const uint8_t *xc = xsb + cp.cpbase * 8;
  uint64_t p[kTaskSlots][N];
  static_for<0, 8>([&](auto mc) {
    constexpr int m = decltype(mc)::value;
    if constexpr (m != K) {
      constexpr int off = (K >= 0 && m > K) ? m - 1 : m;
      uint64_t xv[N];
#pragma unroll
      for (int st = 0; st < N; ++st)
        xv[st] = *reinterpret_cast<const uint64_t *>(xc + st * Stage<Fmt::Q8, N>::kXStreamBytes + off * 8);
#pragma unroll
      for (int r = 0; r < kTaskSlots; ++r) {
        const ScalePair &sc = (K < 0 || m < K) ? s_lo[r] : s_hi[r];
        const uint64_t wq = dequant2(wx[r][m / 2], (2 * m) % 4, wx[r][m / 2], (2 * m) % 4 + 1, sc);
        static_for<0, N>([&](auto sc_) {
          constexpr int s = decltype(sc_)::value;
          if constexpr (m == M0) p[r][s] = fmul2(wq, xv[s]);
          else p[r][s] = ffma2(wq, xv[s], p[r][s]);
        });
      }
    }
  });
#pragma unroll
  for (int r = 0; r < kTaskSlots; ++r)
    static_for<0, N>([&](auto sc_) {
      constexpr int s = decltype(sc_)::value;
      acc[r][s] = fadd2(acc[r][s], p[r][s]);
    });
}

// One twin chunk of class J for the lane's two rows of half h.  Word j of the
// chunk holds column pair cpbase + j (before the scale word) or cpbase + j - 1.
template <int N, int J>
__device__ __forceinline__ void twin_body(const uint8_t *tile, const ChunkParams &cp, const uint8_t *xsb,
                                          uint32_t lane, uint32_t half, uint64_t (&acc)[kTaskSlots][2]) {
  constexpr int J0 = (J == 0) ? 1 : 0;
  uint4 w[kTaskSlots];
  ScalePair sa_lo[kTaskSlots], sb_lo[kTaskSlots], sa_hi[kTaskSlots], sb_hi[kTaskSlots];
#pragma unroll
  for (int r = 0; r < kTaskSlots; ++r) {
    const uint8_t *row = tile + (half * 64 + r * 32 + lane) * kSBBytes;
    w[r] = *reinterpret_cast<const uint4 *>(row + cp.choff);
    if constexpr (J != 0) {
      const uint32_t sw = *reinterpret_cast<const uint32_t *>(row + cp.scale_off);
      sa_lo[r] = make_scale(sw & 0xFFFFu);
      sb_lo[r] = make_scale(sw >> 16);
    }
    if constexpr (J >= 0) {
      const uint32_t sw = word_at<J>(w[r]);
      sa_hi[r] = make_scale(sw & 0xFFFFu);
      sb_hi[r] = make_scale(sw >> 16);
    }
  }
  const uint8_t *xc = xsb + cp.cpbase * 8;
  uint64_t pa[kTaskSlots], pb[kTaskSlots];
  static_for<0, 4>([&](auto jc) {
    constexpr int j = decltype(jc)::value;
    if constexpr (j != J) {
      constexpr int off = (J >= 0 && j > J) ? j - 1 : j;
      const uint64_t xa = *reinterpret_cast<const uint64_t *>(xc + off * 8);
      const uint64_t xb = *reinterpret_cast<const uint64_t *>(xc + Stage<Fmt::Twin, N>::kXStreamBytes + off * 8);
      constexpr bool lo = (J < 0 || j < J);
#pragma unroll
      for (int r = 0; r < kTaskSlots; ++r) {
        const uint32_t wxj = word_at<j>(w[r]) ^ 0x80808080u;
        const uint64_t wa = dequant2(wxj, 1, wxj, 3, lo ? sa_lo[r] : sa_hi[r]);  // model A: high bytes
        const uint64_t wb = dequant2(wxj, 0, wxj, 2, lo ? sb_lo[r] : sb_hi[r]);  // model B: low bytes
        if constexpr (j == J0) {
          pa[r] = fmul2(wa, xa);
          pb[r] = fmul2(wb, xb);
        } else {
          pa[r] = ffma2(wa, xa, pa[r]);
          pb[r] = ffma2(wb, xb, pb[r]);
        }
      }
    }
  });
#pragma unroll
  for (int r = 0; r < kTaskSlots; ++r) {
    acc[r][0] = fadd2(acc[r][0], pa[r]);
    acc[r][1] = fadd2(acc[r][1], pb[r]);
  }
}

template <Fmt F, int N>
__device__ __forceinline__ ChunkParams chunk_params(int c) {
  if constexpr (F == Fmt::Q8) return q8_chunk_params(c);
  else return twin_chunk_params(c);
}

template <Fmt F, int N>
__device__ __forceinline__ void run_chunk(const ChunkParams &cp, const uint8_t *tile, const uint8_t *xsb,
                                          uint32_t lane, uint32_t half,
                                          uint64_t (&acc)[kTaskSlots][Traits<F, N>::kOut]) {
  if constexpr (F == Fmt::Q8) {
    switch (cp.cls) {
      case -1: q8_body<N, -1>(tile, cp, xsb, lane, half, acc); break;
      case 0: q8_body<N, 0>(tile, cp, xsb, lane, half, acc); break;
      case 1: q8_body<N, 1>(tile, cp, xsb, lane, half, acc); break;
      case 2: q8_body<N, 2>(tile, cp, xsb, lane, half, acc); break;
      case 3: q8_body<N, 3>(tile, cp, xsb, lane, half, acc); break;
      case 4: q8_body<N, 4>(tile, cp, xsb, lane, half, acc); break;
      case 5: q8_body<N, 5>(tile, cp, xsb, lane, half, acc); break;
      case 6: q8_body<N, 6>(tile, cp, xsb, lane, half, acc); break;
      default: q8_body<N, 7>(tile, cp, xsb, lane, half, acc); break;
    }
  } else {
    switch (cp.cls) {
      case -1: twin_body<N, -1>(tile, cp, xsb, lane, half, acc); break;
      case 0: twin_body<N, 0>(tile, cp, xsb, lane, half, acc); break;
      case 1: twin_body<N, 1>(tile, cp, xsb, lane, half, acc); break;
      case 2: twin_body<N, 2>(tile, cp, xsb, lane, half, acc); break;
      default: twin_body<N, 3>(tile, cp, xsb, lane, half, acc); break;
    }
  }
}

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

// RMS scale of each input vector, 1 / sqrt(mean(v^2) + eps), from the
// previous kernel's per-tile sums of squares (summed in double, in a fixed
// order, so every CTA derives the same scale); 1 when there are none.
// Warp s < kOut handles vector s; must run after the wait on the previous
// kernel.  A consumer barrier must separate it from the first reader.
template <int kOut>
__device__ __forceinline__ void input_scales(const GemvArgs &a, uint32_t warp, uint32_t lane, float *scale) {
  if (warp >= static_cast<uint32_t>(kOut)) return;
  double s2 = 0.0;
  if (a.sq_in != nullptr)
    for (int32_t t = static_cast<int32_t>(lane); t < a.n_sq_in; t += 32)
      s2 += static_cast<double>(__ldcg(a.sq_in + static_cast<int64_t>(t) * kOut + warp));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s2 += __shfl_xor_sync(0xFFFFFFFFu, s2, o);
  if (lane == 0) scale[warp] = a.sq_in != nullptr ? static_cast<float>(1.0 / sqrt(s2 * a.inv_len_in + a.eps)) : 1.0f;
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
// h; writes x' [kOut][rows] and the tile's sum of x'^2 per vector.
template <int kOut>
__device__ __forceinline__ void down_epilogue(const GemvArgs &a, const float *tile_out, const float *scale,
                                              float *wsum, int32_t rb, uint32_t tid, uint32_t consumer_threads) {
  float v = 0.0f;
  if (tid < static_cast<uint32_t>(kOut * kRowsPerTile)) {
    const int s = static_cast<int>(tid >> 7), r = static_cast<int>(tid & 127u);
    const int64_t row = static_cast<int64_t>(rb) * kRowsPerTile + r;
    if (row < a.rows) {
      v = tile_out[s * kRowsPerTile + r] * scale[s];
      a.y0[s * a.rows + row] = v;
    }
  }
  const uint32_t warp = tid >> 5;
  if (warp < static_cast<uint32_t>(4 * kOut)) {
    const float q = warp_sum(v * v);
    if ((tid & 31u) == 0) wsum[warp] = q;
  }
  named_barrier(kBarConsumers, consumer_threads);
  if (tid < static_cast<uint32_t>(kOut))
    a.sq_out[static_cast<int64_t>(rb) * kOut + tid] =
        (wsum[4 * tid] + wsum[4 * tid + 1]) + (wsum[4 * tid + 2] + wsum[4 * tid + 3]);
}

// Sums the 16 warps' partials of one deferred row-tile segment (red slot `sl`)
// into the tile's totals: straight to the output (Plain) or the epilogue's
// tile buffer when no other CTA shares the tile, else as this CTA's partial,
// the last CTA to finish the tile adding all partials in CTA order.  The
// fused epilogues then run on the complete tile.
template <Fmt F, int N, Epi E>
__device__ __forceinline__ void finish_tile(const GemvArgs &a, const float *red, int sl, int32_t rb, uint32_t tid,
                                            volatile uint32_t *flag, float *epi) {
  using T = Traits<F, N>;
  constexpr int kOut = T::kOut;
  constexpr int kConsumerThreads = T::kWarps * 32;
  float *const tile_out = epi;                                // [kOut][128]
  float *const scale = epi + 4 * kRowsPerTile;                // [kOut]
  float *const wsum = scale + 4;                              // [16]
  const int32_t c_lo = cta_of_unit(static_cast<int64_t>(rb) * a.n_sb, a.units, a.grid);
  const int32_t c_hi = cta_of_unit(static_cast<int64_t>(rb + 1) * a.n_sb - 1, a.units, a.grid);
  const bool shared_tile = c_hi > c_lo;
  auto deliver = [&](int s, int row, float total) {
    if constexpr (E == Epi::Plain) {
      const int64_t row_g = static_cast<int64_t>(rb) * kRowsPerTile + row;
      if (row_g < a.rows) {
        if constexpr (F == Fmt::Q8) a.y0[s * a.rows + row_g] = total;
        else (s == 0 ? a.y0 : a.y1)[row_g] = total;
      }
    } else {
      tile_out[s * kRowsPerTile + row] = total;
    }
  };
  for (int t = tid; t < kOut * kRowsPerTile; t += kConsumerThreads) {
    const int s = t / kRowsPerTile, row = t - s * kRowsPerTile;
    float v[T::kWarps / 2];
#pragma unroll
    for (int q = 0; q < T::kWarps / 2; ++q) {
      const int w = (q >> 2) * 8 + (row >> 6) * 4 + (q & 3);  // the warps whose half is row / 64
      v[q] = red[((sl * T::kWarps + w) * kOut + s) * 64 + (row & 63)];
    }
    const float total = tree_sum(v);
    if (!shared_tile) deliver(s, row, total);
    else a.part[((static_cast<int64_t>(blockIdx.x) * 2 + sl) * kOut + s) * kRowsPerTile + row] = total;
  }
  if (shared_tile) {
    __threadfence();
    named_barrier(kBarConsumers, kConsumerThreads);
    if (tid == 0) {
      const unsigned int prev = atomicAdd(&a.tickets[rb], 1u);
      const bool last = prev == static_cast<unsigned int>(c_hi - c_lo);
      if (last) {
        a.tickets[rb] = 0u;  // leave the workspace zeroed for the next call
        __threadfence();
      }
      flag[1] = last ? 1u : 0u;
    }
    named_barrier(kBarConsumers, kConsumerThreads);
    if (flag[1] == 0) return;
    for (int t = tid; t < kOut * kRowsPerTile; t += kConsumerThreads) {
      const int s = t / kRowsPerTile, row = t - s * kRowsPerTile;
      float total = 0.0f;
      for (int32_t c = c_lo; c <= c_hi; ++c) {
        const int cs = (rb == first_tile_of_cta(c, a.units, a.grid, a.n_sb)) ? 0 : 1;
        float *const slot_ptr = &a.part[((static_cast<int64_t>(c) * 2 + cs) * kOut + s) * kRowsPerTile + row];
        const float v = __ldcg(slot_ptr);
        *slot_ptr = 0.0f;  // the whole workspace is zero again when the call completes
        total = (c == c_lo) ? v : total + v;
      }
      deliver(s, row, total);
    }
  }
  if constexpr (E != Epi::Plain) {
    named_barrier(kBarConsumers, kConsumerThreads);
    if constexpr (E == Epi::GateUp) gateup_epilogue<kOut>(a, tile_out, scale, wsum, rb, tid, kConsumerThreads);
    else down_epilogue<kOut>(a, tile_out, scale, wsum, rb, tid, kConsumerThreads);
  }
}

// tmap: the weight matrix (box 34 x 8 bytes by 128 rows); GateUp: the gate
// matrix and tmap2 the up matrix (boxes of 64 rows each).
template <Fmt F, int N, Epi E>
__global__ void __launch_bounds__(Traits<F, N>::kWarps * 32 + 32, 1)
    gemv_tma_kernel(const __grid_constant__ CUtensorMap tmap, const __grid_constant__ CUtensorMap tmap2,
                    const GemvArgs a) {
  using T = Traits<F, N>;
  using S = Stage<F, N>;
  constexpr int kOut = T::kOut;
  constexpr int kConsumerWarps = T::kWarps;
  constexpr int kConsumerThreads = kConsumerWarps * 32;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *const base_ptr = smem_raw + (base - raw);
  const int stages = a.stages;
  float *const red = reinterpret_cast<float *>(base_ptr + stages * S::kBytes);  // [2][warps][kOut][64]
  const uint32_t bars = base + stages * S::kBytes + S::kRedBytes;             // full[stages], empty[stages]
  const uint32_t flags = bars + 2 * stages * 8;
  volatile uint32_t *const flag = reinterpret_cast<volatile uint32_t *>(base_ptr + (flags - base));
  float *const epi = reinterpret_cast<float *>(base_ptr + (flags - base) + 16);  // kEpiBytes (fused epilogues)

  const uint32_t tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t u0 = static_cast<int64_t>(blockIdx.x) * a.units / a.grid;
  const int64_t u1 = static_cast<int64_t>(blockIdx.x + 1) * a.units / a.grid;

  if (tid == 0) {
    for (int i = 0; i < stages; ++i) {
      mbar_init(bars + 8 * i, 1);
      mbar_init(bars + 8 * (stages + i), kConsumerWarps);
    }
    flag[0] = 0;
    flag[1] = 0;
    mbar_init_fence();
  }
  __syncthreads();
  if (tid == 0) pdl_launch_dependents();

  if (warp == kConsumerWarps) {
    // ---------------- producer: one lane issues every copy --------------------
    if (lane == 0) {
      prefetch_tmap(&tmap);
      if constexpr (E == Epi::GateUp) prefetch_tmap(&tmap2);
      const uint64_t pol = l2_policy_evict_first();
      auto load_w = [&](uint32_t slot, int32_t rb, int32_t sb) {
        const uint32_t dst = base + slot * S::kBytes, bar = bars + 8 * slot;
        if constexpr (E == Epi::GateUp) {
          tma_load_2d(dst, &tmap, 34 * sb, rb * 64, bar, pol);
          tma_load_2d(dst + 64 * kSBBytes, &tmap2, 34 * sb, rb * 64, bar, pol);
        } else {
          tma_load_2d(dst, &tmap, 34 * sb, rb * kRowsPerTile, bar, pol);
        }
      };
      const int64_t nu = u1 - u0;
      const int64_t pre = nu < stages ? nu : stages;
      auto unit_coords = [&](int64_t i, int32_t &rb, int32_t &sb) {
        const int64_t u = u0 + i;
        rb = static_cast<int32_t>(u / a.n_sb);
        sb = static_cast<int32_t>(u - static_cast<int64_t>(rb) * a.n_sb);
      };
      auto load_x = [&](int64_t i, uint32_t slot) {
        int32_t rb, sb;
        unit_coords(i, rb, sb);
        const uint32_t xdst = base + slot * S::kBytes + kStageBytes;
        const uint32_t bar = bars + 8 * slot;
        if constexpr (F == Fmt::Q8) {
#pragma unroll
          for (int st = 0; st < N; ++st)
            bulk_load(xdst + st * S::kXStreamBytes, a.x0 + static_cast<int64_t>(st) * a.cols + static_cast<int64_t>(sb) * T::kColsPerSB,
                      S::kXStreamBytes, bar);
        } else {
          bulk_load(xdst, a.x0 + static_cast<int64_t>(sb) * T::kColsPerSB, S::kXStreamBytes, bar);
          bulk_load(xdst + S::kXStreamBytes, a.x1 + static_cast<int64_t>(sb) * T::kColsPerSB, S::kXStreamBytes, bar);
        }
      };
      // Weights do not depend on the previous kernel in the stream: prefetch
      // the first tiles before waiting for it, then fetch their activations.
      for (int64_t i = 0; i < pre; ++i) {
        int32_t rb, sb;
        unit_coords(i, rb, sb);
        mbar_expect_tx(bars + 8 * i, kStageBytes);
        load_w(static_cast<uint32_t>(i), rb, sb);
      }
      pdl_wait_primary();
      for (int64_t i = 0; i < pre; ++i) {
        mbar_arrive_expect_tx(bars + 8 * i, S::kXBytes);
        load_x(i, static_cast<uint32_t>(i));
      }
      int64_t issued = pre;
      uint32_t st = static_cast<uint32_t>(pre % stages), eph = 0;  // slot and empty-phase parity
      for (int64_t i = pre; i < nu; ++i) {
        const uint32_t empty = bars + 8 * (stages + st);
        if (!mbar_try_wait(empty, eph) && !mbar_wait_bounded(empty, eph, flags)) {
          if (flag[0] == 0) atomicOr(&g_device_error, PTI_DEVERR_EMPTY_TIMEOUT);
          flag[0] = 1;
          break;
        }
        if (flag[0] != 0) break;
        int32_t rb, sb;
        unit_coords(i, rb, sb);
        mbar_arrive_expect_tx(bars + 8 * st, kStageBytes + S::kXBytes);
        load_w(st, rb, sb);
        load_x(i, st);
        issued = i + 1;
        if (++st == static_cast<uint32_t>(stages)) {
          st = 0;
          eph ^= 1u;
        }
      }
      // Stay until every copy issued into this CTA's shared memory has landed.
      for (int64_t i = (issued > stages ? issued - stages : 0); i < issued; ++i) {
        if (!mbar_wait_bounded(bars + 8 * (i % stages), static_cast<uint32_t>((i / stages) & 1), 0))
          atomicOr(&g_device_error, PTI_DEVERR_DRAIN_TIMEOUT);
      }
    }
    return;
  }

  // ---------------- consumers ----------------------------------------------
  uint64_t acc[kTaskSlots][kOut];
  // Warp w runs on scheduler k = w % 4 (warps are dealt to the four schedulers
  // round-robin) and always works on the same two chunks of every unit, rows
  // of half j % 2 (j = w / 4): chunks k + 4(j/2) and k + 4(j/2) + 8, so each
  // scheduler owns chunks k, k+4, k+8, k+12.  Chunk 16 of unit i goes to the
  // warps j = 0, 1 of scheduler i % 4.
  const uint32_t sched = warp & 3u, wj = warp >> 2;
  const uint32_t half = wj & 1u;
  const int ca = static_cast<int>(sched + 4u * (wj >> 1));
  const ChunkParams pa = chunk_params<F, N>(ca), pb = chunk_params<F, N>(ca + 8),
                    p16 = chunk_params<F, N>(16);
  const bool takes16 = (wj >> 1) == 0u;
  if constexpr (E != Epi::Plain) {
    pdl_wait_primary();  // the input's sums of squares come from the previous kernel
    input_scales<kOut>(a, warp, lane, epi + 4 * kRowsPerTile);
  }
  uint32_t st = 0, ph = 0;  // ring slot and phase parity of unit i
  int64_t i = 0;
  const int32_t rb_first = static_cast<int32_t>(u0 / a.n_sb);
  const int32_t rb_last = static_cast<int32_t>((u1 - 1) / a.n_sb);
  for (int32_t rb = rb_first; rb <= rb_last; ++rb) {
    const int32_t sb_begin = (rb == rb_first) ? static_cast<int32_t>(u0 - static_cast<int64_t>(rb) * a.n_sb) : 0;
    const int32_t sb_end = (rb == rb_last) ? static_cast<int32_t>(u1 - static_cast<int64_t>(rb) * a.n_sb) : a.n_sb;
#pragma unroll
    for (int r = 0; r < kTaskSlots; ++r)
#pragma unroll
      for (int s = 0; s < kOut; ++s) acc[r][s] = 0ull;

    for (int32_t sb = sb_begin; sb < sb_end; ++sb, ++i) {
      const uint32_t full = bars + 8 * st;
      bool ok = mbar_try_wait(full, ph);
      if (!ok) {
        ok = flag[0] == 0 && mbar_wait_bounded(full, ph, flags);
        if (!ok && flag[0] == 0) {
          atomicOr(&g_device_error, PTI_DEVERR_FULL_TIMEOUT);
          flag[0] = 1;
        }
      }
      if (ok) {
        const uint8_t *tile = base_ptr + st * S::kBytes;
        const uint8_t *xsb = tile + kStageBytes;
        run_chunk<F, N>(pa, tile, xsb, lane, half, acc);
        run_chunk<F, N>(pb, tile, xsb, lane, half, acc);
        if (takes16 && (static_cast<uint32_t>(i) & 3u) == sched) run_chunk<F, N>(p16, tile, xsb, lane, half, acc);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bars + 8 * (stages + st));
      if (++st == static_cast<uint32_t>(stages)) {
        st = 0;
        ph ^= 1u;
      }
    }

    // ---- park this warp's sums for the tile: slot 0 = first tile of the CTA,
    //      slot 1 = any later one (only the last can be shared with another CTA)
    const int sl = (rb == rb_first) ? 0 : 1;
    const bool middle = rb != rb_first && rb != rb_last;
#pragma unroll
    for (int r = 0; r < kTaskSlots; ++r)
#pragma unroll
      for (int s = 0; s < kOut; ++s) {
        const float2 v = unpack2(acc[r][s]);
        red[((sl * kConsumerWarps + warp) * kOut + s) * 64 + r * 32 + lane] = v.x + v.y;
      }
    if (middle) {
      // a tile wholly inside this CTA's range: finish it now (rare: only when
      // a CTA spans more than two row tiles)
      named_barrier(kBarConsumers, kConsumerThreads);
      finish_tile<F, N, E>(a, red, 1, rb, tid, flag, epi);
      named_barrier(kBarConsumers, kConsumerThreads);
    }
  }
  named_barrier(kBarConsumers, kConsumerThreads);
  finish_tile<F, N, E>(a, red, 0, rb_first, tid, flag, epi);
  if (rb_last != rb_first) {
    named_barrier(kBarConsumers, kConsumerThreads);
    finish_tile<F, N, E>(a, red, 1, rb_last, tid, flag, epi);
  }
}

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
  const int64_t fixed = 1024 + S::kRedBytes + 16 * kMaxStages + 16 + (E == Epi::Plain ? 0 : kEpiBytes);
  p.stages = static_cast<int32_t>(std::min<int64_t>(kMaxStages, (kSmemOptin - fixed) / S::kBytes));
  p.smem = static_cast<size_t>(fixed) + static_cast<size_t>(p.stages) * S::kBytes;
  return p;
}

// Stream-K partials of one call: [kMaxGrid][2 slots][kout][128] floats.
inline size_t partial_bytes(int kout) {
  return static_cast<size_t>(kMaxGrid) * 2 * kout * kRowsPerTile * sizeof(float);
}

template <Fmt F>
size_t fast_workspace_bytes(int64_t rows, int kout) {
  const int64_t n_rb = (rows + kRowsPerTile - 1) / kRowsPerTile;
  const size_t tickets = static_cast<size_t>(n_rb) * sizeof(unsigned int);
  return (partial_bytes(kout) + tickets + 255) & ~static_cast<size_t>(255);
}

// Encodes the 2-D tensor map of a row-major matrix of `rows` rows of
// (cols / 32) blocks, in 8-byte units, with a box of one super-block by
// `box_rows` rows.
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
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Launches the persistent kernel.  `a` carries the operands (x0, x1, y0, y1,
// part, tickets, rows, cols and the epilogue fields); the tiling fields are
// filled in here.  w2 is the up matrix of a GateUp launch.  With `pdl` the
// launch may start while the previous kernel in the stream is still running
// (programmatic dependent launch); the kernel reads only weights before it
// waits for that kernel to complete.
template <Fmt F, int N, Epi E = Epi::Plain>
pti_status launch_gemv(const void *w, const void *w2, GemvArgs a, cudaStream_t stream, bool pdl) {
  using T = Traits<F, N>;
  int dev = 0;
  const int sms = current_device_sms(&dev);
  if (sms <= 0) return PTI_ERR_CUDA;
  const TilePlan p = plan_tiles<F, N, E>(a.rows, a.cols, sms);
  if (p.stages < 2 || p.smem > static_cast<size_t>(kSmemOptin)) return PTI_ERR_SHAPE;

  static std::mutex mu;
  static bool attr_done[128] = {};
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!attr_done[dev]) {
      if (cudaFuncSetAttribute(gemv_tma_kernel<F, N, E>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kSmemOptin) != cudaSuccess)
        return launch_status();
      attr_done[dev] = true;
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
  cfg.blockDim = dim3(T::kWarps * 32 + 32);
  cfg.dynamicSmemBytes = p.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if (cudaLaunchKernelEx(&cfg, gemv_tma_kernel<F, N, E>, tmap, tmap2, a) != cudaSuccess) return launch_status();
  return launch_status();
}

// The plain GEMV: partials at the start of the workspace, tickets after them.
template <Fmt F, int N>
pti_status launch_fast(const void *w, int64_t rows, int64_t cols, const float *x0, const float *x1,
                       float *y0, float *y1, void *workspace, cudaStream_t stream, bool pdl = false) {
  GemvArgs a = {};
  a.x0 = x0;
  a.x1 = x1;
  a.y0 = y0;
  a.y1 = y1;
  a.part = static_cast<float *>(workspace);
  a.tickets = reinterpret_cast<unsigned int *>(static_cast<uint8_t *>(workspace) + partial_bytes(Traits<F, N>::kOut));
  a.rows = rows;
  a.cols = cols;
  return launch_gemv<F, N, Epi::Plain>(w, nullptr, a, stream, pdl);
}

pti_status check_gemv_shape(int64_t rows, int64_t cols) {
  if (rows < 1 || cols < 32 || cols % 32 != 0) return PTI_ERR_SHAPE;
  if (rows > (int64_t{1} << 31) || cols > (int64_t{1} << 31) || rows * cols >= (int64_t{1} << 40))
    return PTI_ERR_SHAPE;
  return PTI_OK;
}

}  // namespace
}  // namespace pti
