// pti_gemv.cu -- N-stream Q8 GEMV and SSQ "mode 16" twin GEMV on sm_103a.
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
//  * One producer warp issues the TMA copies into a 4-stage ring guarded by
//    mbarriers; 16 consumer warps compute.  Lane l of a consumer task owns two
//    rows of the tile and reads its 16-byte chunk of each with one aligned,
//    bank-conflict-free shared load.  The 17 chunk positions need 17
//    specialised code bodies; to keep each scheduler's instruction working set
//    small, scheduler k owns chunks k, k+4, k+8, k+12 (chunk 16 rotates over
//    the schedulers from unit to unit) and its four warps split each owned
//    chunk into two 64-row halves.
//  * The activations of the unit's columns are staged once per CTA segment in
//    shared memory as float2 column pairs; every warp reads them with
//    broadcast loads and reuses them for its 64 rows, so activation traffic
//    does not grow with the number of row tiles (the L2 thrash the pages
//    diagnose for the per-row-block design).
//  * Dequantisation is exact (see pti_device.cuh); products use packed
//    f32x2 FMAs.  Each chunk's products are summed into a fresh partial, which
//    is then added to the running accumulator, so no fp32 chain is longer than
//    a few dozen dependent roundings per output.
// Other shapes use a plain per-row kernel (one warp per row).
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
  int64_t rows, cols, units;
  int32_t n_sb, n_rb, grid, stages;
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

// Sums the 8 warps' partials of one deferred row-tile segment (red slot `sl`)
// and writes them: straight to y when no other CTA shares the tile, else as
// this CTA's partial, the last CTA to finish the tile adding all partials in
// CTA order.
template <Fmt F, int N>
__device__ __forceinline__ void finish_tile(const GemvArgs &a, const float *red, int sl, int32_t rb,
                                            int32_t rb_first_cta, uint32_t tid, volatile uint32_t *flag) {
  using T = Traits<F, N>;
  constexpr int kOut = T::kOut;
  constexpr int kConsumerThreads = T::kWarps * 32;
  const int32_t c_lo = cta_of_unit(static_cast<int64_t>(rb) * a.n_sb, a.units, a.grid);
  const int32_t c_hi = cta_of_unit(static_cast<int64_t>(rb + 1) * a.n_sb - 1, a.units, a.grid);
  const bool shared_tile = c_hi > c_lo;
  for (int t = tid; t < kOut * kRowsPerTile; t += kConsumerThreads) {
    const int s = t / kRowsPerTile, row = t - s * kRowsPerTile;
    float v[T::kWarps / 2];
#pragma unroll
    for (int q = 0; q < T::kWarps / 2; ++q) {
      const int w = (q >> 2) * 8 + (row >> 6) * 4 + (q & 3);  // the warps whose half is row / 64
      v[q] = red[((sl * T::kWarps + w) * kOut + s) * 64 + (row & 63)];
    }
    const float total = tree_sum(v);
    const int64_t row_g = static_cast<int64_t>(rb) * kRowsPerTile + row;
    if (!shared_tile) {
      if (row_g < a.rows) {
        if constexpr (F == Fmt::Q8) a.y0[s * a.rows + row_g] = total;
        else (s == 0 ? a.y0 : a.y1)[row_g] = total;
      }
    } else {
      a.part[((static_cast<int64_t>(blockIdx.x) * 2 + sl) * kOut + s) * kRowsPerTile + row] = total;
    }
  }
  if (!shared_tile) return;
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
    const int64_t row_g = static_cast<int64_t>(rb) * kRowsPerTile + row;
    if (row_g < a.rows) {
      if constexpr (F == Fmt::Q8) a.y0[s * a.rows + row_g] = total;
      else (s == 0 ? a.y0 : a.y1)[row_g] = total;
    }
  }
  (void)rb_first_cta;
}

template <Fmt F, int N>
__global__ void __launch_bounds__(Traits<F, N>::kWarps * 32 + 32, 1)
    gemv_tma_kernel(const __grid_constant__ CUtensorMap tmap, const GemvArgs a) {
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
      const uint64_t pol = l2_policy_evict_first();
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
        tma_load_2d(base + static_cast<uint32_t>(i) * S::kBytes, &tmap, 34 * sb, rb * kRowsPerTile, bars + 8 * i, pol);
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
        tma_load_2d(base + st * S::kBytes, &tmap, 34 * sb, rb * kRowsPerTile, bars + 8 * st, pol);
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
      finish_tile<F, N>(a, red, 1, rb, rb_first, tid, flag);
      named_barrier(kBarConsumers, kConsumerThreads);
    }
  }
  named_barrier(kBarConsumers, kConsumerThreads);
  finish_tile<F, N>(a, red, 0, rb_first, rb_first, tid, flag);
  if (rb_last != rb_first) {
    named_barrier(kBarConsumers, kConsumerThreads);
    finish_tile<F, N>(a, red, 1, rb_last, rb_first, tid, flag);
  }
}

// ---------------------------------------------------------------------------
// Plain per-row kernels for shapes outside the fast path: one warp per row,
// lanes stride over the blocks, each block's products summed into a fresh
// partial and scaled once.
// ---------------------------------------------------------------------------
template <int N>
__global__ void __launch_bounds__(256) q8_rowwise_kernel(const uint8_t *__restrict__ w, int64_t rows,
                                                         int64_t cols, const float *__restrict__ x,
                                                         float *__restrict__ y) {
  const int lane = threadIdx.x & 31;
  const int64_t nb = cols / 32;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t row = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; row < rows; row += warps) {
    float acc[N];
#pragma unroll
    for (int s = 0; s < N; ++s) acc[s] = 0.0f;
    for (int64_t b = lane; b < nb; b += 32) {
      const uint8_t *blk = w + (row * nb + b) * 34;
      const float d = half_bits_to_float(*reinterpret_cast<const uint16_t *>(blk));
      float part[N];
#pragma unroll
      for (int s = 0; s < N; ++s) part[s] = 0.0f;
      for (int i = 0; i < 32; ++i) {
        const float q = static_cast<float>(static_cast<int8_t>(blk[2 + i]));
#pragma unroll
        for (int s = 0; s < N; ++s) part[s] = fmaf(q, x[s * cols + 32 * b + i], part[s]);
      }
#pragma unroll
      for (int s = 0; s < N; ++s) acc[s] = fmaf(d, part[s], acc[s]);
    }
#pragma unroll
    for (int s = 0; s < N; ++s)
      for (int o = 16; o > 0; o >>= 1) acc[s] += __shfl_xor_sync(0xFFFFFFFFu, acc[s], o);
    if (lane == 0)
#pragma unroll
      for (int s = 0; s < N; ++s) y[s * rows + row] = acc[s];
  }
}

__global__ void __launch_bounds__(256) twin_rowwise_kernel(const uint8_t *__restrict__ w, int64_t rows,
                                                           int64_t cols, const float *__restrict__ xa,
                                                           const float *__restrict__ xb,
                                                           float *__restrict__ ya, float *__restrict__ yb) {
  const int lane = threadIdx.x & 31;
  const int64_t nb = cols / 32;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t row = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; row < rows; row += warps) {
    float acc_a = 0.0f, acc_b = 0.0f;
    for (int64_t b = lane; b < nb; b += 32) {
      const uint8_t *blk = w + (row * nb + b) * 68;
      const float da = half_bits_to_float(*reinterpret_cast<const uint16_t *>(blk));
      const float db = half_bits_to_float(*reinterpret_cast<const uint16_t *>(blk + 2));
      float pa = 0.0f, pb = 0.0f;
      for (int i = 0; i < 32; ++i) {
        const uint16_t pw = *reinterpret_cast<const uint16_t *>(blk + 4 + 2 * i);
        const float qa = static_cast<float>(static_cast<int8_t>(pw >> 8));
        const float qb = static_cast<float>(static_cast<int8_t>(pw & 0xFF));
        pa = fmaf(qa, xa[32 * b + i], pa);
        pb = fmaf(qb, xb[32 * b + i], pb);
      }
      acc_a = fmaf(da, pa, acc_a);
      acc_b = fmaf(db, pb, acc_b);
    }
    for (int o = 16; o > 0; o >>= 1) {
      acc_a += __shfl_xor_sync(0xFFFFFFFFu, acc_a, o);
      acc_b += __shfl_xor_sync(0xFFFFFFFFu, acc_b, o);
    }
    if (lane == 0) {
      ya[row] = acc_a;
      yb[row] = acc_b;
    }
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

template <Fmt F, int N>
TilePlan plan_tiles(int64_t rows, int64_t cols, int sms) {
  using T = Traits<F, N>;
  using S = Stage<F, N>;
  TilePlan p;
  p.n_sb = cols / T::kColsPerSB;
  p.n_rb = (rows + kRowsPerTile - 1) / kRowsPerTile;
  p.units = p.n_sb * p.n_rb;
  p.grid = static_cast<int32_t>(std::min<int64_t>({static_cast<int64_t>(sms), p.units, kMaxGrid}));
  const int64_t fixed = 1024 + S::kRedBytes + 16 * kMaxStages + 16;
  p.stages = static_cast<int32_t>(std::min<int64_t>(kMaxStages, (kSmemOptin - fixed) / S::kBytes));
  p.smem = static_cast<size_t>(fixed) + static_cast<size_t>(p.stages) * S::kBytes;
  return p;
}

template <Fmt F>
size_t fast_workspace_bytes(int64_t rows, int kout) {
  const int64_t n_rb = (rows + kRowsPerTile - 1) / kRowsPerTile;
  const size_t part = static_cast<size_t>(kMaxGrid) * 2 * kout * kRowsPerTile * sizeof(float);
  const size_t tickets = static_cast<size_t>(n_rb) * sizeof(unsigned int);
  return (part + tickets + 255) & ~static_cast<size_t>(255);
}

template <Fmt F, int N>
pti_status launch_fast(const void *w, int64_t rows, int64_t cols, const float *x0, const float *x1,
                       float *y0, float *y1, void *workspace, cudaStream_t stream, bool pdl = false) {
  using T = Traits<F, N>;
  int dev = 0;
  const int sms = current_device_sms(&dev);
  if (sms <= 0) return PTI_ERR_CUDA;
  const TilePlan p = plan_tiles<F, N>(rows, cols, sms);
  if (p.stages < 2 || p.smem > static_cast<size_t>(kSmemOptin)) return PTI_ERR_SHAPE;

  static std::mutex mu;
  static bool attr_done[128] = {};
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!attr_done[dev]) {
      if (cudaFuncSetAttribute(gemv_tma_kernel<F, N>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemOptin) !=
          cudaSuccess)
        return launch_status();
      attr_done[dev] = true;
    }
  }

  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (encode == nullptr) return PTI_ERR_CUDA;
  const uint64_t row_bytes = static_cast<uint64_t>(cols / 32) * T::kBlockBytes;
  CUtensorMap tmap;
  std::memset(&tmap, 0, sizeof(tmap));
  const cuuint64_t gdim[2] = {row_bytes / 8, static_cast<cuuint64_t>(rows)};
  const cuuint64_t gstride[1] = {row_bytes};
  const cuuint32_t box[2] = {kSBBytes / 8, kRowsPerTile};
  const cuuint32_t estride[2] = {1, 1};
  if (encode(&tmap, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, const_cast<void *>(w), gdim, gstride, box, estride,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return PTI_ERR_CUDA;

  GemvArgs a;
  a.x0 = x0;
  a.x1 = x1;
  a.y0 = y0;
  a.y1 = y1;
  a.part = static_cast<float *>(workspace);
  a.tickets = reinterpret_cast<unsigned int *>(static_cast<uint8_t *>(workspace) +
                                               static_cast<size_t>(kMaxGrid) * 2 * T::kOut * kRowsPerTile * sizeof(float));
  a.rows = rows;
  a.cols = cols;
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
  if (cudaLaunchKernelEx(&cfg, gemv_tma_kernel<F, N>, tmap, a) != cudaSuccess) return launch_status();
  return launch_status();
}

template <int N>
pti_status launch_q8_rowwise(const void *w, int64_t rows, int64_t cols, const float *x, float *y,
                             cudaStream_t stream) {
  const int sms = current_device_sms();
  if (sms <= 0) return PTI_ERR_CUDA;
  const int64_t blocks = std::min<int64_t>((rows + 7) / 8, static_cast<int64_t>(sms) * 16);
  q8_rowwise_kernel<N><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(static_cast<const uint8_t *>(w), rows,
                                                                          cols, x, y);
  return launch_status();
}

pti_status check_gemv_shape(int64_t rows, int64_t cols) {
  if (rows < 1 || cols < 32 || cols % 32 != 0) return PTI_ERR_SHAPE;
  if (rows > (int64_t{1} << 31) || cols > (int64_t{1} << 31) || rows * cols >= (int64_t{1} << 40))
    return PTI_ERR_SHAPE;
  return PTI_OK;
}

}  // namespace
}  // namespace pti

using namespace pti;

extern "C" const char *pti_status_string(pti_status status) {
  switch (status) {
    case PTI_OK: return "PTI_OK";
    case PTI_ERR_NULL: return "PTI_ERR_NULL: a required pointer is NULL";
    case PTI_ERR_SHAPE: return "PTI_ERR_SHAPE: invalid or unsupported shape";
    case PTI_ERR_NSTREAMS: return "PTI_ERR_NSTREAMS: stream count outside [1, 4]";
    case PTI_ERR_ALIGN: return "PTI_ERR_ALIGN: pointer not aligned as documented";
    case PTI_ERR_ALIAS: return "PTI_ERR_ALIAS: an output overlaps an input or another output";
    case PTI_ERR_CUDA: return "PTI_ERR_CUDA: the CUDA runtime reported an error";
    case PTI_ERR_WORKSPACE: return "PTI_ERR_WORKSPACE: workspace missing or too small";
  }
  return "PTI_ERR_UNKNOWN";
}

extern "C" size_t pti_q8_gemv_workspace_bytes(int64_t rows, int64_t cols, int n_streams) {
  if (check_gemv_shape(rows, cols) != PTI_OK || n_streams < 1 || n_streams > 4) return 0;
  if (cols % 256 != 0) return 0;
  return fast_workspace_bytes<Fmt::Q8>(rows, n_streams);
}

extern "C" size_t pti_ssq_twin_gemv_workspace_bytes(int64_t rows, int64_t cols) {
  if (check_gemv_shape(rows, cols) != PTI_OK) return 0;
  if (cols % 128 != 0) return 0;
  return fast_workspace_bytes<Fmt::Twin>(rows, 2);
}

extern "C" pti_status pti_q8_gemv_nstream(const void *w_q8, int64_t rows, int64_t cols, int n_streams,
                                          const float *x, float *y, void *workspace, size_t workspace_bytes,
                                          pti_stream_t stream) {
  if (w_q8 == nullptr || x == nullptr || y == nullptr) return PTI_ERR_NULL;
  if (const pti_status s = check_gemv_shape(rows, cols); s != PTI_OK) return s;
  if (n_streams < 1 || n_streams > 4) return PTI_ERR_NSTREAMS;
  if (!aligned(w_q8, 16) || !aligned(x, 4) || !aligned(y, 4)) return PTI_ERR_ALIGN;
  const uint64_t w_bytes = static_cast<uint64_t>(rows) * (cols / 32) * 34;
  const uint64_t x_bytes = static_cast<uint64_t>(n_streams) * cols * 4;
  const uint64_t y_bytes = static_cast<uint64_t>(n_streams) * rows * 4;
  if (overlaps(y, y_bytes, w_q8, w_bytes) || overlaps(y, y_bytes, x, x_bytes)) return PTI_ERR_ALIAS;
  const size_t need = pti_q8_gemv_workspace_bytes(rows, cols, n_streams);
  if (need > 0) {
    if (workspace == nullptr || workspace_bytes < need) return PTI_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return PTI_ERR_ALIGN;
    if (overlaps(workspace, need, w_q8, w_bytes) || overlaps(workspace, need, x, x_bytes) ||
        overlaps(workspace, need, y, y_bytes))
      return PTI_ERR_ALIAS;
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (need > 0 && aligned(x, 16)) {
    switch (n_streams) {
      case 1: return launch_fast<Fmt::Q8, 1>(w_q8, rows, cols, x, nullptr, y, nullptr, workspace, st);
      case 2: return launch_fast<Fmt::Q8, 2>(w_q8, rows, cols, x, nullptr, y, nullptr, workspace, st);
      case 3: return launch_fast<Fmt::Q8, 3>(w_q8, rows, cols, x, nullptr, y, nullptr, workspace, st);
      default: return launch_fast<Fmt::Q8, 4>(w_q8, rows, cols, x, nullptr, y, nullptr, workspace, st);
    }
  }
  switch (n_streams) {
    case 1: return launch_q8_rowwise<1>(w_q8, rows, cols, x, y, st);
    case 2: return launch_q8_rowwise<2>(w_q8, rows, cols, x, y, st);
    case 3: return launch_q8_rowwise<3>(w_q8, rows, cols, x, y, st);
    default: return launch_q8_rowwise<4>(w_q8, rows, cols, x, y, st);
  }
}

extern "C" pti_status pti_ssq_twin_gemv(const void *w_twin, int64_t rows, int64_t cols, const float *x_a,
                                        const float *x_b, float *y_a, float *y_b, void *workspace,
                                        size_t workspace_bytes, pti_stream_t stream) {
  if (w_twin == nullptr || x_a == nullptr || x_b == nullptr || y_a == nullptr || y_b == nullptr)
    return PTI_ERR_NULL;
  if (const pti_status s = check_gemv_shape(rows, cols); s != PTI_OK) return s;
  if (!aligned(w_twin, 16) || !aligned(x_a, 4) || !aligned(x_b, 4) || !aligned(y_a, 4) || !aligned(y_b, 4))
    return PTI_ERR_ALIGN;
  const uint64_t w_bytes = static_cast<uint64_t>(rows) * (cols / 32) * 68;
  const uint64_t x_bytes = static_cast<uint64_t>(cols) * 4;
  const uint64_t y_bytes = static_cast<uint64_t>(rows) * 4;
  if (overlaps(y_a, y_bytes, y_b, y_bytes) || overlaps(y_a, y_bytes, w_twin, w_bytes) ||
      overlaps(y_b, y_bytes, w_twin, w_bytes) || overlaps(y_a, y_bytes, x_a, x_bytes) ||
      overlaps(y_a, y_bytes, x_b, x_bytes) || overlaps(y_b, y_bytes, x_a, x_bytes) ||
      overlaps(y_b, y_bytes, x_b, x_bytes))
    return PTI_ERR_ALIAS;
  const size_t need = pti_ssq_twin_gemv_workspace_bytes(rows, cols);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (need > 0) {
    if (workspace == nullptr || workspace_bytes < need) return PTI_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return PTI_ERR_ALIGN;
    if (overlaps(workspace, need, w_twin, w_bytes) || overlaps(workspace, need, x_a, x_bytes) ||
        overlaps(workspace, need, x_b, x_bytes) || overlaps(workspace, need, y_a, y_bytes) ||
        overlaps(workspace, need, y_b, y_bytes))
      return PTI_ERR_ALIAS;
    if (aligned(x_a, 16) && aligned(x_b, 16))
      return launch_fast<Fmt::Twin, 2>(w_twin, rows, cols, x_a, x_b, y_a, y_b, workspace, st);
  }
  const int sms = current_device_sms();
  if (sms <= 0) return PTI_ERR_CUDA;
  const int64_t blocks = std::min<int64_t>((rows + 7) / 8, static_cast<int64_t>(sms) * 16);
  twin_rowwise_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(static_cast<const uint8_t *>(w_twin), rows, cols,
                                                                     x_a, x_b, y_a, y_b);
  return launch_status();
}

// ---------------------------------------------------------------------------
// Allocation-free variant of the N-stream Q8 GEMV.
//
// Some callers cannot allocate device memory for the workspace: a plug-in that
// runs inside another runtime which owns every device allocation through its
// own memory pool and only hands out input and output buffers, or a decode
// loop that must not call into the CUDA allocator once it is running (freeing
// device memory synchronises the whole device and stalls every stream).  For
// them the workspace lives in this file-scope array, reserved when the library
// is loaded and kept by every GPU that loads it until the process exits.
// ---------------------------------------------------------------------------
constexpr size_t kNoAllocScratchBytes = size_t{2} << 20;  // 2 MiB per device
static __device__ __align__(256) unsigned char g_pti_noalloc_scratch[kNoAllocScratchBytes];

namespace {
// Device address of g_pti_noalloc_scratch on the current device.  The first
// call on a device looks the address up (the array's name is only a host-side
// stand-in), zero-fills the array and synchronises the device.
pti_status noalloc_scratch_address(void **out) {
  static std::mutex mu;
  static void *addr[128] = {};
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) {
    cudaGetLastError();
    return PTI_ERR_CUDA;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_pti_noalloc_scratch) != cudaSuccess || p == nullptr) return launch_status();
    if (cudaMemset(p, 0, kNoAllocScratchBytes) != cudaSuccess) return launch_status();
    if (cudaDeviceSynchronize() != cudaSuccess) return launch_status();
    addr[dev] = p;
  }
  *out = addr[dev];
  return PTI_OK;
}
}  // namespace

extern "C" size_t pti_q8_gemv_noalloc_max_scratch_bytes(void) { return kNoAllocScratchBytes; }

extern "C" pti_status pti_q8_gemv_nstream_noalloc(const void *w_q8, int64_t rows, int64_t cols, int n_streams,
                                                  const float *x, float *y, pti_stream_t stream) {
  if (w_q8 == nullptr || x == nullptr || y == nullptr) return PTI_ERR_NULL;
  if (const pti_status st = check_gemv_shape(rows, cols); st != PTI_OK) return st;
  if (n_streams < 1 || n_streams > 4) return PTI_ERR_NSTREAMS;
  const size_t need = pti_q8_gemv_workspace_bytes(rows, cols, n_streams);
  if (need > kNoAllocScratchBytes) return PTI_ERR_WORKSPACE;  // more rows than the built-in scratch serves
  void *scratch = nullptr;
  if (need > 0) {
    if (const pti_status st = noalloc_scratch_address(&scratch); st != PTI_OK) return st;
  }
  return pti_q8_gemv_nstream(w_q8, rows, cols, n_streams, x, y, scratch, need > 0 ? kNoAllocScratchBytes : 0,
                             stream);
}

extern "C" pti_status pti_device_error(uint32_t *code_out) {
  if (code_out == nullptr) return PTI_ERR_NULL;
  if (cudaDeviceSynchronize() != cudaSuccess) return launch_status();
  unsigned int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v)) != cudaSuccess) return launch_status();
  if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero)) != cudaSuccess) return launch_status();
  *code_out = v;
  return PTI_OK;
}
