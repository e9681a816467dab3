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
//    mbarriers; 15 consumer warps compute.  Consumer warp w owns chunk w of
//    every unit (chunks 15 and 16 rotate over the warps), and lane l owns rows
//    l, l+32, l+64, l+96 of the tile: each lane reads its chunk with one
//    aligned, bank-conflict-free 16-byte shared load per row.
//  * The activations of the unit's columns are staged once per CTA segment in
//    shared memory as float2 column pairs; every warp reads them with
//    broadcast loads and reuses them for its 128 rows, so activation traffic
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
constexpr int kSlots = kRowsPerTile / 32;              // rows per lane
constexpr int kStages = 4;
constexpr int kStageBytes = kRowsPerTile * kSBBytes;   // 34816
constexpr int kMaxGrid = 320;
constexpr int kSmemOptin = 232448;                     // 227 KB per CTA
constexpr int kBarBytes = 2 * kStages * 8 + 16;        // full[], empty[], two flag words
constexpr uint32_t kBarConsumers = 1;                  // named barrier of the consumer warps

__device__ unsigned int g_device_error = 0;

enum class Fmt : int { Q8 = 0, Twin = 1 };

template <Fmt F, int N>
struct Traits;
template <int N>
struct Traits<Fmt::Q8, N> {
  static constexpr int kOut = N;                   // output vectors
  static constexpr int kNS = (N == 3) ? 4 : N;     // float2 slots per staged column pair
  // 4 streams need ~136 registers per thread: 14 consumer warps + 1 producer
  // warp keep the CTA within the 64K-register file.
  static constexpr int kWarps = (N == 4) ? 14 : 15;
  static constexpr int kColsPerSB = 256;
  static constexpr int kXBytesPerSB = (kColsPerSB / 2) * kNS * 8;
  static constexpr int kBlockBytes = 34;
};
template <int N>
struct Traits<Fmt::Twin, N> {
  static constexpr int kOut = 2;
  static constexpr int kWarps = 15;
  static constexpr int kColsPerSB = 128;
  static constexpr int kXBytesPerSB = (kColsPerSB / 2) * 16;
  static constexpr int kBlockBytes = 68;
};

struct GemvArgs {
  const float *x0;  // Q8: x [N][cols]; twin: x_a
  const float *x1;  // twin: x_b
  float *y0;        // Q8: y [N][rows]; twin: y_a
  float *y1;        // twin: y_b
  float *part;      // workspace: [grid][2 slots][kOut][128] partial sums
  unsigned int *tickets;  // workspace: [n_rb] arrival counters (zero between calls)
  int64_t rows, cols, units;
  int32_t n_sb, n_rb, grid, xw_sb;
  uint32_t x_region_bytes;
};

// ---------------------------------------------------------------------------
// Chunk geometry (compile time).
// Q8 super-block: block b occupies bytes [34b, 34b+34): scale at 34b, q[i] at
// 34b+2+i (column 32b+i).  A 16-byte chunk's bytes pair up as (2m, 2m+1); the
// two bytes of a pair are always both scale bytes or both weights of one block.
// ---------------------------------------------------------------------------
struct Q8Geom {
  static constexpr int absb(int c, int p) { return 16 * c + p; }
  static constexpr bool is_scale(int c, int p) { return absb(c, p) % 34 < 2; }
  static constexpr int block(int c, int p) { return absb(c, p) / 34; }
  static constexpr int col(int c, int p) { return 32 * block(c, p) + absb(c, p) % 34 - 2; }
  static constexpr int first_pair(int c) {
    for (int m = 0; m < 8; ++m)
      if (!is_scale(c, 2 * m)) return m;
    return -1;
  }
  static constexpr int first_block(int c) { return block(c, 2 * first_pair(c)); }
  static constexpr int last_block(int c) {
    int b = -1;
    for (int m = 0; m < 8; ++m)
      if (!is_scale(c, 2 * m)) b = block(c, 2 * m);
    return b;
  }
  // byte offset of block b's scale inside chunk c, or -1
  static constexpr int scale_in_chunk(int c, int b) {
    return (34 * b - 16 * c >= 0 && 34 * b - 16 * c < 16) ? 34 * b - 16 * c : -1;
  }
};

// Twin super-block: 68 words; block b = words [17b, 17b+17): word 17b holds
// scale_A (low half) and scale_B (high half), word 17b+1+j holds columns
// 32b+2j and 32b+2j+1 as bytes [B_2j, A_2j, B_2j+1, A_2j+1].
struct TwinGeom {
  static constexpr int word(int c, int j) { return 4 * c + j; }
  static constexpr int block(int c, int j) { return word(c, j) / 17; }
  static constexpr bool is_scale(int c, int j) { return word(c, j) % 17 == 0; }
  static constexpr int colpair(int c, int j) { return 16 * block(c, j) + word(c, j) % 17 - 1; }
  static constexpr int first_word(int c) {
    for (int j = 0; j < 4; ++j)
      if (!is_scale(c, j)) return j;
    return -1;
  }
  static constexpr int first_block(int c) { return block(c, first_word(c)); }
  static constexpr int last_block(int c) {
    int b = -1;
    for (int j = 0; j < 4; ++j)
      if (!is_scale(c, j)) b = block(c, j);
    return b;
  }
  static constexpr int scale_in_chunk(int c, int b) {
    return (17 * b - 4 * c >= 0 && 17 * b - 4 * c < 4) ? 17 * b - 4 * c : -1;
  }
};

template <int I>
__device__ __forceinline__ uint32_t word_of(const uint4 &w) {
  if constexpr (I == 0) return w.x;
  else if constexpr (I == 1) return w.y;
  else if constexpr (I == 2) return w.z;
  else return w.w;
}

template <int C, int B>
__device__ __forceinline__ uint32_t q8_scale_bits(const uint4 &w, uint32_t row_addr) {
  constexpr int o = Q8Geom::scale_in_chunk(C, B);
  if constexpr (o >= 0) {
    const uint32_t wd = word_of<o / 4>(w);
    return (o % 4 == 0) ? (wd & 0xFFFFu) : (wd >> 16);
  } else {
    return lds_u16(row_addr + 34 * B);
  }
}

template <int C, int B>
__device__ __forceinline__ uint32_t twin_scale_word(const uint4 &w, uint32_t row_addr) {
  constexpr int j = TwinGeom::scale_in_chunk(C, B);
  if constexpr (j >= 0) {
    return word_of<j>(w);
  } else {
    return lds32(row_addr + 68 * B);
  }
}

// One Q8 chunk C of one unit, for the lane's 4 rows.
template <int N, int C>
__device__ __forceinline__ void q8_chunk(uint32_t tile, uint32_t xsb, uint32_t lane,
                                         uint64_t (&acc)[kSlots][N]) {
  using T = Traits<Fmt::Q8, N>;
  constexpr int B0 = Q8Geom::first_block(C);
  constexpr int B1 = Q8Geom::last_block(C);
  constexpr int M0 = Q8Geom::first_pair(C);
  uint64_t xp[8][N];
  static_for<0, 8>([&](auto mc) {
    constexpr int m = decltype(mc)::value;
    if constexpr (!Q8Geom::is_scale(C, 2 * m)) {
      constexpr int cp = Q8Geom::col(C, 2 * m) / 2;
      const uint32_t a = xsb + cp * T::kNS * 8;
      if constexpr (T::kNS == 4) {
        uint64_t t2, t3;
        lds_2x64(a, xp[m][0], xp[m][1]);
        lds_2x64(a + 16, t2, t3);
        if constexpr (N >= 3) xp[m][2] = t2;
        if constexpr (N == 4) xp[m][3] = t3;
      } else if constexpr (T::kNS == 2) {
        lds_2x64(a, xp[m][0], xp[m][1]);
      } else {
        xp[m][0] = lds64(a);
      }
    }
  });
#pragma unroll
  for (int r = 0; r < kSlots; ++r) {
    const uint32_t row_addr = tile + (r * 32 + lane) * kSBBytes;
    const uint4 w = lds128(row_addr + 16 * C);
    const uint32_t wx[4] = {w.x ^ 0x80808080u, w.y ^ 0x80808080u, w.z ^ 0x80808080u,
                            w.w ^ 0x80808080u};
    const ScalePair s0 = make_scale(q8_scale_bits<C, B0>(w, row_addr));
    ScalePair s1 = s0;
    if constexpr (B1 != B0) s1 = make_scale(q8_scale_bits<C, B1>(w, row_addr));
    uint64_t p[N];
    static_for<0, 8>([&](auto mc) {
      constexpr int m = decltype(mc)::value;
      if constexpr (!Q8Geom::is_scale(C, 2 * m)) {
        constexpr int k = 2 * m;
        const ScalePair &sc = (Q8Geom::block(C, k) == B0) ? s0 : s1;
        const uint64_t wq = dequant2(wx[k / 4], k % 4, wx[k / 4], k % 4 + 1, sc);
        static_for<0, N>([&](auto sc_) {
          constexpr int s = decltype(sc_)::value;
          if constexpr (m == M0) p[s] = fmul2(wq, xp[m][s]);
          else p[s] = ffma2(wq, xp[m][s], p[s]);
        });
      }
    });
    static_for<0, N>([&](auto sc_) {
      constexpr int s = decltype(sc_)::value;
      acc[r][s] = fadd2(acc[r][s], p[s]);
    });
  }
}

// One twin chunk C of one unit, for the lane's 4 rows.
template <int C>
__device__ __forceinline__ void twin_chunk(uint32_t tile, uint32_t xsb, uint32_t lane,
                                           uint64_t (&acc)[kSlots][2]) {
  constexpr int B0 = TwinGeom::first_block(C);
  constexpr int B1 = TwinGeom::last_block(C);
  constexpr int J0 = TwinGeom::first_word(C);
  uint64_t xa[4], xb[4];
  static_for<0, 4>([&](auto jc) {
    constexpr int j = decltype(jc)::value;
    if constexpr (!TwinGeom::is_scale(C, j)) lds_2x64(xsb + TwinGeom::colpair(C, j) * 16, xa[j], xb[j]);
  });
#pragma unroll
  for (int r = 0; r < kSlots; ++r) {
    const uint32_t row_addr = tile + (r * 32 + lane) * kSBBytes;
    const uint4 w = lds128(row_addr + 16 * C);
    const uint32_t sw0 = twin_scale_word<C, B0>(w, row_addr);
    const ScalePair sa0 = make_scale(sw0 & 0xFFFFu), sb0 = make_scale(sw0 >> 16);
    ScalePair sa1 = sa0, sb1 = sb0;
    if constexpr (B1 != B0) {
      const uint32_t sw1 = twin_scale_word<C, B1>(w, row_addr);
      sa1 = make_scale(sw1 & 0xFFFFu);
      sb1 = make_scale(sw1 >> 16);
    }
    uint64_t pa, pb;
    static_for<0, 4>([&](auto jc) {
      constexpr int j = decltype(jc)::value;
      if constexpr (!TwinGeom::is_scale(C, j)) {
        const bool first_blk = TwinGeom::block(C, j) == B0;
        const ScalePair &sa = first_blk ? sa0 : sa1;
        const ScalePair &sb = first_blk ? sb0 : sb1;
        const uint32_t wxj = word_of<j>(w) ^ 0x80808080u;
        const uint64_t wa = dequant2(wxj, 1, wxj, 3, sa);  // model A: high bytes
        const uint64_t wb = dequant2(wxj, 0, wxj, 2, sb);  // model B: low bytes
        if constexpr (j == J0) {
          pa = fmul2(wa, xa[j]);
          pb = fmul2(wb, xb[j]);
        } else {
          pa = ffma2(wa, xa[j], pa);
          pb = ffma2(wb, xb[j], pb);
        }
      }
    });
    acc[r][0] = fadd2(acc[r][0], pa);
    acc[r][1] = fadd2(acc[r][1], pb);
  }
}

template <Fmt F, int N, int C>
__device__ __forceinline__ void chunk_body(uint32_t tile, uint32_t xsb, uint32_t lane,
                                           uint64_t (&acc)[kSlots][Traits<F, N>::kOut]) {
  if constexpr (F == Fmt::Q8) q8_chunk<N, C>(tile, xsb, lane, acc);
  else twin_chunk<C>(tile, xsb, lane, acc);
}

template <Fmt F, int N>
__device__ __forceinline__ void chunk_dispatch(int c, uint32_t tile, uint32_t xsb, uint32_t lane,
                                               uint64_t (&acc)[kSlots][Traits<F, N>::kOut]) {
#define PTI_CHUNK_CASE(C)                          \
  case C:                                          \
    chunk_body<F, N, C>(tile, xsb, lane, acc);     \
    break;
  switch (c) {
    PTI_CHUNK_CASE(0) PTI_CHUNK_CASE(1) PTI_CHUNK_CASE(2) PTI_CHUNK_CASE(3) PTI_CHUNK_CASE(4)
    PTI_CHUNK_CASE(5) PTI_CHUNK_CASE(6) PTI_CHUNK_CASE(7) PTI_CHUNK_CASE(8) PTI_CHUNK_CASE(9)
    PTI_CHUNK_CASE(10) PTI_CHUNK_CASE(11) PTI_CHUNK_CASE(12) PTI_CHUNK_CASE(13)
    case 14:
      if constexpr (Traits<F, N>::kWarps > 14) chunk_body<F, N, 14>(tile, xsb, lane, acc);
      break;
    default: break;
  }
#undef PTI_CHUNK_CASE
}

// Stages the activations of super-blocks [wa, wb) as float2 column pairs.
template <Fmt F, int N>
__device__ __forceinline__ void stage_x(const GemvArgs &a, float *xs, int32_t wa, int32_t wb,
                                        uint32_t tid) {
  using T = Traits<F, N>;
  constexpr int kConsumerThreads = T::kWarps * 32;
  const int64_t k0 = static_cast<int64_t>(wa) * T::kColsPerSB;
  const int32_t len = (wb - wa) * T::kColsPerSB;
  if constexpr (F == Fmt::Q8) {
    for (int32_t e = tid; e < N * len; e += kConsumerThreads) {
      const int32_t s = e / len, kk = e - s * len;
      xs[((kk >> 1) * T::kNS + s) * 2 + (kk & 1)] = a.x0[static_cast<int64_t>(s) * a.cols + k0 + kk];
    }
  } else {
    for (int32_t e = tid; e < 2 * len; e += kConsumerThreads) {
      const int32_t s = e / len, kk = e - s * len;
      const float *src = s ? a.x1 : a.x0;
      xs[((kk >> 1) * 2 + s) * 2 + (kk & 1)] = src[k0 + kk];
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

template <Fmt F, int N>
__global__ void __launch_bounds__(Traits<F, N>::kWarps * 32 + 32, 1)
    gemv_tma_kernel(const __grid_constant__ CUtensorMap tmap, const GemvArgs a) {
  using T = Traits<F, N>;
  constexpr int kOut = T::kOut;
  constexpr int kConsumerWarps = T::kWarps;
  constexpr int kConsumerThreads = kConsumerWarps * 32;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *const base_ptr = smem_raw + (base - raw);
  const uint32_t xreg = base + kStages * kStageBytes;
  float *const xs = reinterpret_cast<float *>(base_ptr + kStages * kStageBytes);
  const uint32_t bars = xreg + a.x_region_bytes;
  const uint32_t flags = bars + 2 * kStages * 8;
  volatile uint32_t *const flag =
      reinterpret_cast<volatile uint32_t *>(base_ptr + kStages * kStageBytes + a.x_region_bytes + 2 * kStages * 8);

  const uint32_t tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t u0 = static_cast<int64_t>(blockIdx.x) * a.units / a.grid;
  const int64_t u1 = static_cast<int64_t>(blockIdx.x + 1) * a.units / a.grid;

  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(bars + 8 * i, 1);
      mbar_init(bars + 8 * (kStages + i), kConsumerWarps);
    }
    flag[0] = 0;
    flag[1] = 0;
    mbar_init_fence();
  }
  __syncthreads();
  if (tid == 0) pdl_launch_dependents();

  if (warp == kConsumerWarps) {
    // ---------------- producer: one lane issues every tile copy -------------
    if (lane == 0) {
      prefetch_tmap(&tmap);
      const uint64_t pol = l2_policy_evict_first();
      const int64_t nu = u1 - u0;
      int64_t issued = 0;
      for (int64_t i = 0; i < nu; ++i) {
        const int stage = static_cast<int>(i % kStages);
        const int64_t j = i / kStages;
        if (j > 0 && !mbar_wait_bounded(bars + 8 * (kStages + stage), static_cast<uint32_t>((j - 1) & 1), flags)) {
          if (flag[0] == 0) atomicOr(&g_device_error, PTI_DEVERR_EMPTY_TIMEOUT);
          flag[0] = 1;
          break;
        }
        if (flag[0] != 0) break;
        const int64_t u = u0 + i;
        const int32_t rb = static_cast<int32_t>(u / a.n_sb);
        const int32_t sb = static_cast<int32_t>(u - static_cast<int64_t>(rb) * a.n_sb);
        mbar_arrive_expect_tx(bars + 8 * stage, kStageBytes);
        tma_load_2d(base + stage * kStageBytes, &tmap, 34 * sb, rb * kRowsPerTile, bars + 8 * stage, pol);
        issued = i + 1;
      }
      // Stay until every copy issued into this CTA's shared memory has landed.
      for (int64_t i = (issued > kStages ? issued - kStages : 0); i < issued; ++i) {
        if (!mbar_wait_bounded(bars + 8 * (i % kStages), static_cast<uint32_t>((i / kStages) & 1), 0))
          atomicOr(&g_device_error, PTI_DEVERR_DRAIN_TIMEOUT);
      }
    }
    return;
  }

  // ---------------- consumers ----------------------------------------------
  pdl_wait_primary();  // x may come from the previous kernel in the stream
  uint64_t acc[kSlots][kOut];
  int64_t i = 0;
  const int32_t rb_first = static_cast<int32_t>(u0 / a.n_sb);
  const int32_t rb_last = static_cast<int32_t>((u1 - 1) / a.n_sb);
  for (int32_t rb = rb_first; rb <= rb_last; ++rb) {
    const int32_t sb_begin = (rb == rb_first) ? static_cast<int32_t>(u0 - static_cast<int64_t>(rb) * a.n_sb) : 0;
    const int32_t sb_end = (rb == rb_last) ? static_cast<int32_t>(u1 - static_cast<int64_t>(rb) * a.n_sb) : a.n_sb;
#pragma unroll
    for (int r = 0; r < kSlots; ++r)
#pragma unroll
      for (int s = 0; s < kOut; ++s) acc[r][s] = 0ull;

    for (int32_t wa = sb_begin; wa < sb_end; wa += a.xw_sb) {
      const int32_t wb = min(sb_end, wa + a.xw_sb);
      named_barrier(kBarConsumers, kConsumerThreads);  // x region free
      stage_x<F, N>(a, xs, wa, wb, tid);
      named_barrier(kBarConsumers, kConsumerThreads);
      for (int32_t sb = wa; sb < wb; ++sb, ++i) {
        const int stage = static_cast<int>(i % kStages);
        bool ok = flag[0] == 0;
        if (ok) ok = mbar_wait_bounded(bars + 8 * stage, static_cast<uint32_t>((i / kStages) & 1), flags);
        if (!ok && flag[0] == 0) {
          atomicOr(&g_device_error, PTI_DEVERR_FULL_TIMEOUT);
          flag[0] = 1;
        }
        if (ok) {
          const uint32_t tile = base + stage * kStageBytes;
          const uint32_t xsb = xreg + (sb - wa) * T::kXBytesPerSB;
          // warp w owns chunk w; the 17 - kConsumerWarps remaining chunks rotate
          chunk_dispatch<F, N>(static_cast<int>(warp), tile, xsb, lane, acc);
          constexpr int kExtra = 17 - kConsumerWarps;
          const int64_t e0 = static_cast<int64_t>(kExtra) * i;
          if constexpr (kExtra == 3) {
            if (warp == static_cast<uint32_t>(e0 % kConsumerWarps)) chunk_body<F, N, 14>(tile, xsb, lane, acc);
          }
          if (warp == static_cast<uint32_t>((e0 + kExtra - 2) % kConsumerWarps))
            chunk_body<F, N, 15>(tile, xsb, lane, acc);
          if (warp == static_cast<uint32_t>((e0 + kExtra - 1) % kConsumerWarps))
            chunk_body<F, N, 16>(tile, xsb, lane, acc);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bars + 8 * (kStages + stage));
      }
    }

    // ---- reduce the 15 warps' partial sums of this row tile (fixed order) ----
    named_barrier(kBarConsumers, kConsumerThreads);  // every warp is done with x
    float *const red = xs;                            // [warp][kOut][128]
#pragma unroll
    for (int r = 0; r < kSlots; ++r)
#pragma unroll
      for (int s = 0; s < kOut; ++s) {
        const float2 v = unpack2(acc[r][s]);
        red[(warp * kOut + s) * kRowsPerTile + r * 32 + lane] = v.x + v.y;
      }
    named_barrier(kBarConsumers, kConsumerThreads);

    const int32_t c_lo = cta_of_unit(static_cast<int64_t>(rb) * a.n_sb, a.units, a.grid);
    const int32_t c_hi = cta_of_unit(static_cast<int64_t>(rb + 1) * a.n_sb - 1, a.units, a.grid);
    const bool shared_tile = c_hi > c_lo;
    const int slot = (rb == rb_first) ? 0 : 1;
    for (int t = tid; t < kOut * kRowsPerTile; t += kConsumerThreads) {
      const int s = t / kRowsPerTile, row = t - s * kRowsPerTile;
      float v[kConsumerWarps];
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) v[w] = red[(w * kOut + s) * kRowsPerTile + row];
      const float total = tree_sum(v);
      const int64_t row_g = static_cast<int64_t>(rb) * kRowsPerTile + row;
      if (!shared_tile) {
        if (row_g < a.rows) {
          if constexpr (F == Fmt::Q8) a.y0[s * a.rows + row_g] = total;
          else (s == 0 ? a.y0 : a.y1)[row_g] = total;
        }
      } else {
        a.part[((static_cast<int64_t>(blockIdx.x) * 2 + slot) * kOut + s) * kRowsPerTile + row] = total;
      }
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
      if (flag[1] != 0) {
        for (int t = tid; t < kOut * kRowsPerTile; t += kConsumerThreads) {
          const int s = t / kRowsPerTile, row = t - s * kRowsPerTile;
          float total = 0.0f;
          for (int32_t c = c_lo; c <= c_hi; ++c) {
            const int sl = (rb == first_tile_of_cta(c, a.units, a.grid, a.n_sb)) ? 0 : 1;
            const float v = __ldcg(&a.part[((static_cast<int64_t>(c) * 2 + sl) * kOut + s) * kRowsPerTile + row]);
            total = (c == c_lo) ? v : total + v;
          }
          const int64_t row_g = static_cast<int64_t>(rb) * kRowsPerTile + row;
          if (row_g < a.rows) {
            if constexpr (F == Fmt::Q8) a.y0[s * a.rows + row_g] = total;
            else (s == 0 ? a.y0 : a.y1)[row_g] = total;
          }
        }
      }
    }
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
  int32_t grid = 0, xw_sb = 0;
  uint32_t x_region = 0;
  size_t smem = 0;
};

template <Fmt F, int N>
TilePlan plan_tiles(int64_t rows, int64_t cols, int sms) {
  using T = Traits<F, N>;
  TilePlan p;
  p.n_sb = cols / T::kColsPerSB;
  p.n_rb = (rows + kRowsPerTile - 1) / kRowsPerTile;
  p.units = p.n_sb * p.n_rb;
  p.grid = static_cast<int32_t>(std::min<int64_t>({static_cast<int64_t>(sms), p.units, kMaxGrid}));
  const int64_t per_cta = (p.units + p.grid - 1) / p.grid;
  const int64_t red_bytes = static_cast<int64_t>(T::kWarps) * T::kOut * kRowsPerTile * 4;
  const int64_t avail = kSmemOptin - 1024 - static_cast<int64_t>(kStages) * kStageBytes - kBarBytes;
  p.xw_sb = static_cast<int32_t>(std::max<int64_t>(1, std::min<int64_t>(per_cta, avail / T::kXBytesPerSB)));
  p.x_region = static_cast<uint32_t>(std::max<int64_t>(static_cast<int64_t>(p.xw_sb) * T::kXBytesPerSB, red_bytes));
  p.x_region = (p.x_region + 15u) & ~15u;
  p.smem = 1024 + static_cast<size_t>(kStages) * kStageBytes + p.x_region + kBarBytes;
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
                       float *y0, float *y1, void *workspace, cudaStream_t stream) {
  using T = Traits<F, N>;
  int dev = 0;
  const int sms = current_device_sms(&dev);
  if (sms <= 0) return PTI_ERR_CUDA;
  const TilePlan p = plan_tiles<F, N>(rows, cols, sms);
  if (p.smem > static_cast<size_t>(kSmemOptin)) return PTI_ERR_SHAPE;

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
  a.xw_sb = p.xw_sb;
  a.x_region_bytes = p.x_region;
  gemv_tma_kernel<F, N><<<p.grid, T::kWarps * 32 + 32, p.smem, stream>>>(tmap, a);
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
  if (need > 0) {
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
    return launch_fast<Fmt::Twin, 2>(w_twin, rows, cols, x_a, x_b, y_a, y_b, workspace, st);
  }
  const int sms = current_device_sms();
  if (sms <= 0) return PTI_ERR_CUDA;
  const int64_t blocks = std::min<int64_t>((rows + 7) / 8, static_cast<int64_t>(sms) * 16);
  twin_rowwise_kernel<<<static_cast<unsigned>(blocks), 256, 0, st>>>(static_cast<const uint8_t *>(w_twin), rows, cols,
                                                                     x_a, x_b, y_a, y_b);
  return launch_status();
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
