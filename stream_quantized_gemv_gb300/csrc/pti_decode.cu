// pti_decode.cu -- the chained decode pass on sm_103a: n_layers gated-MLP
// layers over N token streams, every weight byte streamed once per pass for
// all N streams.
//
// [PTI-readme] "打包双子推理（PTI）" §"带宽分析：为什么会有开销": a decode step costs
// one pass over the weights however many streams share it, so N streams cost
// about one single-stream step.  The layer is the gated MLP (W_gate, W_up,
// W_down) of [CS336-L10] "推理（Inference）" §"2.4 MLP 层的算术强度"; the
// pages name neither its nonlinearity nor a normalisation, and this library
// takes SiLU and an RMS rescale (v / sqrt(mean(v^2) + eps)) after h and after
// the layer.
//
// Per layer l (x = the normalised input, x' = the raw output of the previous
// down projection, x = b x' with b its RMS scale; b = 1 for the first layer):
//   kernel GateUp:  tile = 64 rows of W_gate and the same 64 rows of W_up;
//                   g, u = W x' (N streams), h = SiLU(b g) * (b u) -> h,
//                   per-tile sums of h^2 -> sq_h.
//   kernel Down:    x'' = a (W_down h) with a = 1 / sqrt(sum(sq_h)/ffn + eps),
//                   per-tile sums of x''^2 -> sq_x.
// then one finalise kernel: x_out = b x'' (b from sq_x).  After each GEMV a
// small kernel combines the row tiles that several CTAs shared.  Every kernel
// after the first is launched with programmatic
// dependent launch; each waits for its predecessor to complete before it reads
// anything but weights or writes anything, so one buffer of each kind serves
// every layer.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <vector>

#include "pti.h"
#include "pti_gemv_kernel.cuh"
#include "pti_host.h"

namespace pti {
namespace {

constexpr int kFinalizeThreads = 256;
constexpr int kMaxLayersPerLaunch = 64;  // layers per launch of the persistent pass
constexpr int kMaxLaunches = 64;         // so at most 4096 layers per call

// Workspace of one pass, byte offsets (each 256-byte aligned).
struct DecodeLayout {
  int64_t n_rb_gu = 0, n_rb_down = 0;  // tiles of the GateUp and Down kernels
  size_t part = 0, tickets = 0, counter = 0, grid_bars = 0, h = 0, xraw = 0, sq_h = 0, sq_x = 0, scales = 0, total = 0;
};

size_t round256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

DecodeLayout decode_layout(int64_t hidden, int64_t ffn, int n) {
  DecodeLayout d;
  d.n_rb_gu = (ffn + 63) / 64;
  d.n_rb_down = (hidden + kRowsPerTile - 1) / kRowsPerTile;
  size_t off = 0;
  d.part = off;
  off += partial_bytes(n);
  d.tickets = off;
  off += static_cast<size_t>(std::max(d.n_rb_gu, d.n_rb_down)) * sizeof(unsigned int);
  d.counter = off;
  off += sizeof(unsigned int);
  d.grid_bars = off;  // one grid-barrier counter per launch of the persistent pass
  off = round256(off + kMaxLaunches * sizeof(unsigned int));
  d.h = off;
  off = round256(off + static_cast<size_t>(n) * ffn * sizeof(float));
  d.xraw = off;
  off = round256(off + static_cast<size_t>(n) * hidden * sizeof(float));
  d.sq_h = off;
  off = round256(off + static_cast<size_t>(d.n_rb_gu) * n * sizeof(float));
  d.sq_x = off;
  off = round256(off + static_cast<size_t>(d.n_rb_down) * n * sizeof(float));
  d.scales = off;  // the chained pass: input scales of the GateUp and of the Down step, [2][n]
  off = round256(off + 2 * static_cast<size_t>(n) * sizeof(float));
  d.total = off;
  return d;
}

pti_status check_decode_shape(int64_t hidden, int64_t ffn) {
  if (hidden < 256 || ffn < 256 || hidden % 256 != 0 || ffn % 256 != 0) return PTI_ERR_SHAPE;
  if (check_gemv_shape(ffn, hidden) != PTI_OK || check_gemv_shape(hidden, ffn) != PTI_OK) return PTI_ERR_SHAPE;
  return PTI_OK;
}

struct FinalizeArgs {
  const float *xraw;        // [n][hidden] the last layer's raw output
  const float *sq_x;        // [n_rb_down][n] its per-tile sums of squares
  float *x_out;             // [n][hidden]
  int64_t hidden;
  int32_t n_rb_down;
  double inv_hidden, eps;
};

// x_out = b x'' with b the RMS scale of the last layer's output.
template <int N>
__global__ void __launch_bounds__(kFinalizeThreads) rms_finalize_kernel(const FinalizeArgs f) {
  __shared__ float scale[4];
  const uint32_t tid = threadIdx.x, warp = tid >> 5, lane = tid & 31u;
  pdl_launch_dependents();
  pdl_wait_primary();
  if (warp < static_cast<uint32_t>(N)) {
    double s2 = 0.0;
    for (int32_t t = static_cast<int32_t>(lane); t < f.n_rb_down; t += 32)
      s2 += static_cast<double>(__ldcg(f.sq_x + static_cast<int64_t>(t) * N + warp));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s2 += __shfl_xor_sync(0xFFFFFFFFu, s2, o);
    if (lane == 0) scale[warp] = rms_inv_scale(s2, f.inv_hidden, f.eps);
  }
  __syncthreads();
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kFinalizeThreads;
  const int64_t first = static_cast<int64_t>(blockIdx.x) * kFinalizeThreads + tid;
  for (int64_t i = first; i < N * f.hidden; i += stride) {
    const int s = static_cast<int>(i / f.hidden);
    f.x_out[i] = __ldcg(f.xraw + i) * scale[s];
  }
}

// ---------------------------------------------------------------------------
// Persistent pass: one cooperative launch runs up to kMaxLayersPerLaunch
// layers.  The phases (GateUp of layer 0, Down of layer 0, GateUp of layer
// 1, ...) are separated by a grid barrier (every CTA is resident, which the
// cooperative launch guarantees).  The producer warp streams the weights of
// the next phase into the ring while the consumers finish the current phase
// and cross the barrier, so HBM keeps streaming through the phase changes;
// only activation copies wait for the barrier.
// ---------------------------------------------------------------------------
struct DecodeKernelParams {
  CUtensorMap maps[kMaxLayersPerLaunch][3];  // gate, up (boxes of 64 rows), down (128 rows)
  const float *x_in;        // this launch's input: x_in of the call, or x' of the previous launch
  float *h, *xraw, *sq_h, *sq_x, *part;
  unsigned int *tickets;
  unsigned int *grid_bar;   // this launch's arrival counter (zero at start)
  int64_t hidden, ffn;
  int32_t n_layers, grid, stages;
  int32_t input_scaled;     // 0: x_in is used as is; 1: x_in = x' of a previous launch (scale from sq_x)
  double eps;
};

static_assert(sizeof(DecodeKernelParams) <= 32764, "kernel parameters are limited to 32764 bytes");

// One phase of the pass: its GEMV geometry, buffers and epilogue.
struct Phase {
  bool gateup;
  int64_t rows, cols, units;
  int32_t n_sb, n_rb;
  const float *x0;
  float *y0, *sq_out;
  const float *sq_in;       // null: input scale 1
  int32_t n_sq_in;
  double inv_len;
  const CUtensorMap *m0, *m1;
};

__device__ __forceinline__ Phase make_phase(const DecodeKernelParams &P, int p) {
  Phase ph;
  const int l = p >> 1;
  ph.gateup = (p & 1) == 0;
  const int32_t n_rb_gu = static_cast<int32_t>(P.ffn / 64), n_rb_dn = static_cast<int32_t>(P.hidden / kRowsPerTile);
  if (ph.gateup) {
    ph.rows = P.ffn;
    ph.cols = P.hidden;
    ph.n_sb = static_cast<int32_t>(P.hidden / 256);
    ph.n_rb = n_rb_gu;
    ph.x0 = (l == 0) ? P.x_in : P.xraw;
    ph.y0 = P.h;
    ph.sq_out = P.sq_h;
    ph.sq_in = (l == 0 && !P.input_scaled) ? nullptr : P.sq_x;
    ph.n_sq_in = n_rb_dn;
    ph.inv_len = 1.0 / static_cast<double>(P.hidden);
    ph.m0 = &P.maps[l][0];
    ph.m1 = &P.maps[l][1];
  } else {
    ph.rows = P.hidden;
    ph.cols = P.ffn;
    ph.n_sb = static_cast<int32_t>(P.ffn / 256);
    ph.n_rb = n_rb_dn;
    ph.x0 = P.h;
    ph.y0 = P.xraw;
    ph.sq_out = P.sq_x;
    ph.sq_in = P.sq_h;
    ph.n_sq_in = n_rb_gu;
    ph.inv_len = 1.0 / static_cast<double>(P.ffn);
    ph.m0 = &P.maps[l][2];
    ph.m1 = nullptr;
  }
  ph.units = static_cast<int64_t>(ph.n_sb) * ph.n_rb;
  return ph;
}

__device__ __forceinline__ unsigned int ld_acquire_gpu(const unsigned int *p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Waits (bounded) until `count` CTAs have arrived at the counter.  Returns
// false on timeout or when this CTA's abort flag is raised.
__device__ __noinline__ bool grid_wait(const unsigned int *ctr, unsigned int count, volatile uint32_t *flag) {
  if (ld_acquire_gpu(ctr) >= count) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1; i < (1u << 30); ++i) {
    if (ld_acquire_gpu(ctr) >= count) return true;
    if ((i & 15u) == 0) {
      if (flag[0] != 0) return false;
      if (globaltimer_ns() - t0 > kWaitTimeoutNs) return false;
    }
    __nanosleep(64);
  }
  return false;
}

template <int N>
__global__ void __launch_bounds__(kWarpCount * 32 + 32, 1)
    decode_pass_kernel(const __grid_constant__ DecodeKernelParams P) {
  using T = Traits<Fmt::Q8, N>;
  using S = Stage<Fmt::Q8, N>;
  constexpr int kOut = N;
  constexpr int kConsumerWarps = kWarpCount;
  constexpr int kConsumerThreads = kConsumerWarps * 32;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *const base_ptr = smem_raw + (base - raw);
  const int stages = P.stages;
  float *const red = reinterpret_cast<float *>(base_ptr + stages * S::kBytes);
  const uint32_t bars = base + stages * S::kBytes + S::kRedBytes;  // full[stages], empty[stages], scale_ready
  const uint32_t scale_bar = bars + 16 * stages;
  const uint32_t flags = scale_bar + 8;
  volatile uint32_t *const flag = reinterpret_cast<volatile uint32_t *>(base_ptr + (flags - base));
  float *const epi = reinterpret_cast<float *>(base_ptr + (flags - base) + 16);
  float *const scale = epi + 4 * kRowsPerTile;
  const uint32_t tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_phases = 2 * P.n_layers;
  const int32_t G = P.grid;

  if (tid == 0) {
    for (int i = 0; i < stages; ++i) {
      mbar_init(bars + 8 * i, 1);
      mbar_init(bars + 8 * (stages + i), kConsumerWarps);
    }
    mbar_init(scale_bar, 1);
    flag[0] = 0;
    flag[1] = 0;
    mbar_init_fence();
  }
  __syncthreads();
  if (tid == 0) pdl_launch_dependents();

  if (warp == kConsumerWarps) {
    // ---------------- producer warp ------------------------------------------
    // Lane 0 issues every copy; all lanes compute each phase's input scales.
    const uint64_t pol = l2_policy_evict_first();
    int64_t g = 0;                    // global unit index of this CTA (over all phases)
    int64_t pend_g[kMaxStages];       // units whose activations wait for the grid barrier
    int64_t pend_i[kMaxStages];
    int n_pend = 0;
    bool ok = true;
    if (lane == 0) pdl_wait_primary();  // the input and its sums of squares come from earlier work
    __syncwarp();
    for (int p = 0; p < n_phases && ok; ++p) {
      const Phase ph = make_phase(P, p);
      const int64_t u0 = static_cast<int64_t>(blockIdx.x) * ph.units / G;
      const int64_t u1 = static_cast<int64_t>(blockIdx.x + 1) * ph.units / G;
      bool passed = (p == 0);         // activations of phase p need every CTA done with phase p - 1
      auto load_x = [&](int64_t i, uint32_t slot) {
        const int32_t rb = static_cast<int32_t>(i / ph.n_sb);
        const int32_t sb = static_cast<int32_t>(i - static_cast<int64_t>(rb) * ph.n_sb);
        (void)rb;
        const uint32_t xdst = base + slot * S::kBytes + kStageBytes, bar = bars + 8 * slot;
        mbar_arrive_expect_tx(bar, S::kXBytes);
#pragma unroll
        for (int s = 0; s < N; ++s)
          bulk_load(xdst + s * S::kXStreamBytes, ph.x0 + static_cast<int64_t>(s) * ph.cols + static_cast<int64_t>(sb) * 256,
                    S::kXStreamBytes, bar);
      };
      // Once the barrier is passed: the pending activation copies first (the
      // consumers wait for them), then the input scales of this phase (needed
      // only when the phase's tiles are finished; published through scale_bar).
      auto on_passed = [&]() {
        if (lane == 0) {
          fence_proxy_async_global();  // the activations were written by other CTAs' threads
          for (int k = 0; k < n_pend; ++k) load_x(pend_i[k], static_cast<uint32_t>(pend_g[k] % stages));
        }
        n_pend = 0;
        passed = true;
        double s2[kOut];
#pragma unroll
        for (int s = 0; s < kOut; ++s) s2[s] = 0.0;
        if (ph.sq_in != nullptr) {
#pragma unroll 4
          for (int32_t t = static_cast<int32_t>(lane); t < ph.n_sq_in; t += 32)
#pragma unroll
            for (int s = 0; s < kOut; ++s) s2[s] += static_cast<double>(__ldcg(ph.sq_in + static_cast<int64_t>(t) * kOut + s));
        }
#pragma unroll
        for (int s = 0; s < kOut; ++s)
          for (int o = 16; o > 0; o >>= 1) s2[s] += __shfl_xor_sync(0xFFFFFFFFu, s2[s], o);
        if (lane == 0) {
#pragma unroll
          for (int s = 0; s < kOut; ++s)
            scale[s] = ph.sq_in != nullptr ? rms_inv_scale(s2[s], ph.inv_len, P.eps) : 1.0f;
          mbar_arrive(scale_bar);
        }
      };
      if (passed) on_passed();
      for (int64_t i = u0; i < u1 && ok; ++i, ++g) {
        const uint32_t slot = static_cast<uint32_t>(g % stages);
        if (!passed && n_pend == stages) {
          // the ring holds only units waiting for the barrier: wait for it
          bool w = true;
          if (lane == 0) w = grid_wait(P.grid_bar, static_cast<unsigned int>(p) * G, flag);
          w = __shfl_sync(0xFFFFFFFFu, w, 0);
          if (!w) {
            ok = false;
            break;
          }
          on_passed();
        }
        bool w = true;
        if (lane == 0) {
          if (g >= stages) {
            const uint32_t empty = bars + 8 * (stages + slot);
            const uint32_t eph = static_cast<uint32_t>(((g / stages) - 1) & 1);
            w = mbar_try_wait(empty, eph) || mbar_wait_bounded(empty, eph, flags);
          }
          if (w && flag[0] == 0) {
            const int32_t rb = static_cast<int32_t>(i / ph.n_sb);
            const int32_t sb = static_cast<int32_t>(i - static_cast<int64_t>(rb) * ph.n_sb);
            const uint32_t dst = base + slot * S::kBytes, bar = bars + 8 * slot;
            mbar_expect_tx(bar, kStageBytes);
            if (ph.gateup) {
              tma_load_2d(dst, ph.m0, 34 * sb, rb * 64, bar, pol);
              tma_load_2d(dst + 64 * kSBBytes, ph.m1, 34 * sb, rb * 64, bar, pol);
            } else {
              tma_load_2d(dst, ph.m0, 34 * sb, rb * kRowsPerTile, bar, pol);
            }
            if (passed) load_x(i, slot);
          } else {
            w = false;
          }
        }
        w = __shfl_sync(0xFFFFFFFFu, w, 0);
        if (!w) {
          ok = false;
          break;
        }
        if (!passed) {
          pend_g[n_pend] = g;
          pend_i[n_pend] = i;
          ++n_pend;
          // poll the barrier without blocking
          bool now = false;
          if (lane == 0) now = ld_acquire_gpu(P.grid_bar) >= static_cast<unsigned int>(p) * G;
          now = __shfl_sync(0xFFFFFFFFu, now, 0);
          if (now) on_passed();
        }
      }
      if (ok && !passed) {
        bool w = true;
        if (lane == 0) w = grid_wait(P.grid_bar, static_cast<unsigned int>(p) * G, flag);
        w = __shfl_sync(0xFFFFFFFFu, w, 0);
        if (!w) ok = false;
        else on_passed();
      }
    }
    if (!ok && lane == 0) {
      if (flag[0] == 0) atomicOr(&g_device_error, PTI_DEVERR_EMPTY_TIMEOUT);
      flag[0] = 1;
    }
    // stay until every copy issued into this CTA's shared memory has landed
    if (lane == 0)
      for (int64_t k = (g > stages ? g - stages : 0); k < g; ++k)
        if (!mbar_wait_bounded(bars + 8 * (k % stages), static_cast<uint32_t>((k / stages) & 1), 0))
          atomicOr(&g_device_error, PTI_DEVERR_DRAIN_TIMEOUT);
    return;
  }

  // ---------------- consumers ------------------------------------------------
  const uint32_t half = warp >> 3, blk = warp & 7u;
  const uint32_t win_off = 32u * blk;
  const bool c_hi = (blk & 4u) != 0u;
  auto run = [&](auto ec, auto cc) {
    constexpr int E_ = decltype(ec)::value;
    constexpr int C_ = decltype(cc)::value;
    uint32_t st = 0, phs = 0;
    int64_t i = 0;
    for (int p = 0; p < n_phases; ++p) {
      const Phase ph = make_phase(P, p);
      GemvArgs a = {};
      a.y0 = ph.y0;
      a.part = P.part;
      a.tickets = P.tickets;
      a.combine_in_kernel = 1;
      a.rows = ph.rows;
      a.cols = ph.cols;
      a.units = ph.units;
      a.n_sb = ph.n_sb;
      a.n_rb = ph.n_rb;
      a.grid = G;
      a.stages = stages;
      a.sq_out = ph.sq_out;
      const int64_t u0 = static_cast<int64_t>(blockIdx.x) * ph.units / G;
      const int64_t u1 = static_cast<int64_t>(blockIdx.x + 1) * ph.units / G;
      bool scales_ready = false;
      auto finish = [&](int count, int32_t rb0, int sl0, int32_t rb1, int sl1) {
        if (!scales_ready) {
          if (!mbar_try_wait(scale_bar, static_cast<uint32_t>(p & 1)) &&
              !mbar_wait_bounded(scale_bar, static_cast<uint32_t>(p & 1), flags)) {
            if (flag[0] == 0) atomicOr(&g_device_error, PTI_DEVERR_FULL_TIMEOUT);
            flag[0] = 1;
          }
          scales_ready = true;
        }
        if (ph.gateup) finish_tiles<Fmt::Q8, N, Epi::GateUp>(a, red, count, rb0, sl0, rb1, sl1, tid, flag, epi);
        else finish_tiles<Fmt::Q8, N, Epi::Down>(a, red, count, rb0, sl0, rb1, sl1, tid, flag, epi);
      };
      uint64_t acc[kTaskSlots][kOut];
      const int32_t rb_first = static_cast<int32_t>(u0 / ph.n_sb);
      const int32_t rb_last = static_cast<int32_t>((u1 - 1) / ph.n_sb);
      for (int32_t rb = rb_first; rb <= rb_last; ++rb) {
        const int32_t sb_begin = (rb == rb_first) ? static_cast<int32_t>(u0 - static_cast<int64_t>(rb) * ph.n_sb) : 0;
        const int32_t sb_end = (rb == rb_last) ? static_cast<int32_t>(u1 - static_cast<int64_t>(rb) * ph.n_sb) : ph.n_sb;
#pragma unroll
        for (int r = 0; r < kTaskSlots; ++r)
#pragma unroll
          for (int s = 0; s < kOut; ++s) acc[r][s] = 0ull;
        for (int32_t sb = sb_begin; sb < sb_end; ++sb, ++i) {
          const uint32_t full = bars + 8 * st;
          bool ok = mbar_try_wait(full, phs);
          if (!ok) {
            ok = flag[0] == 0 && mbar_wait_bounded(full, phs, flags);
            if (!ok && flag[0] == 0) {
              atomicOr(&g_device_error, PTI_DEVERR_FULL_TIMEOUT);
              flag[0] = 1;
            }
          }
          if (ok) {
            const uint8_t *tile = base_ptr + st * S::kBytes;
            q8_block_body<N, E_, C_>(tile, tile + kStageBytes + 128u * blk, lane, half, win_off, c_hi, acc);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(bars + 8 * (stages + st));
          if (++st == static_cast<uint32_t>(stages)) {
            st = 0;
            phs ^= 1u;
          }
        }
        const int sl = (rb == rb_first) ? 0 : 1;
#pragma unroll
        for (int r = 0; r < kTaskSlots; ++r)
#pragma unroll
          for (int s = 0; s < kOut; ++s) {
            const float2 v = unpack2(acc[r][s]);
            red[((sl * kConsumerWarps + warp) * kOut + s) * 64 + r * 32 + lane] = v.x + v.y;
          }
        if (rb != rb_first && rb != rb_last) {
          named_barrier(kBarConsumers, kConsumerThreads);
          finish(1, rb, 1, 0, 0);
          named_barrier(kBarConsumers, kConsumerThreads);
        }
      }
      named_barrier(kBarConsumers, kConsumerThreads);
      finish(rb_last != rb_first ? 2 : 1, rb_first, 0, rb_last, 1);
      // this CTA is done with phase p: arrive at the grid barrier
      __threadfence();
      named_barrier(kBarConsumers, kConsumerThreads);
      if (tid == 0) atomicAdd(P.grid_bar, 1u);
    }
  };
  switch (blk & 3u) {  // = warp % 4: one code body per scheduler
    case 0: run(std::integral_constant<int, 0>{}, std::integral_constant<int, 0>{}); break;
    case 1: run(std::integral_constant<int, 1>{}, std::integral_constant<int, 0>{}); break;
    case 2: run(std::integral_constant<int, 0>{}, std::integral_constant<int, 1>{}); break;
    default: run(std::integral_constant<int, 1>{}, std::integral_constant<int, 1>{}); break;
  }
}

// Final kernel of a pass: applies the last RMS scale and zeroes the scratch.
template <int N>
pti_status launch_finalize(const DecodeLayout &d, uint8_t *ws, int64_t hidden, double eps, float *x_out,
                           cudaStream_t stream) {
  FinalizeArgs f;
  f.xraw = reinterpret_cast<const float *>(ws + d.xraw);
  f.sq_x = reinterpret_cast<const float *>(ws + d.sq_x);
  f.x_out = x_out;
  f.hidden = hidden;
  f.n_rb_down = static_cast<int32_t>(d.n_rb_down);
  f.inv_hidden = 1.0 / static_cast<double>(hidden);
  f.eps = eps;
  const int sms = current_device_sms();
  if (sms <= 0) return PTI_ERR_CUDA;
  const int64_t blocks = std::min<int64_t>(sms, (static_cast<int64_t>(N) * hidden + kFinalizeThreads - 1) / kFinalizeThreads);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(kFinalizeThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, rms_finalize_kernel<N>, f) != cudaSuccess) return launch_status();
  return launch_status();
}

// The pass as 2 n_layers separate GEMV launches chained by programmatic
// dependent launch.
template <int N>
pti_status run_decode_chained(const void *const *w_gate, const void *const *w_up, const void *const *w_down,
                              int n_layers, int64_t hidden, int64_t ffn, double eps, const float *x_in, float *x_out,
                              void *workspace, cudaStream_t stream) {
  const DecodeLayout d = decode_layout(hidden, ffn, N);
  uint8_t *const ws = static_cast<uint8_t *>(workspace);
  float *const h = reinterpret_cast<float *>(ws + d.h);
  float *const xraw = reinterpret_cast<float *>(ws + d.xraw);
  float *const sq_h = reinterpret_cast<float *>(ws + d.sq_h);
  float *const sq_x = reinterpret_cast<float *>(ws + d.sq_x);
  float *const scales = reinterpret_cast<float *>(ws + d.scales);
  GemvArgs base = {};
  base.part = reinterpret_cast<float *>(ws + d.part);
  base.tickets = reinterpret_cast<unsigned int *>(ws + d.tickets);
  base.eps = eps;
  base.prefetch_all = 1;
  for (int l = 0; l < n_layers; ++l) {
    GemvArgs gu = base;
    gu.x0 = (l == 0) ? x_in : xraw;
    gu.y0 = h;
    gu.rows = ffn;
    gu.cols = hidden;
    gu.sq_in = (l == 0) ? nullptr : sq_x;
    gu.n_sq_in = static_cast<int32_t>(d.n_rb_down);
    gu.inv_len_in = 1.0 / static_cast<double>(hidden);
    gu.sq_out = sq_h;
    gu.scale_out = scales;
    if (const pti_status s = launch_gemv<Fmt::Q8, N, Epi::GateUp>(w_gate[l], w_up[l], gu, stream, l > 0);
        s != PTI_OK)
      return s;
    GemvArgs dn = base;
    dn.x0 = h;
    dn.y0 = xraw;
    dn.rows = hidden;
    dn.cols = ffn;
    dn.sq_in = sq_h;
    dn.n_sq_in = static_cast<int32_t>(d.n_rb_gu);
    dn.inv_len_in = 1.0 / static_cast<double>(ffn);
    dn.sq_out = sq_x;
    dn.scale_out = scales + N;
    if (const pti_status s = launch_gemv<Fmt::Q8, N, Epi::Down>(w_down[l], nullptr, dn, stream, true); s != PTI_OK)
      return s;
  }
  return launch_finalize<N>(d, ws, hidden, eps, x_out, stream);
}

// Shared memory of the persistent kernel: the ring, the parked warp sums,
// full/empty barriers plus the scales barrier, flags and epilogue scratch.
template <int N>
size_t decode_fixed_smem() {
  return 1024 + Stage<Fmt::Q8, N>::kRedBytes + 8 * (2 * kMaxStages + 1) + 16 + kEpiBytes;
}

// The pass as cooperative persistent launches of up to kMaxLayersPerLaunch
// layers each.  Returns PTI_ERR_CUDA (having launched nothing) when the
// device cannot run a cooperative grid of one CTA per SM.
template <int N>
pti_status run_decode_persistent(const void *const *w_gate, const void *const *w_up, const void *const *w_down,
                                 int n_layers, int64_t hidden, int64_t ffn, double eps, const float *x_in,
                                 float *x_out, void *workspace, cudaStream_t stream) {
  using S = Stage<Fmt::Q8, N>;
  int dev = 0;
  const int sms = current_device_sms(&dev);
  if (sms <= 0) return PTI_ERR_CUDA;
  int coop = 0;
  if (cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess || coop == 0) {
    cudaGetLastError();
    return PTI_ERR_CUDA;
  }
  const int64_t fixed = static_cast<int64_t>(decode_fixed_smem<N>());
  const int stages = static_cast<int>(std::min<int64_t>(kMaxStages, (kSmemOptin - fixed) / S::kBytes));
  if (stages < 2) return PTI_ERR_SHAPE;
  const size_t smem = static_cast<size_t>(fixed) + static_cast<size_t>(stages) * S::kBytes;
  {
    static std::mutex mu;
    static bool attr_done[128] = {};
    std::lock_guard<std::mutex> lock(mu);
    if (!attr_done[dev]) {
      if (cudaFuncSetAttribute(decode_pass_kernel<N>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemOptin) !=
          cudaSuccess)
        return launch_status();
      attr_done[dev] = true;
    }
  }
  const DecodeLayout d = decode_layout(hidden, ffn, N);
  uint8_t *const ws = static_cast<uint8_t *>(workspace);
  const int64_t units_gu = (hidden / 256) * (ffn / 64), units_dn = (ffn / 256) * (hidden / kRowsPerTile);
  const int32_t grid = static_cast<int32_t>(std::min<int64_t>({static_cast<int64_t>(sms), units_gu, units_dn,
                                                               static_cast<int64_t>(kMaxGrid)}));
  const int n_launch = (n_layers + kMaxLayersPerLaunch - 1) / kMaxLayersPerLaunch;
  // the in-kernel tile tickets and the grid-barrier counters start at zero
  if (cudaMemsetAsync(ws + d.tickets, 0, d.h - d.tickets, stream) != cudaSuccess) return launch_status();
  static thread_local DecodeKernelParams P;  // about 25 KB: kept off the stack
  for (int c = 0; c < n_launch; ++c) {
    const int l0 = c * kMaxLayersPerLaunch;
    const int nl = std::min(kMaxLayersPerLaunch, n_layers - l0);
    std::memset(&P, 0, sizeof(P));
    for (int l = 0; l < nl; ++l) {
      if (!encode_weight_map<Fmt::Q8>(&P.maps[l][0], w_gate[l0 + l], ffn, hidden, 64) ||
          !encode_weight_map<Fmt::Q8>(&P.maps[l][1], w_up[l0 + l], ffn, hidden, 64) ||
          !encode_weight_map<Fmt::Q8>(&P.maps[l][2], w_down[l0 + l], hidden, ffn, kRowsPerTile))
        return PTI_ERR_CUDA;
    }
    P.x_in = (c == 0) ? x_in : reinterpret_cast<const float *>(ws + d.xraw);
    P.h = reinterpret_cast<float *>(ws + d.h);
    P.xraw = reinterpret_cast<float *>(ws + d.xraw);
    P.sq_h = reinterpret_cast<float *>(ws + d.sq_h);
    P.sq_x = reinterpret_cast<float *>(ws + d.sq_x);
    P.part = reinterpret_cast<float *>(ws + d.part);
    P.tickets = reinterpret_cast<unsigned int *>(ws + d.tickets);
    P.grid_bar = reinterpret_cast<unsigned int *>(ws + d.grid_bars) + c;
    P.hidden = hidden;
    P.ffn = ffn;
    P.n_layers = nl;
    P.grid = grid;
    P.stages = stages;
    P.input_scaled = c > 0 ? 1 : 0;
    P.eps = eps;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kWarpCount * 32 + 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, decode_pass_kernel<N>, P) != cudaSuccess) return launch_status();
  }
  return launch_finalize<N>(d, ws, hidden, eps, x_out, stream);
}

template <int N>
pti_status run_decode_pass(const void *const *w_gate, const void *const *w_up, const void *const *w_down,
                           int n_layers, int64_t hidden, int64_t ffn, double eps, const float *x_in, float *x_out,
                           void *workspace, cudaStream_t stream, bool chained) {
  if (chained) return run_decode_chained<N>(w_gate, w_up, w_down, n_layers, hidden, ffn, eps, x_in, x_out, workspace, stream);
  return run_decode_persistent<N>(w_gate, w_up, w_down, n_layers, hidden, ffn, eps, x_in, x_out, workspace, stream);
}

}  // namespace

pti_status decode_take_device_error(unsigned int *code_out) {
  unsigned int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v)) != cudaSuccess) return launch_status();
  if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero)) != cudaSuccess) return launch_status();
  *code_out = v;
  return PTI_OK;
}

}  // namespace pti

using namespace pti;

extern "C" size_t pti_mlp_decode_pass_workspace_bytes(int64_t hidden, int64_t ffn, int n_streams) {
  if (check_decode_shape(hidden, ffn) != PTI_OK || n_streams < 1 || n_streams > 4) return 0;
  return decode_layout(hidden, ffn, n_streams).total;
}

extern "C" pti_status pti_mlp_decode_pass_ex(const void *const *w_gate, const void *const *w_up,
                                             const void *const *w_down, int n_layers, int64_t hidden, int64_t ffn,
                                             int n_streams, double eps, const float *x_in, float *x_out,
                                             void *workspace, size_t workspace_bytes, pti_stream_t stream,
                                             uint32_t flags) {
  if ((flags & ~PTI_FLAG_DECODE_PERSISTENT) != 0u) return PTI_ERR_VALUE;
  const bool chained = (flags & PTI_FLAG_DECODE_PERSISTENT) == 0u;
  if (w_gate == nullptr || w_up == nullptr || w_down == nullptr || x_in == nullptr || x_out == nullptr)
    return PTI_ERR_NULL;
  if (n_layers < 1 || n_layers > kMaxLayersPerLaunch * kMaxLaunches) return PTI_ERR_SHAPE;
  if (const pti_status s = check_decode_shape(hidden, ffn); s != PTI_OK) return s;
  if (n_streams < 1 || n_streams > 4) return PTI_ERR_NSTREAMS;
  if (!std::isfinite(eps) || eps < 0.0) return PTI_ERR_VALUE;
  const uint64_t w_bytes = static_cast<uint64_t>(ffn) * (hidden / 32) * 34;  // each of the three matrices
  for (int l = 0; l < n_layers; ++l) {
    if (w_gate[l] == nullptr || w_up[l] == nullptr || w_down[l] == nullptr) return PTI_ERR_NULL;
    if (!aligned(w_gate[l], 16) || !aligned(w_up[l], 16) || !aligned(w_down[l], 16)) return PTI_ERR_ALIGN;
  }
  if (!aligned(x_in, 16) || !aligned(x_out, 4)) return PTI_ERR_ALIGN;
  const size_t need = decode_layout(hidden, ffn, n_streams).total;
  if (workspace == nullptr || workspace_bytes < need) return PTI_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return PTI_ERR_ALIGN;
  const uint64_t x_bytes = static_cast<uint64_t>(n_streams) * hidden * 4;
  if (overlaps(workspace, need, x_in, x_bytes) || overlaps(workspace, need, x_out, x_bytes)) return PTI_ERR_ALIAS;
  for (int l = 0; l < n_layers; ++l) {
    const void *ws[3] = {w_gate[l], w_up[l], w_down[l]};
    for (const void *w : ws)
      if (overlaps(x_out, x_bytes, w, w_bytes) || overlaps(workspace, need, w, w_bytes)) return PTI_ERR_ALIAS;
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  switch (n_streams) {
    case 1: return run_decode_pass<1>(w_gate, w_up, w_down, n_layers, hidden, ffn, eps, x_in, x_out, workspace, st, chained);
    case 2: return run_decode_pass<2>(w_gate, w_up, w_down, n_layers, hidden, ffn, eps, x_in, x_out, workspace, st, chained);
    case 3: return run_decode_pass<3>(w_gate, w_up, w_down, n_layers, hidden, ffn, eps, x_in, x_out, workspace, st, chained);
    default: return run_decode_pass<4>(w_gate, w_up, w_down, n_layers, hidden, ffn, eps, x_in, x_out, workspace, st, chained);
  }
}

extern "C" pti_status pti_mlp_decode_pass(const void *const *w_gate, const void *const *w_up,
                                          const void *const *w_down, int n_layers, int64_t hidden, int64_t ffn,
                                          int n_streams, double eps, const float *x_in, float *x_out,
                                          void *workspace, size_t workspace_bytes, pti_stream_t stream) {
  return pti_mlp_decode_pass_ex(w_gate, w_up, w_down, n_layers, hidden, ffn, n_streams, eps, x_in, x_out, workspace,
                                workspace_bytes, stream, 0u);
}
