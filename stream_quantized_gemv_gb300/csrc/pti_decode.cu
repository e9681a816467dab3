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
constexpr int kMaxLayers = 4096;  // layers per call

// Workspace of one pass, byte offsets (each 256-byte aligned).
struct DecodeLayout {
  int64_t n_rb_gu = 0, n_rb_down = 0;  // tiles of the GateUp and Down kernels
  size_t part = 0, h = 0, xraw = 0, sq_h = 0, sq_x = 0, scales = 0, total = 0;
};

size_t round256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

DecodeLayout decode_layout(int64_t hidden, int64_t ffn, int n) {
  DecodeLayout d;
  d.n_rb_gu = (ffn + 63) / 64;
  d.n_rb_down = (hidden + kRowsPerTile - 1) / kRowsPerTile;
  size_t off = 0;
  d.part = off;
  off = round256(off + partial_bytes(n));
  d.h = off;
  off = round256(off + static_cast<size_t>(n) * ffn * sizeof(float));
  d.xraw = off;
  off = round256(off + static_cast<size_t>(n) * hidden * sizeof(float));
  d.sq_h = off;
  off = round256(off + static_cast<size_t>(d.n_rb_gu) * n * sizeof(float));
  d.sq_x = off;
  off = round256(off + static_cast<size_t>(d.n_rb_down) * n * sizeof(float));
  d.scales = off;  // input scales of the GateUp and of the Down step, [2][n]
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

// Final kernel of a pass: applies the last RMS scale.
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

extern "C" pti_status pti_mlp_decode_pass(const void *const *w_gate, const void *const *w_up,
                                          const void *const *w_down, int n_layers, int64_t hidden, int64_t ffn,
                                          int n_streams, double eps, const float *x_in, float *x_out,
                                          void *workspace, size_t workspace_bytes, pti_stream_t stream) {
  if (w_gate == nullptr || w_up == nullptr || w_down == nullptr || x_in == nullptr || x_out == nullptr)
    return PTI_ERR_NULL;
  if (n_layers < 1 || n_layers > kMaxLayers) return PTI_ERR_SHAPE;
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
    case 1: return run_decode_chained<1>(w_gate, w_up, w_down, n_layers, hidden, ffn, eps, x_in, x_out, workspace, st);
    case 2: return run_decode_chained<2>(w_gate, w_up, w_down, n_layers, hidden, ffn, eps, x_in, x_out, workspace, st);
    case 3: return run_decode_chained<3>(w_gate, w_up, w_down, n_layers, hidden, ffn, eps, x_in, x_out, workspace, st);
    default: return run_decode_chained<4>(w_gate, w_up, w_down, n_layers, hidden, ffn, eps, x_in, x_out, workspace, st);
  }
}
