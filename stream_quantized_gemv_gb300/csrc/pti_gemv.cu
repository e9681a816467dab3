// pti_gemv.cu -- C ABI of the N-stream Q8 GEMV, the SSQ twin GEMV, the
// allocation-free Q8 GEMV and the device error word.  The kernels live in
// pti_gemv_kernel.cuh.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "pti.h"
#include "pti_gemv_kernel.cuh"
#include "pti_host.h"

namespace pti {
namespace {

// ---------------------------------------------------------------------------
// Plain per-row kernel for shapes outside the fast path: one warp per row,
// lanes stride over the blocks, each block's products summed into a fresh
// partial that is scaled once.  The block layout is a parameter: a block of
// kBlock bytes holds its binary16 scale at byte kScale and the int8 of column
// i at byte kQ + kStride * i.  Q8 is (34, 0, 2, 1); a twin block is read as
// model A (68, 0, 5, 2), whose bytes are the upper halves of the payload's
// little-endian 16-bit elements, and as model B (68, 2, 4, 2), the lower
// halves.
// ---------------------------------------------------------------------------
template <int N, int kBlock, int kScale, int kQ, int kStride>
__global__ void __launch_bounds__(256) rowwise_kernel(const uint8_t *__restrict__ w, int64_t rows, int64_t cols,
                                                      const float *__restrict__ x, float *__restrict__ y) {
  const int lane = threadIdx.x & 31;
  const int64_t nb = cols / 32;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t row = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; row < rows; row += warps) {
    float acc[N];
#pragma unroll
    for (int s = 0; s < N; ++s) acc[s] = 0.0f;
    for (int64_t b = lane; b < nb; b += 32) {
      const uint8_t *blk = w + (row * nb + b) * kBlock;
      const float d = half_bits_to_float(*reinterpret_cast<const uint16_t *>(blk + kScale));
      const float *xb = x + 32 * b;
      float part[N];
#pragma unroll
      for (int s = 0; s < N; ++s) part[s] = 0.0f;
      for (int i = 0; i < 32; ++i) {
        const float q = static_cast<float>(static_cast<int8_t>(blk[kQ + kStride * i]));
#pragma unroll
        for (int s = 0; s < N; ++s) part[s] = fmaf(q, xb[s * cols + i], part[s]);
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

template <int N, int kBlock, int kScale, int kQ, int kStride>
pti_status launch_rowwise(const void *w, int64_t rows, int64_t cols, const float *x, float *y,
                          cudaStream_t stream) {
  const int sms = current_device_sms();
  if (sms <= 0) return PTI_ERR_CUDA;
  const int64_t blocks = std::min<int64_t>((rows + 7) / 8, static_cast<int64_t>(sms) * 16);
  rowwise_kernel<N, kBlock, kScale, kQ, kStride><<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
      static_cast<const uint8_t *>(w), rows, cols, x, y);
  return launch_status();
}

template <int N>
pti_status launch_q8_rowwise(const void *w, int64_t rows, int64_t cols, const float *x, float *y,
                             cudaStream_t stream) {
  return launch_rowwise<N, 34, 0, 2, 1>(w, rows, cols, x, y, stream);
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
    case PTI_ERR_VALUE: return "PTI_ERR_VALUE: a scalar argument is outside its range";
  }
  return "PTI_ERR_UNKNOWN";
}

extern "C" size_t pti_q8_gemv_workspace_bytes(int64_t rows, int64_t cols, int n_streams) {
  if (check_gemv_shape(rows, cols) != PTI_OK || n_streams < 1 || n_streams > 4) return 0;
  if (cols % 256 != 0) return 0;
  return fast_workspace_bytes(n_streams);
}

extern "C" size_t pti_ssq_twin_gemv_workspace_bytes(int64_t rows, int64_t cols) {
  if (check_gemv_shape(rows, cols) != PTI_OK) return 0;
  if (cols % 128 != 0) return 0;
  return fast_workspace_bytes(2);
}

extern "C" size_t pti_ssq_twin_gemv_nstream_workspace_bytes(int64_t rows, int64_t cols, int n_streams) {
  if (check_gemv_shape(rows, cols) != PTI_OK || n_streams < 1 || n_streams > 2) return 0;
  if (cols % 128 != 0) return 0;
  return fast_workspace_bytes(2 * n_streams);
}

namespace {
// The consumer a Q8 call's flags ask for (false: an invalid combination).
bool cores_of_flags(uint32_t flags, Cores *cores) {
  const uint32_t c = flags & (PTI_FLAG_CUDA_CORES | PTI_FLAG_TENSOR_CORES);
  if (c == (PTI_FLAG_CUDA_CORES | PTI_FLAG_TENSOR_CORES)) return false;
  *cores = c == PTI_FLAG_CUDA_CORES ? Cores::Cuda : c == PTI_FLAG_TENSOR_CORES ? Cores::Tensor : Cores::Auto;
  return true;
}

pti_status q8_gemv(const void *w_q8, int64_t rows, int64_t cols, int n_streams, const float *x, float *y,
                   void *workspace, size_t workspace_bytes, pti_stream_t stream, uint32_t flags) {
  if ((flags & ~(PTI_FLAG_PDL | PTI_FLAG_CUDA_CORES | PTI_FLAG_TENSOR_CORES)) != 0u) return PTI_ERR_VALUE;
  Cores cores = Cores::Auto;
  if (!cores_of_flags(flags, &cores)) return PTI_ERR_VALUE;
  const bool pdl = (flags & PTI_FLAG_PDL) != 0u;
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
      case 1: return launch_fast<Fmt::Q8, 1>(w_q8, rows, cols, x, nullptr, y, nullptr, workspace, st, pdl, cores);
      case 2: return launch_fast<Fmt::Q8, 2>(w_q8, rows, cols, x, nullptr, y, nullptr, workspace, st, pdl, cores);
      case 3: return launch_fast<Fmt::Q8, 3>(w_q8, rows, cols, x, nullptr, y, nullptr, workspace, st, pdl, cores);
      default: return launch_fast<Fmt::Q8, 4>(w_q8, rows, cols, x, nullptr, y, nullptr, workspace, st, pdl, cores);
    }
  }
  switch (n_streams) {
    case 1: return launch_q8_rowwise<1>(w_q8, rows, cols, x, y, st);
    case 2: return launch_q8_rowwise<2>(w_q8, rows, cols, x, y, st);
    case 3: return launch_q8_rowwise<3>(w_q8, rows, cols, x, y, st);
    default: return launch_q8_rowwise<4>(w_q8, rows, cols, x, y, st);
  }
}

// Twin GEMV with n activation streams per model (x_a, x_b [n][cols];
// y_a, y_b [n][rows]).
pti_status twin_gemv(const void *w_twin, int64_t rows, int64_t cols, int n, const float *x_a, const float *x_b,
                     float *y_a, float *y_b, void *workspace, size_t workspace_bytes, pti_stream_t stream,
                     uint32_t flags) {
  if ((flags & ~PTI_FLAG_PDL) != 0u) return PTI_ERR_VALUE;
  const bool pdl = (flags & PTI_FLAG_PDL) != 0u;
  if (w_twin == nullptr || x_a == nullptr || x_b == nullptr || y_a == nullptr || y_b == nullptr)
    return PTI_ERR_NULL;
  if (const pti_status s = check_gemv_shape(rows, cols); s != PTI_OK) return s;
  if (n < 1 || n > 2) return PTI_ERR_NSTREAMS;
  if (!aligned(w_twin, 16) || !aligned(x_a, 4) || !aligned(x_b, 4) || !aligned(y_a, 4) || !aligned(y_b, 4))
    return PTI_ERR_ALIGN;
  const uint64_t w_bytes = static_cast<uint64_t>(rows) * (cols / 32) * 68;
  const uint64_t x_bytes = static_cast<uint64_t>(n) * cols * 4;
  const uint64_t y_bytes = static_cast<uint64_t>(n) * rows * 4;
  if (overlaps(y_a, y_bytes, y_b, y_bytes) || overlaps(y_a, y_bytes, w_twin, w_bytes) ||
      overlaps(y_b, y_bytes, w_twin, w_bytes) || overlaps(y_a, y_bytes, x_a, x_bytes) ||
      overlaps(y_a, y_bytes, x_b, x_bytes) || overlaps(y_b, y_bytes, x_a, x_bytes) ||
      overlaps(y_b, y_bytes, x_b, x_bytes))
    return PTI_ERR_ALIAS;
  const size_t need = (check_gemv_shape(rows, cols) == PTI_OK && cols % 128 == 0) ? fast_workspace_bytes(2 * n) : 0;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (need > 0) {
    if (workspace == nullptr || workspace_bytes < need) return PTI_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return PTI_ERR_ALIGN;
    if (overlaps(workspace, need, w_twin, w_bytes) || overlaps(workspace, need, x_a, x_bytes) ||
        overlaps(workspace, need, x_b, x_bytes) || overlaps(workspace, need, y_a, y_bytes) ||
        overlaps(workspace, need, y_b, y_bytes))
      return PTI_ERR_ALIAS;
    if (aligned(x_a, 16) && aligned(x_b, 16) && (n == 1 || (cols * 4) % 16 == 0)) {
      if (n == 1) return launch_fast<Fmt::Twin, 1>(w_twin, rows, cols, x_a, x_b, y_a, y_b, workspace, st, pdl);
      return launch_fast<Fmt::Twin, 2>(w_twin, rows, cols, x_a, x_b, y_a, y_b, workspace, st, pdl);
    }
  }
  // the plain kernel, once per model (model A: upper bytes, model B: lower)
  const pti_status e = n == 1 ? launch_rowwise<1, 68, 0, 5, 2>(w_twin, rows, cols, x_a, y_a, st)
                              : launch_rowwise<2, 68, 0, 5, 2>(w_twin, rows, cols, x_a, y_a, st);
  if (e != PTI_OK) return e;
  return n == 1 ? launch_rowwise<1, 68, 2, 4, 2>(w_twin, rows, cols, x_b, y_b, st)
                : launch_rowwise<2, 68, 2, 4, 2>(w_twin, rows, cols, x_b, y_b, st);
}

}  // namespace

extern "C" pti_status pti_q8_gemv_nstream(const void *w_q8, int64_t rows, int64_t cols, int n_streams,
                                          const float *x, float *y, void *workspace, size_t workspace_bytes,
                                          pti_stream_t stream) {
  return q8_gemv(w_q8, rows, cols, n_streams, x, y, workspace, workspace_bytes, stream, 0u);
}

extern "C" pti_status pti_q8_gemv_nstream_ex(const void *w_q8, int64_t rows, int64_t cols, int n_streams,
                                             const float *x, float *y, void *workspace, size_t workspace_bytes,
                                             pti_stream_t stream, uint32_t flags) {
  return q8_gemv(w_q8, rows, cols, n_streams, x, y, workspace, workspace_bytes, stream, flags);
}

extern "C" pti_status pti_ssq_twin_gemv(const void *w_twin, int64_t rows, int64_t cols, const float *x_a,
                                        const float *x_b, float *y_a, float *y_b, void *workspace,
                                        size_t workspace_bytes, pti_stream_t stream) {
  return twin_gemv(w_twin, rows, cols, 1, x_a, x_b, y_a, y_b, workspace, workspace_bytes, stream, 0u);
}

extern "C" pti_status pti_ssq_twin_gemv_ex(const void *w_twin, int64_t rows, int64_t cols, const float *x_a,
                                           const float *x_b, float *y_a, float *y_b, void *workspace,
                                           size_t workspace_bytes, pti_stream_t stream, uint32_t flags) {
  return twin_gemv(w_twin, rows, cols, 1, x_a, x_b, y_a, y_b, workspace, workspace_bytes, stream, flags);
}

extern "C" pti_status pti_ssq_twin_gemv_nstream(const void *w_twin, int64_t rows, int64_t cols, int n_streams,
                                                const float *x_a, const float *x_b, float *y_a, float *y_b,
                                                void *workspace, size_t workspace_bytes, pti_stream_t stream,
                                                uint32_t flags) {
  return twin_gemv(w_twin, rows, cols, n_streams, x_a, x_b, y_a, y_b, workspace, workspace_bytes, stream, flags);
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
// Device address of g_pti_noalloc_scratch on the current device (looked up
// once per device; the array's name is only a host-side stand-in).
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
  if (need > kNoAllocScratchBytes) return PTI_ERR_WORKSPACE;  // cannot happen for a valid shape today
  void *scratch = nullptr;
  if (need > 0) {
    if (const pti_status st = noalloc_scratch_address(&scratch); st != PTI_OK) return st;
  }
  return pti_q8_gemv_nstream(w_q8, rows, cols, n_streams, x, y, scratch, need > 0 ? kNoAllocScratchBytes : 0,
                             stream);
}

// Testing hook: the fast-path Q8 GEMV with a stalled copy (see pti.h).
extern "C" pti_status pti_test_q8_gemv_stall(const void *w_q8, int64_t rows, int64_t cols, int n_streams,
                                             const float *x, float *y, void *workspace, size_t workspace_bytes,
                                             pti_stream_t stream, int64_t stall_unit, uint64_t wait_ns,
                                             uint32_t flags) {
  Cores cores = Cores::Auto;
  if ((flags & ~(PTI_FLAG_CUDA_CORES | PTI_FLAG_TENSOR_CORES)) != 0u || !cores_of_flags(flags, &cores))
    return PTI_ERR_VALUE;
  if (w_q8 == nullptr || x == nullptr || y == nullptr || workspace == nullptr) return PTI_ERR_NULL;
  if (const pti_status st = check_gemv_shape(rows, cols); st != PTI_OK) return st;
  if (cols % 256 != 0) return PTI_ERR_SHAPE;
  if (n_streams < 1 || n_streams > 4) return PTI_ERR_NSTREAMS;
  if (!aligned(w_q8, 16) || !aligned(x, 16) || !aligned(y, 4) || !aligned(workspace, 256)) return PTI_ERR_ALIGN;
  if (workspace_bytes < fast_workspace_bytes(n_streams)) return PTI_ERR_WORKSPACE;
  if (wait_ns < 1000 || wait_ns > kWaitTimeoutNs) return PTI_ERR_VALUE;
  const int sms = current_device_sms();
  if (sms <= 0) return PTI_ERR_CUDA;
  const TilePlan p = plan_tiles<Fmt::Q8, 1, Epi::Plain>(rows, cols, sms);
  const int64_t cta0_units = p.units / p.grid;
  if (stall_unit < kMaxStages || stall_unit >= cta0_units) return PTI_ERR_VALUE;
  // (the grid and the unit split do not depend on the stream count)
  const uint64_t w_bytes = static_cast<uint64_t>(rows) * (cols / 32) * 34;
  const uint64_t y_bytes = static_cast<uint64_t>(n_streams) * rows * 4;
  const uint64_t x_bytes = static_cast<uint64_t>(n_streams) * cols * 4;
  const size_t need = fast_workspace_bytes(n_streams);
  if (overlaps(y, y_bytes, w_q8, w_bytes) || overlaps(y, y_bytes, x, x_bytes) || overlaps(workspace, need, y, y_bytes) ||
      overlaps(workspace, need, w_q8, w_bytes) || overlaps(workspace, need, x, x_bytes))
    return PTI_ERR_ALIAS;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  switch (n_streams) {
    case 1: return launch_fast<Fmt::Q8, 1>(w_q8, rows, cols, x, nullptr, y, nullptr, workspace, s, false, cores, wait_ns,
                                           stall_unit);
    case 2: return launch_fast<Fmt::Q8, 2>(w_q8, rows, cols, x, nullptr, y, nullptr, workspace, s, false, cores, wait_ns,
                                           stall_unit);
    case 3: return launch_fast<Fmt::Q8, 3>(w_q8, rows, cols, x, nullptr, y, nullptr, workspace, s, false, cores, wait_ns,
                                           stall_unit);
    default: return launch_fast<Fmt::Q8, 4>(w_q8, rows, cols, x, nullptr, y, nullptr, workspace, s, false, cores, wait_ns,
                                             stall_unit);
  }
}

extern "C" pti_status pti_device_error(uint32_t *code_out) {
  if (code_out == nullptr) return PTI_ERR_NULL;
  if (cudaDeviceSynchronize() != cudaSuccess) return launch_status();
  unsigned int v = 0, zero = 0, v_decode = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(v)) != cudaSuccess) return launch_status();
  if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(zero)) != cudaSuccess) return launch_status();
  if (const pti_status s = decode_take_device_error(&v_decode); s != PTI_OK) return s;
  *code_out = v | v_decode;
  return PTI_OK;
}
