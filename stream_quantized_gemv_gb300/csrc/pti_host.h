// pti_host.h -- host-side helpers shared by the library's translation units:
// argument checks, device properties and launch-error mapping.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "pti.h"

namespace pti {

inline bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Do the byte ranges [a, a+na) and [b, b+nb) overlap?
inline bool overlaps(const void *a, uint64_t na, const void *b, uint64_t nb) {
  if (a == nullptr || b == nullptr || na == 0 || nb == 0) return false;
  const uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
  return pa < pb + nb && pb < pa + na;
}

struct DeviceInfo {
  int sms = 0;
  bool ok = false;
};

// Number of SMs of the current device (cached per device); 0 on error.
inline int current_device_sms(int *device_out = nullptr) {
  static std::mutex mu;
  static DeviceInfo cache[128];
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) {
    cudaGetLastError();
    return 0;
  }
  if (device_out) *device_out = dev;
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev].ok) {
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return 0;
    }
    cache[dev].sms = sms;
    cache[dev].ok = true;
  }
  return cache[dev].sms;
}

inline pti_status launch_status() {
  return cudaGetLastError() == cudaSuccess ? PTI_OK : PTI_ERR_CUDA;
}

// Each translation unit with kernels keeps its own device error word; these
// read and clear the decode pass's (pti_decode.cu).
pti_status decode_take_device_error(unsigned int *code_out);

}  // namespace pti
