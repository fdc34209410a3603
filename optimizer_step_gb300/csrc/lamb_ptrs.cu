// Writes a step's grad-pointer array into device memory with a kernel whose
// arguments carry the pointers.  An ordinary host-to-device copy would go
// through a copy engine, where it can queue behind an unrelated bulk copy (for
// example the next step's grads streaming in from host memory) and stall the
// step behind it.
#include <cuda_runtime.h>

#include <cstdint>

#include "lamb_internal.h"

namespace lambgb {
namespace {

constexpr int kPtrsPerLaunch = 480;  // 3840 bytes of arguments per launch

struct PtrChunk {
  const void* p[kPtrsPerLaunch];
};

__global__ void write_ptrs_kernel(const void** dst, int count, PtrChunk chunk) {
  const int i = threadIdx.x;
  if (i < count) dst[i] = chunk.p[i];
}

}  // namespace

int write_grad_ptrs(const void** dst, const void* const* src, int32_t n, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  for (int32_t at = 0; at < n; at += kPtrsPerLaunch) {
    const int count = n - at < kPtrsPerLaunch ? int(n - at) : kPtrsPerLaunch;
    PtrChunk c;
    for (int i = 0; i < count; ++i) c.p[i] = src[at + i];
    write_ptrs_kernel<<<1, kPtrsPerLaunch, 0, s>>>(dst + at, count, c);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return int(e);
  }
  return 0;
}

}  // namespace lambgb
