// Allocation-free variant of the grad-norm pass (lamb_grad_norm_noalloc).
//
// Some callers cannot allocate device memory when they need this pass: a
// framework whose caching allocator has already reserved nearly all of HBM
// (a raw cudaMalloc behind its back fails or fragments the pool), or an
// out-of-memory recovery path that must check the grads for inf/NaN exactly
// when no memory is left.  This entry point takes the caller's grads and a
// caller-provided output, and keeps everything else it needs -- the tensor
// table, the per-CTA partial sums and the completion ticket -- in one
// file-scope device array of fixed size, so it never calls cudaMalloc,
// cudaFree or any other allocating routine.  The array lives in every GPU
// that loads this library until the process exits.
//
// The computation is the same as the first kernel of lamb_step: the norm of
// g / S over all tensors (fp32 partial sums of at most 128 squares, fp64
// above that, partials summed in a fixed order by the CTA that finishes
// last), the inf/NaN check on the exponent bits, and the clip factor.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>
#include <string>

#include "lamb_internal.h"

namespace {

constexpr int kNaThreads = 256;
constexpr int kNaWarps = kNaThreads / 32;
constexpr int kNaMaxCtas = 1024;
constexpr int kNaMaxDevices = 64;

struct NaTensor {
  const uint16_t* g;
  int64_t n;
};

struct NaHeader {
  uint32_t ticket;     // CTAs finished in the current call
  uint32_t nonfinite;  // OR of every CTA's inf/NaN flag
};

constexpr size_t kHeaderBytes = 256;
constexpr size_t kPartialBytes = size_t(kNaMaxCtas) * sizeof(double);
constexpr size_t kTableBytes = size_t(LAMB_NOALLOC_MAX_TENSORS) * sizeof(NaTensor);
constexpr size_t kScratchBytes = kHeaderBytes + kPartialBytes + kTableBytes;
static_assert(kScratchBytes == LAMB_NOALLOC_SCRATCH_BYTES, "scratch size in lamb.h is stale");

}  // namespace

// The whole scratch area: header | per-CTA partials | tensor table.  In host
// code this name is only a handle for cudaGetSymbolAddress, never an address.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

namespace {

template <int DT>
__device__ __forceinline__ float2 na_decode2(uint32_t x) {
  if (DT == LAMB_GRAD_BF16)
    return make_float2(__uint_as_float(x << 16), __uint_as_float(x & 0xFFFF0000u));
  return make_float2(__half2float(__ushort_as_half(static_cast<unsigned short>(x & 0xFFFFu))),
                     __half2float(__ushort_as_half(static_cast<unsigned short>(x >> 16))));
}

template <int DT>
__device__ __forceinline__ uint32_t na_nonfinite2(uint32_t x) {
  constexpr uint32_t kExp = DT == LAMB_GRAD_BF16 ? 0x7F807F80u : 0x7C007C00u;
  const uint32_t u = ~x & kExp;
  return uint32_t((u & 0xFFFFu) == 0u) | uint32_t((u >> 16) == 0u);
}

__device__ __forceinline__ double na_warp_sum(double x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

__device__ __forceinline__ double na_block_sum(double x, double* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  x = na_warp_sum(x);
  if (lane == 0) red[warp] = x;
  __syncthreads();
  double y = lane < kNaWarps ? red[lane] : 0.0;
  y = na_warp_sum(y);
  __syncthreads();
  return y;
}

// Every CTA walks every tensor with a grid-wide stride; out receives
// {||g/S||, clip factor, inf/NaN flag} (+inf, 0, 1 when a grad is not finite).
template <int DT>
__global__ void __launch_bounds__(kNaThreads) grad_norm_noalloc_kernel(unsigned char* scratch,
                                                                       int32_t n_tensors,
                                                                       float clip,
                                                                       double loss_scale,
                                                                       double* out) {
  __shared__ double red[kNaWarps];
  __shared__ int is_last;
  NaHeader* hd = reinterpret_cast<NaHeader*>(scratch);
  double* partial = reinterpret_cast<double*>(scratch + kHeaderBytes);
  const NaTensor* tab = reinterpret_cast<const NaTensor*>(scratch + kHeaderBytes + kPartialBytes);
  const int64_t gtid = int64_t(blockIdx.x) * kNaThreads + threadIdx.x;
  const int64_t stride = int64_t(gridDim.x) * kNaThreads;
  double dacc = 0.0;
  uint32_t bad = 0;
  for (int32_t i = 0; i < n_tensors; ++i) {
    const NaTensor t = tab[i];
    const int64_t nv = t.n >> 3;
    for (int64_t k0 = gtid; k0 < nv; k0 += 16 * stride) {
      float acc = 0.0f;  // at most 16 vectors = 128 squares in fp32
#pragma unroll 4
      for (int j = 0; j < 16; ++j) {
        const int64_t k = k0 + int64_t(j) * stride;
        if (k < nv) {
          const uint4 q = __ldcs(reinterpret_cast<const uint4*>(t.g + 8 * k));
          const uint32_t wv[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            const float2 f = na_decode2<DT>(wv[h]);
            acc = __fmaf_rn(f.x, f.x, acc);
            acc = __fmaf_rn(f.y, f.y, acc);
            bad |= na_nonfinite2<DT>(wv[h]);
          }
        }
      }
      dacc += double(acc);
    }
    const int64_t tail = t.n - (nv << 3);
    if (gtid < tail) {
      const uint16_t x = t.g[(nv << 3) + gtid];
      const float f = na_decode2<DT>(uint32_t(x) | (uint32_t(x) << 16)).x;
      dacc += double(f) * double(f);
      bad |= na_nonfinite2<DT>(uint32_t(x) | (uint32_t(x) << 16));
    }
  }
  const double s_blk = na_block_sum(dacc, red);
  bad = __syncthreads_or(bad);
  if (threadIdx.x == 0) {
    partial[blockIdx.x] = s_blk;
    if (bad) atomicOr(&hd->nonfinite, 1u);
    __threadfence();
    const uint32_t prev = atomicAdd(&hd->ticket, 1u);
    is_last = prev == gridDim.x - 1;
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  double s = 0.0;
  for (int i = threadIdx.x; i < int(gridDim.x); i += kNaThreads) s += __ldcg(&partial[i]);
  s = na_block_sum(s, red);
  if (threadIdx.x == 0) {
    const uint32_t nf = atomicExch(&hd->nonfinite, 0u);
    if (nf) {
      out[0] = __longlong_as_double(0x7FF0000000000000ll);
      out[1] = 0.0;
      out[2] = 1.0;
    } else {
      const double gn = sqrt(s) / loss_scale;
      out[0] = gn;
      out[1] = (clip > 0.0f && gn > double(clip)) ? double(clip) / gn : 1.0;
      out[2] = 0.0;
    }
    hd->ticket = 0u;
  }
}

// Writes entries [at, at + count) of the tensor table into the scratch array
// from the kernel's own arguments (kNaTablePerLaunch entries, 3840 bytes, under
// the 4 KB parameter limit), and the first launch of a call clears the ticket
// and the inf/NaN flag.  Each launch carries its entries by value, so a call
// never reads host memory after it returns.
constexpr int kNaTablePerLaunch = 240;

struct NaTableChunk {
  NaTensor e[kNaTablePerLaunch];
};

__global__ void noalloc_table_kernel(unsigned char* scratch, int32_t at, int32_t count,
                                     int32_t clear_header, NaTableChunk chunk) {
  NaTensor* tab = reinterpret_cast<NaTensor*>(scratch + kHeaderBytes + kPartialBytes);
  const int i = threadIdx.x;
  if (i < count) tab[at + i] = chunk.e[i];
  if (clear_header && i == 0) {
    NaHeader* hd = reinterpret_cast<NaHeader*>(scratch);
    hd->ticket = 0u;
    hd->nonfinite = 0u;
  }
}

int na_fail(int code, const std::string& msg) {
  lambgb::set_last_error(msg);
  return code;
}

// Per-device set-up: the device address of the scratch array and the grid.
std::mutex na_mutex;
void* na_scratch_addr[kNaMaxDevices] = {};
int na_grid[kNaMaxDevices] = {};

}  // namespace

extern "C" {

LAMB_API int lamb_grad_norm_noalloc(int32_t n_tensors, const int64_t* sizes,
                                    const void* const* grads, int32_t grad_dtype,
                                    float loss_scale, float clip, double* out, void* stream) {
  lambgb::set_last_error("");
  if (n_tensors < 0) return na_fail(LAMB_ERR_INVALID, "n_tensors must be >= 0");
  if (n_tensors > LAMB_NOALLOC_MAX_TENSORS)
    return na_fail(LAMB_ERR_INVALID,
                   "n_tensors = " + std::to_string(n_tensors) +
                       " exceeds LAMB_NOALLOC_MAX_TENSORS (" +
                       std::to_string(LAMB_NOALLOC_MAX_TENSORS) + ")");
  if (n_tensors > 0 && (!sizes || !grads))
    return na_fail(LAMB_ERR_INVALID, "sizes and grads must be non-NULL");
  if (!out) return na_fail(LAMB_ERR_INVALID, "out is NULL");
  if ((reinterpret_cast<uintptr_t>(out) & 7u) != 0)
    return na_fail(LAMB_ERR_ALIGN, "out is not 8-byte aligned");
  if (grad_dtype != LAMB_GRAD_BF16 && grad_dtype != LAMB_GRAD_FP16)
    return na_fail(LAMB_ERR_INVALID, "grad_dtype must be LAMB_GRAD_BF16 or LAMB_GRAD_FP16");
  if (!(loss_scale > 0.0f) || !std::isfinite(loss_scale))
    return na_fail(LAMB_ERR_INVALID, "loss_scale must be finite and > 0");
  if (std::isnan(clip)) return na_fail(LAMB_ERR_INVALID, "clip is NaN");
  for (int32_t i = 0; i < n_tensors; ++i) {
    if (sizes[i] < 0) return na_fail(LAMB_ERR_INVALID, "sizes[" + std::to_string(i) + "] < 0");
    if (sizes[i] == 0) continue;
    if (!grads[i]) return na_fail(LAMB_ERR_INVALID, "grads[" + std::to_string(i) + "] is NULL");
    if ((reinterpret_cast<uintptr_t>(grads[i]) & 15u) != 0)
      return na_fail(LAMB_ERR_ALIGN, "grads[" + std::to_string(i) + "] is not 16-byte aligned");
  }

  int dev = 0;
  cudaError_t ce = cudaGetDevice(&dev);
  if (ce != cudaSuccess) return na_fail(LAMB_ERR_CUDA, "cudaGetDevice failed");
  if (dev < 0 || dev >= kNaMaxDevices) return na_fail(LAMB_ERR_INVALID, "device index too large");
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  std::lock_guard<std::mutex> lock(na_mutex);
  if (!na_scratch_addr[dev]) {
    // First call on this device, which is current: find where the array
    // lives in this device's memory, and size the grid.
    void* p = nullptr;
    ce = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (ce != cudaSuccess || !p)
      return na_fail(LAMB_ERR_CUDA, std::string("cudaGetSymbolAddress: ") +
                                        cudaGetErrorString(ce));
    int sms = 0, per_sm = 0;
    ce = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (ce == cudaSuccess)
      ce = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
          &per_sm, grad_norm_noalloc_kernel<LAMB_GRAD_BF16>, kNaThreads, 0);
    if (ce != cudaSuccess || sms <= 0 || per_sm <= 0)
      return na_fail(LAMB_ERR_CUDA, "occupancy query failed");
    // Load the other kernels now too (lazy module loading would otherwise
    // load each one, and take device memory for its code, at its first use).
    cudaFuncAttributes fa;
    ce = cudaFuncGetAttributes(&fa, grad_norm_noalloc_kernel<LAMB_GRAD_FP16>);
    if (ce == cudaSuccess) ce = cudaFuncGetAttributes(&fa, noalloc_table_kernel);
    if (ce != cudaSuccess)
      return na_fail(LAMB_ERR_CUDA, std::string("loading the kernels: ") +
                                        cudaGetErrorString(ce));
    na_grid[dev] = sms * per_sm < kNaMaxCtas ? sms * per_sm : kNaMaxCtas;
    na_scratch_addr[dev] = p;
  }
  unsigned char* scratch = static_cast<unsigned char*>(na_scratch_addr[dev]);

  // Write the tensor table (empty tensors left out) and clear the ticket and
  // the inf/NaN flag, stream-ordered after any earlier call on this stream.
  int32_t used = 0;
  NaTableChunk chunk;
  int count = 0;
  bool first = true;
  auto flush = [&]() {
    noalloc_table_kernel<<<1, kNaTablePerLaunch, 0, s>>>(scratch, used - count, count,
                                                         first ? 1 : 0, chunk);
    first = false;
    count = 0;
    return cudaGetLastError();
  };
  ce = cudaSuccess;
  for (int32_t i = 0; i < n_tensors && ce == cudaSuccess; ++i) {
    if (sizes[i] == 0) continue;
    chunk.e[count].g = static_cast<const uint16_t*>(grads[i]);
    chunk.e[count].n = sizes[i];
    ++count;
    ++used;
    if (count == kNaTablePerLaunch) ce = flush();
  }
  if (ce == cudaSuccess && (count > 0 || first)) ce = flush();
  if (ce != cudaSuccess)
    return na_fail(LAMB_ERR_CUDA, std::string("writing the tensor table: ") +
                                      cudaGetErrorString(ce));
  if (grad_dtype == LAMB_GRAD_FP16)
    grad_norm_noalloc_kernel<LAMB_GRAD_FP16><<<na_grid[dev], kNaThreads, 0, s>>>(
        scratch, used, clip, double(loss_scale), out);
  else
    grad_norm_noalloc_kernel<LAMB_GRAD_BF16><<<na_grid[dev], kNaThreads, 0, s>>>(
        scratch, used, clip, double(loss_scale), out);
  ce = cudaGetLastError();
  if (ce != cudaSuccess)
    return na_fail(LAMB_ERR_CUDA, std::string("kernel launch: ") + cudaGetErrorString(ce));
  return LAMB_OK;
}

}  // extern "C"
