// Test support: exhaustive check of the hardware FP4 / FP8 conversions the
// quantizers and the Direct-P mapping rely on (cvt.rn.satfinite.e2m1x2.f32,
// cvt.rn.satfinite.e4m3x2.f32).  For every fp32 bit pattern u in (lo, hi] the
// kernel compares the code of u with the code of u-1 and records each place
// where it changes, so a short list describes the conversion of every pattern.
#include "internal.h"

namespace fp4attn {
namespace {

__device__ __forceinline__ uint32_t convert_one(int format, uint32_t bits) {
  const float x = __uint_as_float(bits);
  if (format == 0) return cvt_e2m1x8(x, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f) & 0xFu;
  return cvt_e4m3(x);
}

__global__ void __launch_bounds__(256) cvt_transitions_kernel(int format, uint32_t lo, uint32_t hi,
                                                              uint32_t* __restrict__ pairs, int capacity,
                                                              int* __restrict__ count) {
  const uint64_t stride = static_cast<uint64_t>(gridDim.x) * blockDim.x;
  for (uint64_t u = static_cast<uint64_t>(lo) + 1 + static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
       u <= hi; u += stride) {
    const uint32_t c1 = convert_one(format, static_cast<uint32_t>(u));
    const uint32_t c0 = convert_one(format, static_cast<uint32_t>(u - 1));
    if (c1 != c0) {
      const int i = atomicAdd(count, 1);
      if (i < capacity) {
        pairs[2 * i] = static_cast<uint32_t>(u);
        pairs[2 * i + 1] = c1;
      }
    }
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    const int i = atomicAdd(count, 1);
    if (i < capacity) {
      pairs[2 * i] = lo;
      pairs[2 * i + 1] = convert_one(format, lo);
    }
  }
}

// The failure path of the bounded waits, exercised without a fault: one warp
// waits on an mbarrier that nothing ever arrives at, through the same
// mbar_wait the forward kernel uses but with a short limit, so the wait gives
// up, records site 90 in the status word, and the kernel returns.
__global__ void __launch_bounds__(32) wait_timeout_kernel(uint64_t limit_ns, DeviceStatus* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncwarp();
  mbar_wait(&bar, 0, &abort_flag, status, 90, limit_ns);
}

}  // namespace
}  // namespace fp4attn

using namespace fp4attn;

extern "C" int fp4attn_debug_wait_timeout(int limit_us, void* stream) {
  if (limit_us <= 0 || limit_us > 1000000) return FP4ATTN_ERR_INVALID_ARG;
  DeviceStatus* status = device_status_ptr();
  if (!status) return FP4ATTN_ERR_CUDA;
  wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(static_cast<uint64_t>(limit_us) * 1000u,
                                                                      status);
  return cuda_status(cudaGetLastError());
}

extern "C" int fp4attn_debug_cvt_transitions(int format, uint32_t lo, uint32_t hi, uint32_t* pairs, int capacity,
                                             int* count, void* stream) {
  if ((format != 0 && format != 1) || hi < lo || !pairs || !count || capacity <= 0) return FP4ATTN_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(count, 0, sizeof(int), s) != cudaSuccess) return FP4ATTN_ERR_CUDA;
  cvt_transitions_kernel<<<sm_count() * 8, 256, 0, s>>>(format, lo, hi, pairs, capacity, count);
  return cuda_status(cudaGetLastError());
}
