// Test support: exhaustive check of the hardware FP4 / FP8 conversions the
// quantizers and the Direct-P mapping rely on (cvt.rn.satfinite.e2m1x2.f32,
// cvt.rn.satfinite.e4m3x2.f32).  For every fp32 bit pattern u in (lo, hi] the
// kernel compares the code of u with the code of u-1 and records each place
// where it changes, so a short list describes the conversion of every pattern.
#include "fp8.cuh"
#include "internal.h"

namespace fp4attn {
namespace {

__device__ __forceinline__ uint32_t convert_one(int format, uint32_t bits) {
  const float x = __uint_as_float(bits);
  if (format == 0) return cvt_e2m1x8(x, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f) & 0xFu;
  if (format == 2) return cvt_fp8x4<kFmtE5M2>(x, 0.f, 0.f, 0.f) & 0xFFu;
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

// Dense tensor-core throughput of the block-scaled products the forward
// issues, for the roofline: one CTA per SM, one elected thread issues `iters`
// rounds of M = 128, N = 128 products from shared-memory operands into one
// TMEM accumulator.  kind 0: kind::mxf4nvf4 (E2M1, 16-element UE4M3 scales,
// two K = 64 products per round, the QK^T form); kind 1: kind::mxf4 (E2M1,
// 32-element UE8M0 scales, two K = 64 products, the PV form); kind 2:
// kind::mxf8f6f4 (E4M3, one UE8M0 scale per 32 elements, four K = 32
// products, the FP8 PV form).  Every round is 2*128*128*128 FLOP.  Operands
// are E2M1 / E4M3 ones with unit scales.
constexpr int kPeakThreads = 128;
// 35 KB used; the request is padded so that one CTA holds each SM
constexpr int kPeakSmem = 120 * 1024;

__global__ void __launch_bounds__(kPeakThreads, 1) mma_peak_kernel(int kind, int iters, DeviceStatus* status) {
  extern __shared__ uint8_t raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  uint8_t* a = smem;              // 128 rows x 64 B (E2M1) or 128 B (E4M3)
  uint8_t* b = smem + 16384;      // the same
  uint8_t* sf = smem + 32768;     // A scale atoms (2), B scale atoms (2)
  uint64_t* bar = reinterpret_cast<uint64_t*>(smem + 32768 + 4 * 512);
  uint32_t* slot = reinterpret_cast<uint32_t*>(smem + 32768 + 4 * 512 + 8);
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5;
  const uint32_t one4 = (kind == 2) ? 0x38383838u : 0x22222222u;    // E4M3 1.0 / two E2M1 1.0
  const uint32_t unit4 = (kind == 0) ? 0x38383838u : 0x7F7F7F7Fu;   // UE4M3 1.0 / UE8M0 1.0
  for (int i = threadIdx.x; i < 32768 / 16; i += kPeakThreads)
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(one4, one4, one4, one4);
  for (int i = threadIdx.x; i < 4 * 512 / 16; i += kPeakThreads)
    reinterpret_cast<uint4*>(sf)[i] = make_uint4(unit4, unit4, unit4, unit4);
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  fence_proxy_async_smem();
  if (warp == 0) {
    tmem_alloc(slot, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *slot;
  if (warp == 0) {
    const uint32_t d = tmem, sfa = tmem + 128, sfb = tmem + 136;
    for (int i = 0; i < 2; ++i) {
      tc_cp_sf_atom_warp(sfa + 4 * i, smem_u32(sf + 512 * i));
      tc_cp_sf_atom_warp(sfb + 4 * i, smem_u32(sf + 1024 + 512 * i));
    }
    if (kind == 2) {
      const uint64_t ad = smem_desc(smem_u32(a), 16, 1024, 2), bd = smem_desc(smem_u32(b), 16, 1024, 2);
      for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_mxf8_warp(d, ad + 2 * k, bd + 2 * k, idesc_mxf8_block_scaled(128, 128, k, k), sfa, sfb, it > 0 || k > 0);
      }
    } else if (kind == 1) {
      const uint64_t ad = smem_desc(smem_u32(a), 16, 512, 4), bd = smem_desc(smem_u32(b), 16, 512, 4);
      constexpr uint32_t i0 = idesc_fp4_block_scaled(128, 128, 1, 0, 0), i1 = idesc_fp4_block_scaled(128, 128, 1, 2, 2);
      for (int it = 0; it < iters; ++it) {
        mma_mxf4_warp(d, ad, bd, i0, sfa, sfb, it > 0);
        mma_mxf4_warp(d, ad + 2, bd + 2, i1, sfa, sfb, true);
      }
    } else {
      const uint64_t ad = smem_desc(smem_u32(a), 16, 512, 4), bd = smem_desc(smem_u32(b), 16, 512, 4);
      constexpr uint32_t i0 = idesc_fp4_block_scaled(128, 128, 0, 0, 0);
      for (int it = 0; it < iters; ++it) {
        mma_nvf4_warp(d, ad, bd, i0, sfa, sfb, it > 0);
        mma_nvf4_warp(d, ad + 2, bd + 2, i0, sfa + 4, sfb + 4, true);
      }
    }
    tc_commit_warp(bar);
    mbar_wait_drain(bar, 0, &abort_flag, status, 91);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) {
    __syncwarp();
    tmem_dealloc(tmem, 256);
  }
}

}  // namespace
}  // namespace fp4attn

using namespace fp4attn;

extern "C" int fp4attn_debug_mma_peak(int kind, int iters, void* stream) {
  if (kind < 0 || kind > 2 || iters <= 0 || iters > (1 << 26)) return FP4ATTN_ERR_INVALID_ARG;
  DeviceStatus* status = device_status_ptr();
  if (!status) return FP4ATTN_ERR_CUDA;
  if (cudaFuncSetAttribute(mma_peak_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPeakSmem) != cudaSuccess)
    return FP4ATTN_ERR_CUDA;
  mma_peak_kernel<<<sm_count(), kPeakThreads, kPeakSmem, static_cast<cudaStream_t>(stream)>>>(kind, iters, status);
  return cuda_status(cudaGetLastError());
}

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
  if ((format < 0 || format > 2) || hi < lo || !pairs || !count || capacity <= 0) return FP4ATTN_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(count, 0, sizeof(int), s) != cudaSuccess) return FP4ATTN_ERR_CUDA;
  cvt_transitions_kernel<<<sm_count() * 8, 256, 0, s>>>(format, lo, hi, pairs, capacity, count);
  return cuda_status(cudaGetLastError());
}
