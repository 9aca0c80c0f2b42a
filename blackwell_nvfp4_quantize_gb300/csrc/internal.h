// Host-side internals shared by the translation units of libfp4attn.so.
#pragma once
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "../../include/fp4attn.h"
#include "ptx.cuh"

namespace fp4attn {

// Per-device 256-byte status word (DeviceStatus at its start), set up by the
// first call on each device.  Returns nullptr if the set-up failed.
DeviceStatus* device_status_ptr();

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shape checks common to all entry points.
inline int check_shape(int B, int H, int N, int D) {
  if (B <= 0 || H <= 0 || N <= 0) return FP4ATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return FP4ATTN_ERR_UNSUPPORTED;
  const long long rows = static_cast<long long>(B) * H * N;
  if (rows >= (1ll << 31)) return FP4ATTN_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * H > 65535) return FP4ATTN_ERR_UNSUPPORTED;
  return FP4ATTN_OK;
}

inline int n_row_tiles(int N) { return (N + 127) / 128; }

inline size_t nvfp4_payload_bytes(int B, int H, int N, int D) {
  return static_cast<size_t>(B) * H * N * (D / 2);
}
inline size_t nvfp4_sf_bytes(int B, int H, int N, int D) {
  return static_cast<size_t>(B) * H * n_row_tiles(N) * (D / 64) * 512;
}
inline size_t mxfp4_payload_bytes(int B, int H, int N, int D) {
  return static_cast<size_t>(B) * H * D * (n_row_tiles(N) * 64);
}
inline size_t mxfp8_payload_bytes(int B, int H, int N, int D) {
  return static_cast<size_t>(B) * H * D * (n_row_tiles(N) * 128);
}
inline size_t mxfp4_sf_bytes(int B, int H, int N, int /*D*/) {
  return static_cast<size_t>(B) * H * n_row_tiles(N) * 512;
}

inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? FP4ATTN_OK : FP4ATTN_ERR_CUDA; }

int sm_count();

}  // namespace fp4attn
