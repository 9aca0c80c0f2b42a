// C-ABI glue of libfp4attn.so: status strings, buffer size queries, and the
// per-device status word that bounded device-side waits report into.
#include <mutex>

#include "internal.h"

namespace fp4attn {
namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
DeviceStatus* g_status[kMaxDevices] = {};
int g_sms[kMaxDevices] = {};
}  // namespace

DeviceStatus* device_status_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_status[dev]) {
    void* p = nullptr;
    if (cudaMalloc(&p, 256) != cudaSuccess) return nullptr;
    if (cudaMemset(p, 0, 256) != cudaSuccess) {
      cudaFree(p);
      return nullptr;
    }
    g_status[dev] = static_cast<DeviceStatus*>(p);
  }
  return g_status[dev];
}

int sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_sms[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    g_sms[dev] = n;
  }
  return g_sms[dev];
}

}  // namespace fp4attn

using namespace fp4attn;

extern "C" const char* fp4attn_status_string(int status) {
  switch (status) {
    case FP4ATTN_OK: return "ok";
    case FP4ATTN_ERR_INVALID_ARG: return "invalid argument (null or misaligned pointer, bad size or scale)";
    case FP4ATTN_ERR_UNSUPPORTED: return "unsupported shape (D must be 64 or 128; B*H <= 65535; B*H*N < 2^31)";
    case FP4ATTN_ERR_CUDA: return "CUDA runtime error";
    case FP4ATTN_ERR_TIMEOUT: return "a bounded device-side wait timed out; outputs are incomplete";
    default: return "unknown status";
  }
}

extern "C" int fp4attn_nvfp4_bytes(int B, int H, int N, int D, size_t* payload_bytes, size_t* sf_bytes) {
  const int st = check_shape(B, H, N, D);
  if (st != FP4ATTN_OK) return st;
  if (!payload_bytes || !sf_bytes) return FP4ATTN_ERR_INVALID_ARG;
  *payload_bytes = nvfp4_payload_bytes(B, H, N, D);
  *sf_bytes = nvfp4_sf_bytes(B, H, N, D);
  return FP4ATTN_OK;
}

extern "C" int fp4attn_mxfp4_v_bytes(int B, int H, int N, int D, size_t* payload_bytes, size_t* sf_bytes) {
  const int st = check_shape(B, H, N, D);
  if (st != FP4ATTN_OK) return st;
  if (!payload_bytes || !sf_bytes) return FP4ATTN_ERR_INVALID_ARG;
  *payload_bytes = mxfp4_payload_bytes(B, H, N, D);
  *sf_bytes = mxfp4_sf_bytes(B, H, N, D);
  return FP4ATTN_OK;
}

extern "C" int fp4attn_mxfp8_v_bytes(int B, int H, int N, int D, size_t* payload_bytes, size_t* sf_bytes) {
  const int st = check_shape(B, H, N, D);
  if (st != FP4ATTN_OK) return st;
  if (!payload_bytes || !sf_bytes) return FP4ATTN_ERR_INVALID_ARG;
  *payload_bytes = mxfp8_payload_bytes(B, H, N, D);
  *sf_bytes = mxfp4_sf_bytes(B, H, N, D);  // the same atoms
  return FP4ATTN_OK;
}

extern "C" int fp4attn_device_status(void* stream) {
  DeviceStatus* d = device_status_ptr();
  if (!d) return FP4ATTN_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return FP4ATTN_ERR_CUDA;
  DeviceStatus h{};
  if (cudaMemcpy(&h, d, sizeof h, cudaMemcpyDeviceToHost) != cudaSuccess) return FP4ATTN_ERR_CUDA;
  if (h.timeout) {
    if (cudaMemset(d, 0, sizeof h) != cudaSuccess) return FP4ATTN_ERR_CUDA;
    return FP4ATTN_ERR_TIMEOUT;
  }
  return FP4ATTN_OK;
}

extern "C" int fp4attn_debug_status_word_exists(int* exists) {
  if (!exists) return FP4ATTN_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FP4ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  *exists = g_status[dev] != nullptr ? 1 : 0;
  return FP4ATTN_OK;
}
