// Forwards of independent problems straight from host memory, pipelined the
// way a serving loop runs them back to back: step i+1's upload and step
// i-1's download overlap step i's kernels.  Host code only; the device work
// is the library's own quantizers and forward kernels.
//
// Two device slots each hold one problem's bf16 Q, K, V and its O and LSE;
// one set of quantized operands is reused in stream order.
//   upload stream    H2D of step i's Q, K, V into slot i % 2, once step i-2's
//                    kernels have finished reading that slot
//   caller's stream  NVFP4 quantization of Q and K, MXFP4 or MXFP8 of V, the
//                    forward; waits for step i's upload and for step i-2's
//                    download out of the same slot
//   download stream  D2H of step i's O and LSE, once its forward is done
// The caller's stream finally waits for the download stream, so events the
// caller records on it around the call span the whole pipeline.
#include <cuda_runtime.h>

#include <cmath>

#include "internal.h"

namespace fp4attn {
namespace {

constexpr size_t kAlign = 256;
inline size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// Byte offsets of the workspace regions.
struct HostBatchPlan {
  size_t in_bytes, lse_bytes, slot_bytes;   // one slot: Q, K, V, O (bf16) and LSE
  size_t qk_payload, qk_sf, qk_bytes;       // one NVFP4 tensor: payload, atoms, g
  size_t v_payload, v_sf;                   // quantized V
  size_t total;
};

HostBatchPlan host_batch_plan(int B, int H, int N, int D, bool fp8pv) {
  HostBatchPlan p{};
  p.in_bytes = round_up(static_cast<size_t>(B) * H * N * D * 2);
  p.lse_bytes = round_up(static_cast<size_t>(B) * H * N * 4);
  p.slot_bytes = 4 * p.in_bytes + p.lse_bytes;
  p.qk_payload = round_up(nvfp4_payload_bytes(B, H, N, D));
  p.qk_sf = round_up(nvfp4_sf_bytes(B, H, N, D));
  p.qk_bytes = p.qk_payload + p.qk_sf + kAlign;
  p.v_payload = round_up(fp8pv ? mxfp8_payload_bytes(B, H, N, D) : mxfp4_payload_bytes(B, H, N, D));
  p.v_sf = round_up(mxfp4_sf_bytes(B, H, N, D));
  p.total = 2 * p.slot_bytes + 2 * p.qk_bytes + p.v_payload + p.v_sf;
  return p;
}

// Streams and events of one call, released when the call returns (CUDA
// defers the release of a stream or event until its pending work is done).
struct HostBatchSync {
  cudaStream_t up = nullptr, down = nullptr;
  cudaEvent_t start = nullptr, fin = nullptr, ev_up[2] = {}, ev_comp[2] = {}, ev_down[2] = {};
  cudaError_t create() {
    cudaError_t e = cudaStreamCreateWithFlags(&up, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&down, cudaStreamNonBlocking);
    cudaEvent_t* all[] = {&start, &fin, &ev_up[0], &ev_up[1], &ev_comp[0], &ev_comp[1], &ev_down[0], &ev_down[1]};
    for (cudaEvent_t* ev : all)
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
    return e;
  }
  ~HostBatchSync() {
    for (cudaEvent_t ev : {start, fin, ev_up[0], ev_up[1], ev_comp[0], ev_comp[1], ev_down[0], ev_down[1]})
      if (ev) cudaEventDestroy(ev);
    if (up) cudaStreamDestroy(up);
    if (down) cudaStreamDestroy(down);
  }
};

}  // namespace
}  // namespace fp4attn

using namespace fp4attn;

extern "C" int fp4attn_fwd_host_batch_workspace_bytes(int B, int H, int N, int D, int flags, size_t* bytes) {
  const int st = check_shape(B, H, N, D);
  if (st != FP4ATTN_OK) return st;
  if (!bytes || (flags & ~(FP4ATTN_HB_CAUSAL | FP4ATTN_HB_FP8PV)) != 0) return FP4ATTN_ERR_INVALID_ARG;
  *bytes = host_batch_plan(B, H, N, D, (flags & FP4ATTN_HB_FP8PV) != 0).total;
  return FP4ATTN_OK;
}

extern "C" int fp4attn_fwd_host_batch(int nsteps, const void* const* q_h, const void* const* k_h,
                                      const void* const* v_h, void* const* o_h, float* const* lse_h, int B, int H,
                                      int N, int D, float softmax_scale, int flags, void* workspace,
                                      size_t workspace_bytes, void* stream) {
  const int st = check_shape(B, H, N, D);
  if (st != FP4ATTN_OK) return st;
  if (nsteps < 1 || !q_h || !k_h || !v_h || !o_h || !lse_h || !workspace) return FP4ATTN_ERR_INVALID_ARG;
  if ((flags & ~(FP4ATTN_HB_CAUSAL | FP4ATTN_HB_FP8PV)) != 0) return FP4ATTN_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.0f) || !std::isfinite(softmax_scale)) return FP4ATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0) return FP4ATTN_ERR_INVALID_ARG;
  const bool causal = (flags & FP4ATTN_HB_CAUSAL) != 0, fp8pv = (flags & FP4ATTN_HB_FP8PV) != 0;
  const HostBatchPlan pl = host_batch_plan(B, H, N, D, fp8pv);
  if (workspace_bytes < pl.total) return FP4ATTN_ERR_INVALID_ARG;
  for (int i = 0; i < nsteps; ++i)
    if (!q_h[i] || !k_h[i] || !v_h[i] || !o_h[i] || !lse_h[i]) return FP4ATTN_ERR_INVALID_ARG;

  uint8_t* const base = static_cast<uint8_t*>(workspace);
  uint8_t* const qpay = base + 2 * pl.slot_bytes;
  uint8_t* const qsf = qpay + pl.qk_payload;
  float* const qg = reinterpret_cast<float*>(qsf + pl.qk_sf);
  uint8_t* const kpay = qpay + pl.qk_bytes;
  uint8_t* const ksf = kpay + pl.qk_payload;
  float* const kg = reinterpret_cast<float*>(ksf + pl.qk_sf);
  uint8_t* const vpay = kpay + pl.qk_bytes;
  uint8_t* const vsf = vpay + pl.v_payload;
  const fp4attn_nvfp4_t qq{qpay, qsf, qg}, kq{kpay, ksf, kg};
  const fp4attn_mxfp4_t v4{vpay, vsf};
  const fp4attn_mxfp8_t v8{vpay, vsf};
  const size_t io_bytes = static_cast<size_t>(B) * H * N * D * 2;
  const size_t lse_bytes = static_cast<size_t>(B) * H * N * 4;

  cudaStream_t comp = static_cast<cudaStream_t>(stream);
  HostBatchSync sync;
  cudaError_t e = sync.create();
  // the pipeline starts after the work already queued on the caller's stream
  if (e == cudaSuccess) e = cudaEventRecord(sync.start, comp);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(sync.up, sync.start, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(sync.down, sync.start, 0);
  int rc = cuda_status(e);
  for (int i = 0; i < nsteps && rc == FP4ATTN_OK; ++i) {
    const int s = i % 2;
    uint8_t* const slot = base + s * pl.slot_bytes;
    uint8_t *q = slot, *k = slot + pl.in_bytes, *v = slot + 2 * pl.in_bytes, *o = slot + 3 * pl.in_bytes;
    float* lse = reinterpret_cast<float*>(slot + 4 * pl.in_bytes);
    if (i >= 2) e = cudaStreamWaitEvent(sync.up, sync.ev_comp[s], 0);
    if (e == cudaSuccess) e = cudaMemcpyAsync(q, q_h[i], io_bytes, cudaMemcpyHostToDevice, sync.up);
    if (e == cudaSuccess) e = cudaMemcpyAsync(k, k_h[i], io_bytes, cudaMemcpyHostToDevice, sync.up);
    if (e == cudaSuccess) e = cudaMemcpyAsync(v, v_h[i], io_bytes, cudaMemcpyHostToDevice, sync.up);
    if (e == cudaSuccess) e = cudaEventRecord(sync.ev_up[s], sync.up);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(comp, sync.ev_up[s], 0);
    if (e == cudaSuccess && i >= 2) e = cudaStreamWaitEvent(comp, sync.ev_down[s], 0);
    if ((rc = cuda_status(e)) != FP4ATTN_OK) break;
    rc = fp4attn_quant_qk_nvfp4(q, qpay, qsf, qg, B, H, N, D, comp);
    if (rc == FP4ATTN_OK) rc = fp4attn_quant_qk_nvfp4(k, kpay, ksf, kg, B, H, N, D, comp);
    if (rc == FP4ATTN_OK)
      rc = fp8pv ? fp4attn_quant_v_mxfp8(v, vpay, vsf, B, H, N, D, comp)
                 : fp4attn_quant_v_mxfp4(v, vpay, vsf, B, H, N, D, comp);
    if (rc == FP4ATTN_OK) {
      if (fp8pv)
        rc = fp4attn_fwd_directp_fp8pv(&qq, &kq, &v8, o, lse, B, H, N, D, softmax_scale, causal ? 1 : 0, comp);
      else if (causal)
        rc = fp4attn_fwd_directp_causal(&qq, &kq, &v4, o, lse, B, H, N, D, softmax_scale, comp);
      else
        rc = fp4attn_fwd_directp(&qq, &kq, &v4, o, lse, B, H, N, D, softmax_scale, comp);
    }
    if (rc != FP4ATTN_OK) break;
    e = cudaEventRecord(sync.ev_comp[s], comp);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(sync.down, sync.ev_comp[s], 0);
    if (e == cudaSuccess) e = cudaMemcpyAsync(o_h[i], o, io_bytes, cudaMemcpyDeviceToHost, sync.down);
    if (e == cudaSuccess) e = cudaMemcpyAsync(lse_h[i], lse, lse_bytes, cudaMemcpyDeviceToHost, sync.down);
    if (e == cudaSuccess) e = cudaEventRecord(sync.ev_down[s], sync.down);
    rc = cuda_status(e);
  }
  // Whatever was queued, the caller's stream orders after it: the last
  // download (which follows every compute step) and the last upload.
  if (sync.fin) {
    for (cudaStream_t side : {sync.down, sync.up}) {
      if (!side) continue;
      cudaError_t f = cudaEventRecord(sync.fin, side);
      if (f == cudaSuccess) f = cudaStreamWaitEvent(comp, sync.fin, 0);
      if (f != cudaSuccess && rc == FP4ATTN_OK) rc = FP4ATTN_ERR_CUDA;
    }
  }
  return rc;
}
