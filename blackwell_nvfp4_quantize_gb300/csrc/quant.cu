// Quantizers of the Direct-P attention forward ("Hardware-Aware FP4
// FlashAttention-4", section "What the paper found": Q and K in NVFP4, the PV
// product on MXFP4 E2M1 operands).
//
//  amax_kernel        : |x| maximum of a bf16 tensor -> one fp32 (as bits) in g
//  nvfp4_quant_kernel : 16-element blocks along D, E4M3 block scale, E2M1 codes
//  nvfp4_finalize     : g = amax / 2688 (1 for an all-zero tensor)
//  mxfp4_v_kernel     : 32-key blocks per channel, E8M0 scale, codes written
//                       key-inner (V transposed)
//  mxfp8_t_kernel     : the same for FP8 codes, one byte per token: E4M3 V of
//                       the FP8 P/V variant (training keeps FP8 probabilities
//                       and values) and the backward's sequence-blocked
//                       operands (E4M3 Q, K; E5M2 dO)
//  mxfp8_rows_kernel  : 32-element blocks along D, FP8 codes row-major (the
//                       backward's E4M3 V and E5M2 dO for dP = dO V^T)
//
// The data kernels are HBM-bound streaming passes: 16-byte vector loads with
// 4 to 16 of them in flight per thread (a read stream on this GPU needs about
// 8 to approach the DRAM peak; the transposing kernels keep 32 coalesced
// 4-byte loads in flight per thread instead), grids in multiples of the SM
// count, warp-shuffle reductions and coalesced stores.  fp32 arithmetic uses explicitly rounded intrinsics so that
// no multiply-add contraction changes a code.
#include <cuda_bf16.h>

#include "fp8.cuh"
#include "internal.h"

namespace fp4attn {
namespace {

constexpr float kNvfp4GlobalDiv = 2688.0f;  // 6 (E2M1 max) * 448 (E4M3 max)

__device__ __forceinline__ float e4m3_value(uint32_t code) {
  const uint32_t e = (code >> 3) & 15u, m = code & 7u;
  if (e == 0) return static_cast<float>(m) * 0x1p-9f;  // exact
  return __uint_as_float(((e + 120u) << 23) | (m << 20));
}

// 16-byte load of data read once: not kept in L1, with a 256-byte L2
// prefetch so each DRAM burst brings whole lines the neighbouring lanes use.
__device__ __forceinline__ uint4 ld_stream(const uint4* ptr) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(ptr));
  return v;
}

__device__ __forceinline__ float global_scale(float amax) {
  return amax > 0.0f ? __fdiv_rn(amax, kNvfp4GlobalDiv) : 1.0f;
}

// Max of |bf16| over the 8 bf16 values of a 16-byte vector, as bf16 bits.
__device__ __forceinline__ uint32_t absmax_vec(const uint4& v, uint32_t m2) {
  m2 = __vmaxu2(m2, v.x & 0x7FFF7FFFu);
  m2 = __vmaxu2(m2, v.y & 0x7FFF7FFFu);
  m2 = __vmaxu2(m2, v.z & 0x7FFF7FFFu);
  m2 = __vmaxu2(m2, v.w & 0x7FFF7FFFu);
  return m2;
}

// Each warp streams contiguous chunks of 32 * kAmaxUnroll vectors (8 KB),
// all of a chunk's loads in flight at once; chunks go round-robin over warps.
constexpr int kAmaxUnroll = 16;

__global__ void __launch_bounds__(256) amax_kernel(const uint4* __restrict__ x, long long nvec,
                                                   unsigned int* __restrict__ amax_bits) {
  uint32_t m2 = 0;
  const int lane = threadIdx.x & 31;
  constexpr long long kChunk = 32ll * kAmaxUnroll;
  const long long wstride = static_cast<long long>(gridDim.x) * blockDim.x * kAmaxUnroll;
  long long base = (static_cast<long long>(blockIdx.x) * blockDim.x + (threadIdx.x & ~31)) * kAmaxUnroll;
  for (; base + kChunk <= nvec; base += wstride) {
    uint4 a[kAmaxUnroll];
#pragma unroll
    for (int u = 0; u < kAmaxUnroll; ++u) a[u] = ld_stream(x + base + 32 * u + lane);
#pragma unroll
    for (int u = 0; u < kAmaxUnroll; ++u) m2 = absmax_vec(a[u], m2);
  }
  // the partial last chunk falls to the one warp whose turn it is
  for (long long i = base + lane; i < nvec; i += 32) m2 = absmax_vec(ld_stream(x + i), m2);
  uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
  m = __reduce_max_sync(0xFFFFFFFFu, m);
  __shared__ uint32_t red[8];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    uint32_t v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0u;
    v = __reduce_max_sync(0xFFFFFFFFu, v);
    // non-negative floats order like their bit patterns
    if (threadIdx.x == 0 && v != 0) atomicMax(amax_bits, v << 16);
  }
}

// One thread per 16-element block; a warp covers 32 consecutive blocks, so
// the 4 scale bytes of one atom word come from 4 neighbouring lanes.  Each
// warp takes kQuantUnroll such groups (4 KB of input) at a time, with all of
// their loads in flight before the first block is encoded.
constexpr int kQuantUnroll = 4;

__global__ void __launch_bounds__(256) nvfp4_quant_kernel(const uint4* __restrict__ x, uint2* __restrict__ payload,
                                                          uint8_t* __restrict__ sf, const float* __restrict__ amax_in,
                                                          int N, int D, long long nblocks) {
  const float g = global_scale(*amax_in);
  const float six_g = __fmul_rn(6.0f, g);
  const int kbs = D / 16;  // 4 or 8 blocks per row
  const int kbs_log2 = (D == 128) ? 3 : 2;
  const int ntiles = (N + 127) / 128;
  const int lane = threadIdx.x & 31;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x * kQuantUnroll;
  for (long long base0 = (static_cast<long long>(blockIdx.x) * blockDim.x + (threadIdx.x & ~31)) * kQuantUnroll;
       base0 < nblocks; base0 += stride) {
    uint4 va[kQuantUnroll], vb[kQuantUnroll];
#pragma unroll
    for (int u = 0; u < kQuantUnroll; ++u) {
      const long long blk = base0 + 32 * u + lane;
      if (blk < nblocks) {
        va[u] = ld_stream(x + 2 * blk);
        vb[u] = ld_stream(x + 2 * blk + 1);
      }
    }
#pragma unroll
    for (int u = 0; u < kQuantUnroll; ++u) {
      const long long blk = base0 + 32 * u + lane;
      const bool active = blk < nblocks;
      uint32_t sb = 0;
      if (active) {
        const uint4 a = va[u], b = vb[u];
        uint32_t m2 = absmax_vec(b, absmax_vec(a, 0u));
        const float amax_b = __uint_as_float(max(m2 & 0xFFFFu, m2 >> 16) << 16);
        sb = cvt_e4m3(__fdiv_rn(amax_b, six_g));
        const float s = __fmul_rn(e4m3_value(sb), g);
        uint2 out = make_uint2(0u, 0u);
        if (s != 0.0f) {
          const float inv = __frcp_rn(s);
          const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
          float y[16];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            y[2 * k] = __fmul_rn(__uint_as_float(w[k] << 16), inv);
            y[2 * k + 1] = __fmul_rn(__uint_as_float(w[k] & 0xFFFF0000u), inv);
          }
          out.x = cvt_e2m1x8(y[0], y[1], y[2], y[3], y[4], y[5], y[6], y[7]);
          out.y = cvt_e2m1x8(y[8], y[9], y[10], y[11], y[12], y[13], y[14], y[15]);
        }
        __stcs(payload + blk, out);
      }
      // gather the four scale bytes of one atom word into the lane with k == 0
      uint32_t word = sb << (8 * (lane & 3));
      word |= __shfl_xor_sync(0xFFFFFFFFu, word, 1);
      word |= __shfl_xor_sync(0xFFFFFFFFu, word, 2);
      if (active && (lane & 3) == 0) {
        // row = (b*H + h)*N + n < 2^31; for N a multiple of 128 the row's
        // 128-row tile index is row / 128 without splitting off the head
        const int row = static_cast<int>(blk >> kbs_log2);
        const int kb = static_cast<int>(blk) & (kbs - 1);
        long long tile;
        int r;
        if ((N & 127) == 0) {
          tile = row >> 7;
          r = row & 127;
        } else {
          const int bh = row / N, n = row - bh * N;
          tile = static_cast<long long>(bh) * ntiles + (n >> 7);
          r = n & 127;
        }
        const long long atom = tile * (kbs / 4) + (kb >> 2);
        *reinterpret_cast<uint32_t*>(sf + atom * 512 + (r & 31) * 16 + (r >> 5) * 4) = word;
      }
    }
  }
}

__global__ void nvfp4_finalize_kernel(float* g) { *g = global_scale(*g); }

// Channels d0, d0 + 1 of keys key0 .. key0 + 31 of head bh as 32-bit words
// (one per key; keys >= N read 0).  The lanes of a warp take consecutive
// channel pairs of the same keys, so each of the 32 loads, all in flight at
// once, reads 128 contiguous bytes of one key row.
template <int D>
__device__ __forceinline__ void load_pair_block(const uint4* __restrict__ v, long long bh, int N, int key0, int d0,
                                                uint32_t (&w2)[32]) {
  const int nk = N - key0;
  const uint32_t* col = reinterpret_cast<const uint32_t*>(v) + ((bh * N + key0) * D + d0) / 2;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    uint32_t x = 0u;
    if (i < nk) asm volatile("ld.global.nc.L1::no_allocate.L2::256B.u32 %0, [%1];" : "=r"(x) : "l"(col + i * (D / 2)));
    w2[i] = x;
  }
}

// V [B,H,N,D] bf16 -> V^T codes [B,H,D,Npad/2] + E8M0 atoms.  One CTA per
// (128-key tile, b*H+h); a thread takes the channel pair (d, d+1) of one
// 32-key block straight from global memory (no staging: the loads of a warp
// are coalesced key rows) and writes each channel's 16 code bytes with a
// plain write-back store, so L2 joins them with the neighbouring blocks'
// halves of each 32-byte sector before they reach DRAM.
template <int D>
__global__ void __launch_bounds__(256) mxfp4_v_kernel(const uint4* __restrict__ v, uint8_t* __restrict__ payload_t,
                                                      uint8_t* __restrict__ sf, int N) {
  __shared__ __align__(16) uint32_t atom[128];
  const int kt = blockIdx.x;
  const long long bh = blockIdx.y;
  const int ntiles = gridDim.x;
  const int npad_half = ntiles * 64;  // bytes per V^T row
  if (threadIdx.x < 128) atom[threadIdx.x] = 0u;
  __syncthreads();
  for (int pidx = threadIdx.x; pidx < 2 * D; pidx += 256) {
    const int d0 = 2 * (pidx % (D / 2)), kb = pidx / (D / 2);
    uint32_t w2[32];
    load_pair_block<D>(v, bh, N, kt * 128 + kb * 32, d0, w2);
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int d = d0 + c;
      uint32_t m = 0;
#pragma unroll
      for (int i = 0; i < 32; ++i) m = max(m, (c ? (w2[i] >> 16) : w2[i]) & 0x7FFFu);
      // e = smallest integer >= -127 with amax <= 6 * 2^e, from the bits of amax
      const uint32_t ebits = m >> 7, frac = m & 0x7Fu;  // bf16: 8 exponent, 7 mantissa bits
      int e = -127;
      if (ebits != 0) e = max(-127, static_cast<int>(ebits) - 127 - (frac <= 0x40u ? 2 : 1));
      const float inv_scale = __uint_as_float(static_cast<uint32_t>(127 - e) << 23);  // 2^-e, e <= 126
      float y[32];
#pragma unroll
      for (int i = 0; i < 32; ++i)
        y[i] = __fmul_rn(__uint_as_float(c ? (w2[i] & 0xFFFF0000u) : (w2[i] << 16)), inv_scale);
      uint4 out;
      out.x = cvt_e2m1x8(y[0], y[1], y[2], y[3], y[4], y[5], y[6], y[7]);
      out.y = cvt_e2m1x8(y[8], y[9], y[10], y[11], y[12], y[13], y[14], y[15]);
      out.z = cvt_e2m1x8(y[16], y[17], y[18], y[19], y[20], y[21], y[22], y[23]);
      out.w = cvt_e2m1x8(y[24], y[25], y[26], y[27], y[28], y[29], y[30], y[31]);
      *reinterpret_cast<uint4*>(payload_t + (bh * D + d) * npad_half + kt * 64 + kb * 16) = out;
      reinterpret_cast<uint8_t*>(atom)[(d & 31) * 16 + (d >> 5) * 4 + kb] = static_cast<uint8_t>(e + 127);
    }
  }
  __syncthreads();
  if (threadIdx.x < 32)
    reinterpret_cast<uint4*>(sf + (bh * ntiles + kt) * 512)[threadIdx.x] =
        reinterpret_cast<const uint4*>(atom)[threadIdx.x];
}

// MXFP8 along the sequence, transposed: the same loads, stores and atoms as
// mxfp4_v_kernel; the scale is the smallest 2^e with amax <= fmt_max * 2^e
// and each token keeps one FP8 byte.
template <int D, int FMT>
__global__ void __launch_bounds__(256) mxfp8_t_kernel(const uint4* __restrict__ v, uint8_t* __restrict__ payload_t,
                                                      uint8_t* __restrict__ sf, int N) {
  __shared__ __align__(16) uint32_t atom[128];
  const int kt = blockIdx.x;
  const long long bh = blockIdx.y;
  const int ntiles = gridDim.x;
  const int npad = ntiles * 128;  // bytes per transposed row
  if (threadIdx.x < 128) atom[threadIdx.x] = 0u;
  __syncthreads();
  for (int pidx = threadIdx.x; pidx < 2 * D; pidx += 256) {  // channel pairs, as in mxfp4_v_kernel
    const int d0 = 2 * (pidx % (D / 2)), kb = pidx / (D / 2);
    uint32_t w2[32];
    load_pair_block<D>(v, bh, N, kt * 128 + kb * 32, d0, w2);
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int d = d0 + c;
      uint32_t m = 0;
#pragma unroll
      for (int i = 0; i < 32; ++i) m = max(m, (c ? (w2[i] >> 16) : w2[i]) & 0x7FFFu);
      const int e = mx_exp_bf16<FMT>(m);
      const float inv_scale = pow2_neg(e);
      float y[32];
#pragma unroll
      for (int i = 0; i < 32; ++i)
        y[i] = __fmul_rn(__uint_as_float(c ? (w2[i] & 0xFFFF0000u) : (w2[i] << 16)), inv_scale);
      uint32_t wd[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) wd[i] = cvt_fp8x4<FMT>(y[4 * i], y[4 * i + 1], y[4 * i + 2], y[4 * i + 3]);
      uint4* dst = reinterpret_cast<uint4*>(payload_t + (bh * D + d) * npad + kt * 128 + kb * 32);
      dst[0] = make_uint4(wd[0], wd[1], wd[2], wd[3]);
      dst[1] = make_uint4(wd[4], wd[5], wd[6], wd[7]);
      reinterpret_cast<uint8_t*>(atom)[(d & 31) * 16 + (d >> 5) * 4 + kb] = static_cast<uint8_t>(e + 127);
    }
  }
  __syncthreads();
  if (threadIdx.x < 32)
    reinterpret_cast<uint4*>(sf + (bh * ntiles + kt) * 512)[threadIdx.x] =
        reinterpret_cast<const uint4*>(atom)[threadIdx.x];
}

// MXFP8 along D, row-major: one thread per 32-element block (four 16-byte
// loads, 32 code bytes out); the block's scale byte goes to its row's atom
// (row n % 128 of the (b, h, n / 128) atom, block d / 32).  The atoms are
// cleared beforehand, so blocks past D and rows past N read 0.
template <int D, int FMT>
__global__ void __launch_bounds__(256) mxfp8_rows_kernel(const uint4* __restrict__ x, uint4* __restrict__ payload,
                                                         uint8_t* __restrict__ sf, int N, long long nblocks) {
  constexpr int KB = D / 32;
  const int ntiles = (N + 127) / 128;
  for (long long b = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; b < nblocks;
       b += static_cast<long long>(gridDim.x) * blockDim.x) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = ld_stream(x + 4 * b + u);
    uint32_t m2 = 0;
#pragma unroll
    for (int u = 0; u < 4; ++u) m2 = absmax_vec(v[u], m2);
    const int e = mx_exp_bf16<FMT>(max(m2 & 0xFFFFu, m2 >> 16));
    const float inv_scale = pow2_neg(e);
    uint32_t wd[8];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
      float y[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        y[2 * i] = __fmul_rn(__uint_as_float(w[i] << 16), inv_scale);
        y[2 * i + 1] = __fmul_rn(__uint_as_float(w[i] & 0xFFFF0000u), inv_scale);
      }
      wd[2 * u] = cvt_fp8x4<FMT>(y[0], y[1], y[2], y[3]);
      wd[2 * u + 1] = cvt_fp8x4<FMT>(y[4], y[5], y[6], y[7]);
    }
    __stcs(payload + 2 * b, make_uint4(wd[0], wd[1], wd[2], wd[3]));
    __stcs(payload + 2 * b + 1, make_uint4(wd[4], wd[5], wd[6], wd[7]));
    const long long row = b / KB;
    const int kb = static_cast<int>(b % KB);
    const long long bh = row / N;
    const int n = static_cast<int>(row % N), r = n & 127;
    sf[(bh * ntiles + (n >> 7)) * 512 + (r & 31) * 16 + (r >> 5) * 4 + kb] = static_cast<uint8_t>(e + 127);
  }
}

int grid_for(long long work_items, int threads) {
  const long long want = (work_items + threads - 1) / threads;
  const long long cap = static_cast<long long>(sm_count()) * 8;  // 8 x 256 threads per SM
  return static_cast<int>(want < 1 ? 1 : (want < cap ? want : cap));
}

}  // namespace
}  // namespace fp4attn

using namespace fp4attn;

extern "C" int fp4attn_quant_qk_nvfp4(const void* x, uint8_t* payload, uint8_t* sf, float* g, int B, int H, int N,
                                      int D, void* stream) {
  int st = check_shape(B, H, N, D);
  if (st != FP4ATTN_OK) return st;
  if (!x || !payload || !sf || !g) return FP4ATTN_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(payload) || !aligned16(sf) || !aligned16(g)) return FP4ATTN_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const long long elems = static_cast<long long>(B) * H * N * D;
  const long long nvec = elems / 8;
  const long long nblocks = elems / 16;
  cudaError_t e = cudaMemsetAsync(g, 0, sizeof(float), s);
  if (e == cudaSuccess && (N % 128) != 0) e = cudaMemsetAsync(sf, 0, nvfp4_sf_bytes(B, H, N, D), s);
  if (e != cudaSuccess) return FP4ATTN_ERR_CUDA;
  amax_kernel<<<grid_for(nvec, 256 * kAmaxUnroll), 256, 0, s>>>(static_cast<const uint4*>(x), nvec,
                                                      reinterpret_cast<unsigned int*>(g));
  nvfp4_quant_kernel<<<grid_for(nblocks, 256 * kQuantUnroll), 256, 0, s>>>(static_cast<const uint4*>(x),
                                                             reinterpret_cast<uint2*>(payload), sf, g, N, D, nblocks);
  nvfp4_finalize_kernel<<<1, 1, 0, s>>>(g);
  return cuda_status(cudaGetLastError());
}

extern "C" int fp4attn_quant_v_mxfp4(const void* v, uint8_t* payload_t, uint8_t* sf, int B, int H, int N, int D,
                                     void* stream) {
  int st = check_shape(B, H, N, D);
  if (st != FP4ATTN_OK) return st;
  if (!v || !payload_t || !sf) return FP4ATTN_ERR_INVALID_ARG;
  if (!aligned16(v) || !aligned16(payload_t) || !aligned16(sf)) return FP4ATTN_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  dim3 grid(n_row_tiles(N), B * H);
  if (D == 128)
    mxfp4_v_kernel<128><<<grid, 256, 0, s>>>(static_cast<const uint4*>(v), payload_t, sf, N);
  else
    mxfp4_v_kernel<64><<<grid, 256, 0, s>>>(static_cast<const uint4*>(v), payload_t, sf, N);
  return cuda_status(cudaGetLastError());
}

extern "C" int fp4attn_quant_v_mxfp8(const void* v, uint8_t* payload_t, uint8_t* sf, int B, int H, int N, int D,
                                     void* stream) {
  return fp4attn_quant_mxfp8_t(v, payload_t, sf, FP4ATTN_FP8_E4M3, B, H, N, D, stream);
}

extern "C" int fp4attn_quant_mxfp8_t(const void* x, uint8_t* payload_t, uint8_t* sf, int fmt, int B, int H, int N,
                                     int D, void* stream) {
  int st = check_shape(B, H, N, D);
  if (st != FP4ATTN_OK) return st;
  if (!x || !payload_t || !sf) return FP4ATTN_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(payload_t) || !aligned16(sf)) return FP4ATTN_ERR_INVALID_ARG;
  if (fmt != FP4ATTN_FP8_E4M3 && fmt != FP4ATTN_FP8_E5M2) return FP4ATTN_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  dim3 grid(n_row_tiles(N), B * H);
  const uint4* src = static_cast<const uint4*>(x);
  if (D == 128) {
    if (fmt == FP4ATTN_FP8_E4M3) mxfp8_t_kernel<128, kFmtE4M3><<<grid, 256, 0, s>>>(src, payload_t, sf, N);
    else mxfp8_t_kernel<128, kFmtE5M2><<<grid, 256, 0, s>>>(src, payload_t, sf, N);
  } else {
    if (fmt == FP4ATTN_FP8_E4M3) mxfp8_t_kernel<64, kFmtE4M3><<<grid, 256, 0, s>>>(src, payload_t, sf, N);
    else mxfp8_t_kernel<64, kFmtE5M2><<<grid, 256, 0, s>>>(src, payload_t, sf, N);
  }
  return cuda_status(cudaGetLastError());
}

extern "C" int fp4attn_quant_mxfp8_rows(const void* x, uint8_t* payload, uint8_t* sf, int fmt, int B, int H, int N,
                                        int D, void* stream) {
  int st = check_shape(B, H, N, D);
  if (st != FP4ATTN_OK) return st;
  if (!x || !payload || !sf) return FP4ATTN_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(payload) || !aligned16(sf)) return FP4ATTN_ERR_INVALID_ARG;
  if (fmt != FP4ATTN_FP8_E4M3 && fmt != FP4ATTN_FP8_E5M2) return FP4ATTN_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(sf, 0, mxfp4_sf_bytes(B, H, N, D), s) != cudaSuccess) return FP4ATTN_ERR_CUDA;
  const long long nblocks = static_cast<long long>(B) * H * N * (D / 32);
  const int grid = grid_for(nblocks, 256);
  const uint4* src = static_cast<const uint4*>(x);
  uint4* dst = reinterpret_cast<uint4*>(payload);
  if (D == 128) {
    if (fmt == FP4ATTN_FP8_E4M3) mxfp8_rows_kernel<128, kFmtE4M3><<<grid, 256, 0, s>>>(src, dst, sf, N, nblocks);
    else mxfp8_rows_kernel<128, kFmtE5M2><<<grid, 256, 0, s>>>(src, dst, sf, N, nblocks);
  } else {
    if (fmt == FP4ATTN_FP8_E4M3) mxfp8_rows_kernel<64, kFmtE4M3><<<grid, 256, 0, s>>>(src, dst, sf, N, nblocks);
    else mxfp8_rows_kernel<64, kFmtE5M2><<<grid, 256, 0, s>>>(src, dst, sf, N, nblocks);
  }
  return cuda_status(cudaGetLastError());
}
