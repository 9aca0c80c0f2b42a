// Causal Direct-P attention backward for sm_103a.
//
// Method: "Hardware-Aware FP4 FlashAttention-4" ("What the paper found": for
// causal training the forward saves the quantized Q/K payloads, scales and
// LSE values; the backward reconstructs the probabilities from them and uses
// FP8 gradient operands, including E5M2 output gradients; the abstract says
// the same of the causal path).
//
// Every product runs on the tensor cores:
//   S   = Q^ K^T            saved NVFP4 Q, K        kind::mxf4nvf4 (as the forward)
//   dP  = dO V^T            E5M2 dO, E4M3 V         kind::mxf8f6f4, blocks along D
//   dV += P~^T dO           E4M3 P, E5M2 dO         blocks along the queries
//   dK += dS~^T Q           E5M2 dS, E4M3 Q         blocks along the queries
//   dQ += dS~ K             E5M2 dS, E4M3 K         blocks along the keys
// with P = 2^(c S - L) rebuilt from the saved LSE (L = LSE log2 e) and
// dS = P (dP - Delta), Delta = rowsum(dO o O).  FP8 operands carry one E8M0
// scale per 32 elements along the product's contraction axis.
//
// Two kernels of one template:
//   KV  one CTA per (128-key tile j, b*H+h), streaming the query tiles
//       i >= j.  Rows are keys: S^T and then dP^T pass through one TMEM bank
//       (S^T goes to registers as P^T before dP^T is computed into the bank),
//       and the dV and dK accumulators stay in TMEM for the whole run.
//   Q   one CTA per (128-query tile i, b*H+h), streaming the key tiles j <= i;
//       rows are queries, one dQ accumulator.
// Roles: kRowWarps row warps, kSplit per TMEM lane quarter: warp w takes
// columns kCols (w / 4) .. + kCols - 1 of the rows of lane quarter w % 4
// (row = TMEM lane); then the TMA producer warp and the MMA issuer warp
// (also the TMEM owner).  Every
// wait is bounded (the library's status word records where one gave up).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <mutex>

#include "fp8.cuh"
#include "internal.h"

namespace fp4attn {
namespace {

// Row warps per TMEM lane quarter (kSplit) and the columns each row thread takes.
constexpr int kSplit = 4;
constexpr int kRowWarps = 4 * kSplit;
constexpr int kCols = 128 / kSplit;  // one thread's columns of its row
constexpr int kBlk = kCols / 32;     // its 32-column scale blocks
constexpr int kBwdThreads = 32 * kRowWarps + 64;
constexpr int kWarpLoad = kRowWarps, kWarpMma = kRowWarps + 1;
constexpr uint32_t kBwdTmemCols = 512;

// kind::mxf8f6f4 instruction descriptor with the A and B formats (E4M3 0,
// E5M2 1), K-major operands, fp32 accumulate, UE8M0 scales and the byte of
// the 32-bit scale column each operand's scale is read from.
__host__ __device__ constexpr uint32_t idesc_mxf8_fmt(uint32_t M, uint32_t N, uint32_t afmt, uint32_t bfmt,
                                                      uint32_t a_sf_id, uint32_t b_sf_id) {
  return (b_sf_id & 3u) << 4 | (afmt & 7u) << 7 | (bfmt & 7u) << 10 | ((N >> 3) & 0x3Fu) << 17 | (1u << 23) |
         ((M >> 4) & 0x1Fu) << 24 | (a_sf_id & 3u) << 29;
}

// Shared-memory plan.  "Stationary" operands are loaded once per CTA, the
// others once per streamed tile, in two rings:
//   A4  NVFP4 tile of the stationary side (KV: K^, Q: Q^), 128 x D/2 bytes
//   A8  MXFP8 rows of the stationary side (KV: E4M3 V, Q: E5M2 dO), 128 x D
//   W1  the first tile the row threads write (KV: E4M3 P~^T, Q: E5M2 dS~),
//       128 x 128 bytes; W2 (KV only) the second (E5M2 dS~^T)
//   ring A (operands of S and dP, needed first in a step): B4 (KV: Q^, Q:
//       K^) with its scale atoms, B8 (KV: E5M2 dO rows, Q: E4M3 V rows) with
//       its atom, and (KV only) the tile's 128 fp32 -L and 128 fp32 Delta
//   ring B (operands of the step's last products): T1 (sequence-blocked,
//       transposed: KV: E5M2 dO^T, Q: E4M3 K^T), T2 (KV only: E4M3 Q^T),
//       with their atoms
// Ring A gets the deeper ring: its slot is free as soon as the step's S and
// dP products are complete and its -L / Delta read, well before the step's
// last products release ring B.  128-byte-swizzled tiles start on 1024-byte
// boundaries.
template <int D, bool KV>
struct BwdLayout {
  static constexpr int kT4 = 128 * D / 2;
  static constexpr int kT8 = 128 * D;  // also D x 128 (transposed tiles)
  static constexpr int kTW = 128 * 128;
  static constexpr int kSf4 = (D / 64) * 512;
  static constexpr int kA4 = 0;
  static constexpr int kA8 = kA4 + kT4;
  static constexpr int kW1 = kA8 + kT8;
  static constexpr int kW2 = kW1 + kTW;
  static constexpr int kRing0 = kW2 + (KV ? kTW : 0);
  static constexpr int kBigA = kT4 + kT8;                    // B4, B8
  static constexpr int kBigB = kT8 + (KV ? kT8 : 0);         // T1, T2
  static constexpr int kSmallA = kSf4 + 512 + (KV ? 1024 : 0);  // B4 scales, B8 atom, -L, Delta
  static constexpr int kSmallB = 512 + (KV ? 512 : 0);          // T1 atom, T2 atom
  static constexpr int kFixedSmall = kSf4 + 512 + 512 + (KV ? 512 : 0);
  static constexpr int kNumBarsMax = 1 + 2 * 8 + 10;
  static constexpr int kBudget = 225 * 1024;
  static constexpr int kAvail = kBudget - kRing0 - kFixedSmall - kNumBarsMax * 8 - 64;
  static constexpr int kFitA = (kAvail - 2 * (kBigB + kSmallB)) / (kBigA + kSmallA);
  static constexpr int kStagesA = kFitA < 4 ? kFitA : 4;
  static constexpr int kFitB = (kAvail - kStagesA * (kBigA + kSmallA)) / (kBigB + kSmallB);
  static constexpr int kStagesB = kFitB < 4 ? kFitB : 4;
  // ring tiles
  static constexpr int kB4 = 0, kB8 = kT4;  // within an A slot
  static constexpr int kT1 = 0, kT2 = kT8;  // within a B slot
  static constexpr int kRingB0 = kRing0 + kStagesA * kBigA;
  __host__ __device__ static constexpr int big_a(int s) { return kRing0 + s * kBigA; }
  __host__ __device__ static constexpr int big_b(int s) { return kRingB0 + s * kBigB; }
  // small buffers after every big tile
  static constexpr int kSmall = kRingB0 + kStagesB * kBigB;
  static constexpr int kSfA4 = kSmall;
  static constexpr int kAtA8 = kSfA4 + kSf4;
  static constexpr int kAtW1 = kAtA8 + 512;
  static constexpr int kAtW2 = kAtW1 + 512;  // KV only
  static constexpr int kSmallA0 = kAtW1 + 512 + (KV ? 512 : 0);
  static constexpr int kSsB4 = 0, kSsB8 = kSf4, kSsL = kSf4 + 512, kSsDelta = kSf4 + 1024;  // in an A slot
  static constexpr int kSsT1 = 0, kSsT2 = 512;                                              // in a B slot
  static constexpr int kSmallB0 = kSmallA0 + kStagesA * kSmallA;
  __host__ __device__ static constexpr int small_a(int s) { return kSmallA0 + s * kSmallA; }
  __host__ __device__ static constexpr int small_b(int s) { return kSmallB0 + s * kSmallB; }
  static constexpr int kBars = kSmallB0 + kStagesB * kSmallB;
  static constexpr int kNumBars = 1 + 2 * kStagesA + 2 * kStagesB + 10;
  static constexpr int kMisc = kBars + kNumBars * 8;
  static constexpr int kBytes = kMisc + 16;
  static constexpr int kAlloc = (kBytes + 1024 > 120 * 1024) ? kBytes + 1024 : 120 * 1024;
  static_assert(kStagesA >= 2 && kStagesB >= 2, "each ring needs two slots");
  static_assert(kNumBars <= kNumBarsMax, "barrier space");
  static_assert(kAlloc <= 227 * 1024, "shared memory of one CTA");
  static_assert(kA8 % 1024 == 0 && kW1 % 1024 == 0 && kRing0 % 1024 == 0 && kBigA % 1024 == 0 &&
                    kBigB % 1024 == 0 && kB8 % 1024 == 0 && kT2 % 1024 == 0 && kRingB0 % 1024 == 0,
                "tiles keep 1024-B alignment");
};

// TMEM plan: the S and dP banks, the accumulators, the scale-factor
// columns.  Where the columns allow (the dQ kernel, and the dK/dV kernel at
// D = 64) S and dP have banks of their own; the dK/dV kernel at D = 128
// passes both through one bank (S goes to registers before dP is computed).
template <int D, bool KV>
struct BwdCols {
  static constexpr bool kTwoBanks = !KV || D == 64;
  static constexpr uint32_t kBankS = 0;                       // 128 fp32 columns
  static constexpr uint32_t kBankDP = kTwoBanks ? 128 : 0;    // 128 fp32 columns
  static constexpr uint32_t kAcc0 = kTwoBanks ? 256 : 128;    // KV: dV, Q: dQ (D columns)
  static constexpr uint32_t kAcc1 = kAcc0 + D;                // KV: dK
  static constexpr uint32_t kSfA4 = kAcc0 + (KV ? 2 * D : D);  // D/64 atoms of 4 columns
  static constexpr uint32_t kSfB4 = kSfA4 + 4 * (D / 64);
  static constexpr uint32_t kSfA8 = kSfB4 + 4 * (D / 64);
  static constexpr uint32_t kSfB8 = kSfA8 + 4;
  static constexpr uint32_t kSfW1 = kSfB8 + 4;
  static constexpr uint32_t kSfT1 = kSfW1 + 4;
  static constexpr uint32_t kSfW2 = kSfT1 + 4;
  static constexpr uint32_t kSfT2 = kSfW2 + 4;
  static_assert(kSfT2 + 4 <= kBwdTmemCols, "TMEM plan exceeds 512 columns");
};

struct BwdParams {
  const uint8_t* sf_a4;  // stationary NVFP4 scale atoms (KV: K, Q: Q)
  const uint8_t* sf_b4;  // streamed NVFP4 scale atoms (KV: Q, Q: K)
  const uint8_t* at_a8;  // stationary row atoms (KV: V rows, Q: dO rows)
  const uint8_t* at_b8;  // streamed row atoms (KV: dO rows, Q: V rows)
  const uint8_t* at_t1;  // streamed transposed atoms (KV: dO^T, Q: K^T)
  const uint8_t* at_t2;  // KV: Q^T atoms
  const float* nl2;      // [B*H, Npad] -LSE log2 e (-inf past N)
  const float* delta;    // [B*H, Npad] rowsum(dO o O) (0 past N)
  const float* g_q;
  const float* g_k;
  float* out0;  // KV: dV, Q: dQ   [B,H,N,D] fp32
  float* out1;  // KV: dK
  DeviceStatus* status;
  int N;
  int ntiles;
  float softmax_scale;
};

// One 32-element block of fp32 values -> MX FP8 codes: the block's scale
// exponent (returned) and 32 code bytes stored as two 16-byte chunks of a
// 128-byte row under the 128-byte swizzle (chunk c of row r at c ^ (r % 8)).
template <int FMT>
__device__ __forceinline__ int mx_block_store(const float* x, uint32_t row_base, int blk, int row) {
  float amax = fabsf(x[0]);
#pragma unroll
  for (int i = 1; i < 31; i += 2) amax = fmax3(amax, fabsf(x[i]), fabsf(x[i + 1]));
  amax = fmaxf(amax, fabsf(x[31]));
  const int e = mx_exp_f32<FMT>(amax);
  const float inv = pow2_neg(e);
  float y[32];
#pragma unroll
  for (int i = 0; i < 32; i += 2) fmul2(y[i], y[i + 1], x[i], x[i + 1], inv, inv);
  uint32_t w[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) w[q] = cvt_fp8x4<FMT>(y[4 * q], y[4 * q + 1], y[4 * q + 2], y[4 * q + 3]);
  const int c0 = 2 * blk, c1 = 2 * blk + 1;
  sts_u4(row_base + ((c0 ^ (row & 7)) * 16), w[0], w[1], w[2], w[3]);
  sts_u4(row_base + ((c1 ^ (row & 7)) * 16), w[4], w[5], w[6], w[7]);
  return e;
}

template <int D, bool KV>
__global__ void __launch_bounds__(kBwdThreads, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap tm_a4, const __grid_constant__ CUtensorMap tm_b4,
               const __grid_constant__ CUtensorMap tm_a8, const __grid_constant__ CUtensorMap tm_b8,
               const __grid_constant__ CUtensorMap tm_t1, const __grid_constant__ CUtensorMap tm_t2,
               const BwdParams p) {
  using L = BwdLayout<D, KV>;
  using C = BwdCols<D, KV>;
  constexpr int kSA = L::kStagesA, kSB = L::kStagesB;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBars);
  uint64_t* bar_fixed = bars;
  uint64_t* bar_full_a = bars + 1;                 // [kSA] ring A slot landed
  uint64_t* bar_empty_a = bar_full_a + kSA;        // [kSA] ring A slot free
  uint64_t* bar_full_b = bar_empty_a + kSA;        // [kSB] ring B slot landed
  uint64_t* bar_empty_b = bar_full_b + kSB;        // [kSB] ring B slot free
  uint64_t* bar_s_full = bar_empty_b + kSB;        // S (S^T) is in the bank
  uint64_t* bar_pulled = bar_s_full + 1;          // the row threads hold S (one bank: it may take dP)
  uint64_t* bar_dp_full = bar_s_full + 2;         // dP (dP^T) is in its bank
  uint64_t* bar_bank_free = bar_s_full + 3;       // dP pulled (one bank: it may take the next S)
  uint64_t* bar_w1_full = bar_s_full + 4;         // W1 tile and atom written
  uint64_t* bar_w1_done = bar_s_full + 5;         // the product reading W1 is complete
  uint64_t* bar_w2_full = bar_s_full + 6;         // KV: W2 written
  uint64_t* bar_w2_done = bar_s_full + 7;         // KV: its product is complete
  uint64_t* bar_drain = bar_s_full + 8;           // the MMA warp's last commit
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.y;
  const int N = p.N;
  const int T = p.ntiles;
  const int npad = T * 128;
  // stationary tile and streamed tiles: KV: key tile j, query tiles j .. T-1;
  // Q: query tile i (largest first), key tiles 0 .. i
  const int tile0 = KV ? static_cast<int>(blockIdx.x) : T - 1 - static_cast<int>(blockIdx.x);
  const int nsteps = KV ? T - tile0 : tile0 + 1;
  auto streamed = [&](int t) { return KV ? tile0 + t : t; };

  if (threadIdx.x == 0) {
    mbar_init(bar_fixed, 1);
    for (int s = 0; s < kSA; ++s) {
      mbar_init(bar_full_a + s, 1);
      mbar_init(bar_empty_a + s, 1);
    }
    for (int s = 0; s < kSB; ++s) {
      mbar_init(bar_full_b + s, 1);
      mbar_init(bar_empty_b + s, 1);
    }
    mbar_init(bar_s_full, 1);
    mbar_init(bar_pulled, kRowWarps);
    mbar_init(bar_dp_full, 1);
    mbar_init(bar_bank_free, kRowWarps);
    mbar_init(bar_w1_full, kRowWarps);
    mbar_init(bar_w1_done, 1);
    mbar_init(bar_w2_full, kRowWarps);
    mbar_init(bar_w2_done, 1);
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(tmem_slot, kBwdTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // The only CTA on the SM holds all 512 columns: its allocation starts at 0.
  const uint32_t tmem_base = *tmem_slot;
  constexpr uint32_t tmem = 0;
  if (tmem_base != 0) {
    if (threadIdx.x == 0 && atomicCAS(&p.status->timeout, 0u, 1u) == 0u) p.status->where = 99;
  } else if (warp == kWarpLoad) {
    // ------------------------------------------------------------ TMA producer
    const bool leader = elect_one();
    const size_t sf4_bytes = L::kSf4;
    if (leader) {
      prefetch_tmap(&tm_a4);
      prefetch_tmap(&tm_b4);
      prefetch_tmap(&tm_a8);
      prefetch_tmap(&tm_b8);
      prefetch_tmap(&tm_t1);
      if (KV) prefetch_tmap(&tm_t2);
      mbar_arrive_expect_tx(bar_fixed, L::kT4 + L::kT8 + L::kSf4 + 512);
      tma_load_3d(smem + L::kA4, &tm_a4, bar_fixed, 0, tile0 * 128, bh);
      tma_load_3d(smem + L::kA8, &tm_a8, bar_fixed, 0, tile0 * 128, bh);
      bulk_load(smem + L::kSfA4, p.sf_a4 + (static_cast<size_t>(bh) * T + tile0) * sf4_bytes, L::kSf4, bar_fixed);
      bulk_load(smem + L::kAtA8, p.at_a8 + (static_cast<size_t>(bh) * T + tile0) * 512, 512, bar_fixed);
    }
    int issued = 0;
    for (int t = 0; t < nsteps; ++t) {
      const int sa = t % kSA, sb = t % kSB;
      if (t >= kSA) {
        const bool ok = mbar_wait(bar_empty_a + sa, ((t / kSA) - 1) & 1, abort_flag, p.status, 30);
        if (!__all_sync(0xFFFFFFFFu, ok)) break;
      }
      const int u = streamed(t);
      const size_t at = (static_cast<size_t>(bh) * T + u) * 512;
      if (leader) {
        uint8_t* big = smem + L::big_a(sa);
        uint8_t* small = smem + L::small_a(sa);
        constexpr uint32_t kTxA = L::kT4 + L::kT8 + L::kSf4 + 512 + (KV ? 1024 : 0);
        mbar_arrive_expect_tx(bar_full_a + sa, kTxA);
        tma_load_3d(big + L::kB4, &tm_b4, bar_full_a + sa, 0, u * 128, bh);
        tma_load_3d(big + L::kB8, &tm_b8, bar_full_a + sa, 0, u * 128, bh);
        bulk_load(small + L::kSsB4, p.sf_b4 + (static_cast<size_t>(bh) * T + u) * sf4_bytes, L::kSf4,
                  bar_full_a + sa);
        bulk_load(small + L::kSsB8, p.at_b8 + at, 512, bar_full_a + sa);
        if (KV) {
          const size_t lo = static_cast<size_t>(bh) * npad + static_cast<size_t>(u) * 128;
          bulk_load(small + L::kSsL, p.nl2 + lo, 512, bar_full_a + sa);
          bulk_load(small + L::kSsDelta, p.delta + lo, 512, bar_full_a + sa);
        }
      }
      __syncwarp();
      if (t >= kSB) {
        const bool ok = mbar_wait(bar_empty_b + sb, ((t / kSB) - 1) & 1, abort_flag, p.status, 29);
        if (!__all_sync(0xFFFFFFFFu, ok)) {
          issued = -(t + 1);  // ring A of step t was issued, ring B was not
          break;
        }
      }
      if (leader) {
        uint8_t* big = smem + L::big_b(sb);
        uint8_t* small = smem + L::small_b(sb);
        constexpr uint32_t kTxB = L::kT8 + 512 + (KV ? L::kT8 + 512 : 0);
        mbar_arrive_expect_tx(bar_full_b + sb, kTxB);
        tma_load_2d(big + L::kT1, &tm_t1, bar_full_b + sb, u * 128, bh * D);
        bulk_load(small + L::kSsT1, p.at_t1 + at, 512, bar_full_b + sb);
        if (KV) {
          tma_load_2d(big + L::kT2, &tm_t2, bar_full_b + sb, u * 128, bh * D);
          bulk_load(small + L::kSsT2, p.at_t2 + at, 512, bar_full_b + sb);
        }
      }
      issued = t + 1;
      __syncwarp();
    }
    // no copy into this CTA's shared memory may be in flight when it leaves
    const int issued_a = issued < 0 ? -issued : issued, issued_b = issued < 0 ? -issued - 1 : issued;
    for (int t = issued_a - kSA < 0 ? 0 : issued_a - kSA; t < issued_a; ++t)
      mbar_wait_drain(bar_full_a + (t % kSA), (t / kSA) & 1, abort_flag, p.status, 31);
    for (int t = issued_b - kSB < 0 ? 0 : issued_b - kSB; t < issued_b; ++t)
      mbar_wait_drain(bar_full_b + (t % kSB), (t / kSB) & 1, abort_flag, p.status, 28);
    mbar_wait_drain(bar_fixed, 0, abort_flag, p.status, 32);
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    auto wait = [&](uint64_t* bar, uint32_t parity, unsigned site) {
      return __all_sync(0xFFFFFFFFu, mbar_wait(bar, parity, abort_flag, p.status, site));
    };
    constexpr uint32_t kSw4 = (D == 128) ? 4u : 6u;  // NVFP4 rows of 64 or 32 bytes
    constexpr uint32_t kSbo4 = 8 * (D / 2);
    constexpr uint32_t kSw8 = (D == 128) ? 2u : 4u;  // MXFP8 rows of D bytes: 128- or 64-byte swizzle
    constexpr uint32_t kSbo8 = 8 * D;
    // stationary and streamed operand formats of the dP product
    constexpr uint32_t kFmtA8 = KV ? kFmtE4M3 : kFmtE5M2, kFmtB8 = KV ? kFmtE5M2 : kFmtE4M3;
    constexpr uint32_t idesc_s = idesc_fp4_block_scaled(128, 128, 0, 0, 0);
    const uint64_t a4 = smem_desc(smem_u32(smem + L::kA4), 16, kSbo4, kSw4);
    const uint64_t a8 = smem_desc(smem_u32(smem + L::kA8), 16, kSbo8, kSw8);
    const uint64_t w1 = smem_desc(smem_u32(smem + L::kW1), 16, 1024, 2u);
    const uint64_t w2 = smem_desc(smem_u32(smem + L::kW2), 16, 1024, 2u);
    const uint32_t bank_s = tmem + C::kBankS, bank_dp = tmem + C::kBankDP;
    bool ok = wait(bar_fixed, 0, 33);
    if (ok) {
      tc_fence_after();
#pragma unroll
      for (int a = 0; a < D / 64; ++a) tc_cp_sf_atom_warp(tmem + C::kSfA4 + 4 * a, smem_u32(smem + L::kSfA4 + a * 512));
      tc_cp_sf_atom_warp(tmem + C::kSfA8, smem_u32(smem + L::kAtA8));
    }
    // S = A4 B4^T of step t into the bank (its stage has landed, the bank is free)
    auto issue_s = [&](int t) {
      const int s = t % kSA;
      if (!wait(bar_full_a + s, (t / kSA) & 1, 34)) return false;
      // the S bank is free once the row threads hold the previous S (two
      // banks) or the previous dP (one bank)
      if (t > 0 && !wait(C::kTwoBanks ? bar_pulled : bar_bank_free, (t - 1) & 1, 35)) return false;
      tc_fence_after();
      uint8_t* small = smem + L::small_a(s);
#pragma unroll
      for (int a = 0; a < D / 64; ++a)
        tc_cp_sf_atom_warp(tmem + C::kSfB4 + 4 * a, smem_u32(small + L::kSsB4 + a * 512));
      const uint64_t b4 = smem_desc(smem_u32(smem + L::big_a(s) + L::kB4), 16, kSbo4, kSw4);
#pragma unroll
      for (int ks = 0; ks < D / 64; ++ks)
        mma_nvf4_warp(bank_s, a4 + 2 * ks, b4 + 2 * ks, idesc_s, tmem + C::kSfA4 + 4 * ks, tmem + C::kSfB4 + 4 * ks,
                      ks > 0);
      tc_commit_warp(bar_s_full);
      return true;
    };
    // dP = A8 B8^T of step t: into its own bank once the previous dP is
    // pulled (two banks), or into the S bank once the row threads hold S
    auto issue_dp = [&](int t) {
      const int s = t % kSA;
      if (C::kTwoBanks ? (t > 0 && !wait(bar_bank_free, (t - 1) & 1, 36)) : !wait(bar_pulled, t & 1, 36))
        return false;
      tc_fence_after();
      tc_cp_sf_atom_warp(tmem + C::kSfB8, smem_u32(smem + L::small_a(s) + L::kSsB8));
      const uint64_t b8 = smem_desc(smem_u32(smem + L::big_a(s) + L::kB8), 16, kSbo8, kSw8);
#pragma unroll
      for (int ks = 0; ks < D / 32; ++ks)
        mma_mxf8_warp(bank_dp, a8 + 2 * ks, b8 + 2 * ks, idesc_mxf8_fmt(128, 128, kFmtA8, kFmtB8, ks, ks),
                      tmem + C::kSfA8, tmem + C::kSfB8, ks > 0);
      tc_commit_warp(bar_dp_full);
      // Q: ring A of step t is free once S(t) and dP(t) are complete (the row
      // threads read nothing from it)
      if (!KV) tc_commit_warp(bar_empty_a + s);
      return true;
    };
    // acc0 += W1 T1^T  (KV: dV += P~^T dO, Q: dQ += dS~ K)
    auto issue_w1 = [&](int t) {
      const int s = t % kSB;
      if (!wait(bar_full_b + s, (t / kSB) & 1, 48)) return false;
      if (!wait(bar_w1_full, t & 1, 37)) return false;
      tc_fence_after();
      tc_cp_sf_atom_warp(tmem + C::kSfW1, smem_u32(smem + L::kAtW1));
      tc_cp_sf_atom_warp(tmem + C::kSfT1, smem_u32(smem + L::small_b(s) + L::kSsT1));
      const uint64_t t1 = smem_desc(smem_u32(smem + L::big_b(s) + L::kT1), 16, 1024, 2u);
      constexpr uint32_t kFmtW1 = KV ? kFmtE4M3 : kFmtE5M2, kFmtT1 = KV ? kFmtE5M2 : kFmtE4M3;
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_mxf8_warp(tmem + C::kAcc0, w1 + 2 * ks, t1 + 2 * ks, idesc_mxf8_fmt(128, D, kFmtW1, kFmtT1, ks, ks),
                      tmem + C::kSfW1, tmem + C::kSfT1, t > 0 || ks > 0);
      tc_commit_warp(bar_w1_done);
      return true;
    };
    // KV: acc1 += W2 T2^T  (dK += dS~^T Q)
    auto issue_w2 = [&](int t) {
      const int s = t % kSB;
      if (!wait(bar_w2_full, t & 1, 38)) return false;
      // KV: the row threads are done with the step's -L and Delta: ring A's
      // slot is free (S and dP of the step are complete: dP has been pulled)
      if (KV && lane == 0) mbar_arrive(bar_empty_a + (t % kSA));
      tc_fence_after();
      tc_cp_sf_atom_warp(tmem + C::kSfW2, smem_u32(smem + L::kAtW2));
      tc_cp_sf_atom_warp(tmem + C::kSfT2, smem_u32(smem + L::small_b(s) + L::kSsT2));
      const uint64_t t2 = smem_desc(smem_u32(smem + L::big_b(s) + L::kT2), 16, 1024, 2u);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_mxf8_warp(tmem + C::kAcc1, w2 + 2 * ks, t2 + 2 * ks, idesc_mxf8_fmt(128, D, kFmtE5M2, kFmtE4M3, ks, ks),
                      tmem + C::kSfW2, tmem + C::kSfT2, t > 0 || ks > 0);
      tc_commit_warp(bar_w2_done);
      return true;
    };
    // Software pipeline: each product is issued as soon as its bank and
    // operands are ready, ahead of the current step's last products.
    //   one bank,  KV step t: S(t+1) [after the dP(t) pull; ahead of dV(t),
    //              which is only needed before the next P~ is written],
    //              dV(t), dK(t), dP(t+1) [after the S(t+1) pull]
    //   two banks, KV step t: S(t+1) [after the S(t) pull], dV(t), dP(t+1)
    //              [after the dP(t) pull], dK(t)
    //   two banks, Q  step t: S(t+1), dP(t+1), dQ(t) [dS~ is written last]
    ok = ok && issue_s(0) && issue_dp(0);
    for (int t = 0; ok && t < nsteps; ++t) {
      const bool more = t + 1 < nsteps;
      if constexpr (C::kTwoBanks) {
        if (more && !(ok = issue_s(t + 1))) break;
        if (KV && !(ok = issue_w1(t))) break;
        if (more && !(ok = issue_dp(t + 1))) break;
        if (!(ok = KV ? issue_w2(t) : issue_w1(t))) break;
        tc_commit_warp(bar_empty_b + (t % kSB));
      } else {
        if (more && !(ok = issue_s(t + 1))) break;
        if (!(ok = issue_w1(t))) break;
        if (!(ok = issue_w2(t))) break;
        tc_commit_warp(bar_empty_b + (t % kSB));
        if (more && !(ok = issue_dp(t + 1))) break;
      }
    }
    // every MMA and scale copy must be complete before TMEM is freed
    tc_commit_warp(bar_drain);
    mbar_wait_drain(bar_drain, 0, abort_flag, p.status, 39);
  } else {
    // ------------------------------------------------------------ row threads
    const int row = threadIdx.x & 127;  // == TMEM lane
    const int part = warp >> 2;         // columns kCols part .. kCols part + kCols - 1
    const int col0 = kCols * part;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t t_bank = tmem + lane_base + C::kBankS + col0;
    const uint32_t t_dpbank = tmem + lane_base + C::kBankDP + col0;
    const int row_id = tile0 * 128 + row;  // KV: key, Q: query
    const float c = static_cast<float>(((static_cast<double>(p.softmax_scale) * 1.4426950408889634074) *
                                        static_cast<double>(*p.g_q)) * static_cast<double>(*p.g_k));
    // Q: this row's -L and Delta
    float nl2_row = 0.0f, delta_row = 0.0f;
    if constexpr (!KV) {
      nl2_row = p.nl2[static_cast<size_t>(bh) * npad + row_id];
      delta_row = p.delta[static_cast<size_t>(bh) * npad + row_id];
    }
    const uint32_t w1_row = smem_u32(smem + L::kW1 + row * 128);
    const uint32_t w2_row = smem_u32(smem + L::kW2 + row * 128);
    // this thread's scale bytes in its row's atom word
    const int at_off = (row & 31) * 16 + (row >> 5) * 4 + col0 / 32;
    auto store_scales = [&](uint32_t atom, const int (&e)[kBlk]) {
      if constexpr (kBlk == 2)
        sts_u16(atom + at_off, static_cast<uint16_t>((e[0] + 127) | ((e[1] + 127) << 8)));
      else
        sts_u8(atom + at_off, static_cast<uint32_t>(e[0] + 127));
    };
    bool ok = true;
    for (int t = 0; t < nsteps; ++t) {
      const int s = t % kSA;
      const uint32_t st_nl2 = smem_u32(smem + L::small_a(s) + L::kSsL) + 4 * col0;
      const uint32_t st_delta = smem_u32(smem + L::small_a(s) + L::kSsDelta) + 4 * col0;
      const bool diag = streamed(t) == tile0;
      ok = mbar_wait(bar_s_full, t & 1, abort_flag, p.status, 40);
      // KV: this step's L and Delta are read from the stage, so the row
      // threads observe the stage's own TMA barrier as well
      if (KV && ok) ok = mbar_wait(bar_full_a + s, (t / kSA) & 1, abort_flag, p.status, 46);
      if (!__all_sync(0xFFFFFFFFu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float pr[kCols];
#pragma unroll
      for (int b = 0; b < kBlk; ++b) tmem_ld32(t_bank + 32 * b, *reinterpret_cast<float(*)[32]>(pr + 32 * b));
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_pulled);
      // P = 2^(c S - L), one FMA and ex2 per element; causal mask on the
      // diagonal tile (KV: query col < key row; Q: key col > query row)
#pragma unroll
      for (int i = 0; i < kCols; i += 4) {
        const float4 l = KV ? lds_f4(st_nl2 + 4 * i) : make_float4(nl2_row, nl2_row, nl2_row, nl2_row);
        ffma2(pr[i], pr[i + 1], c, c, pr[i], pr[i + 1], l.x, l.y);
        ffma2(pr[i + 2], pr[i + 3], c, c, pr[i + 2], pr[i + 3], l.z, l.w);
#pragma unroll
        for (int u = 0; u < 4; ++u) pr[i + u] = ex2_approx(pr[i + u]);
      }
      if (diag) {
#pragma unroll
        for (int i = 0; i < kCols; ++i)
          if (KV ? (col0 + i < row) : (col0 + i > row)) pr[i] = 0.0f;
      }
      if constexpr (KV) {
        // P~^T: E4M3 codes blocked along the queries (this row's columns)
        if (t > 0) {
          ok = mbar_wait(bar_w1_done, (t - 1) & 1, abort_flag, p.status, 41);
          if (!__all_sync(0xFFFFFFFFu, ok)) {
            ok = false;
            break;
          }
        }
        int e[kBlk];
#pragma unroll
        for (int b = 0; b < kBlk; ++b) e[b] = mx_block_store<kFmtE4M3>(pr + 32 * b, w1_row, col0 / 32 + b, row);
        store_scales(smem_u32(smem + L::kAtW1), e);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_w1_full);
      }
      // dP to registers; the bank goes back for the next S at once
      ok = mbar_wait(bar_dp_full, t & 1, abort_flag, p.status, 42);
      if (!__all_sync(0xFFFFFFFFu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float dp[kCols];
#pragma unroll
      for (int b = 0; b < kBlk; ++b) tmem_ld32(t_dpbank + 32 * b, *reinterpret_cast<float(*)[32]>(dp + 32 * b));
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_bank_free);
      // dS = P (dP - Delta), E5M2 codes blocked along this row's columns
#pragma unroll
      for (int i = 0; i < kCols; i += 4) {
        const float4 dl = KV ? lds_f4(st_delta + 4 * i) : make_float4(delta_row, delta_row, delta_row, delta_row);
        fsub2(dp[i], dp[i + 1], dp[i], dp[i + 1], dl.x, dl.y);
        fsub2(dp[i + 2], dp[i + 3], dp[i + 2], dp[i + 3], dl.z, dl.w);
        fmul2(dp[i], dp[i + 1], pr[i], pr[i + 1], dp[i], dp[i + 1]);
        fmul2(dp[i + 2], dp[i + 3], pr[i + 2], pr[i + 3], dp[i + 2], dp[i + 3]);
      }
      if (t > 0) {
        ok = mbar_wait(KV ? bar_w2_done : bar_w1_done, (t - 1) & 1, abort_flag, p.status, 43);
        if (!__all_sync(0xFFFFFFFFu, ok)) {
          ok = false;
          break;
        }
      }
      const uint32_t ds_row = KV ? w2_row : w1_row;
      int e[kBlk];
#pragma unroll
      for (int b = 0; b < kBlk; ++b) e[b] = mx_block_store<kFmtE5M2>(dp + 32 * b, ds_row, col0 / 32 + b, row);
      store_scales(smem_u32(smem + (KV ? L::kAtW2 : L::kAtW1)), e);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(KV ? bar_w2_full : bar_w1_full);
    }
    // ------------------------------------------------------------ epilogue
    const int last = nsteps - 1;
    if (ok) ok = mbar_wait(bar_w1_done, last & 1, abort_flag, p.status, 44);
    if (KV && ok) ok = mbar_wait(bar_w2_done, last & 1, abort_flag, p.status, 45);
    if (__all_sync(0xFFFFFFFFu, ok)) {
      tc_fence_after();
      const bool store = row_id < N;
      // this thread writes channels kOut part .. kOut part + kOut - 1 of its row
      constexpr int kOut = D / kSplit;
      const size_t off = (static_cast<size_t>(bh) * N + (store ? row_id : 0)) * D + kOut * part;
#pragma unroll
      for (int acc = 0; acc < (KV ? 2 : 1); ++acc) {
        // KV: acc 0 = dV (unscaled), acc 1 = dK; Q: dQ
        const float scale = (KV && acc == 0) ? 1.0f : p.softmax_scale;
        float* dst = (acc == 0 ? p.out0 : p.out1) + off;
        const uint32_t src = tmem + lane_base + (acc == 0 ? C::kAcc0 : C::kAcc1) + kOut * part;
        if constexpr (kOut >= 32) {
#pragma unroll
          for (int cc = 0; cc < kOut / 32; ++cc) {
            float v[32];
            tmem_ld32(src + 32 * cc, v);
            tmem_wait_ld();
            if (store) {
#pragma unroll
              for (int i = 0; i < 8; ++i)
                reinterpret_cast<float4*>(dst + 32 * cc)[i] =
                    make_float4(v[4 * i] * scale, v[4 * i + 1] * scale, v[4 * i + 2] * scale, v[4 * i + 3] * scale);
            }
          }
        } else {
          float v[16];
          tmem_ld16(src, v);
          tmem_wait_ld();
          if (store) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
              reinterpret_cast<float4*>(dst)[i] =
                  make_float4(v[4 * i] * scale, v[4 * i + 1] * scale, v[4 * i + 2] * scale, v[4 * i + 3] * scale);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpMma) {
    __syncwarp();
    tmem_dealloc(tmem_base, kBwdTmemCols);
  }
}

// Delta = rowsum(dO o O) in fp32 and -L = -fp32(LSE * fp32(log2 e)) into the
// padded [B*H, Npad] arrays the backward kernels read (-L = -inf, Delta = 0
// past N, so those queries get P = 0); the exponent c S - L is then one FMA.  Eight lanes per row, one 16-byte load of dO
// and of O per lane and step.
template <int D>
__global__ void __launch_bounds__(256) bwd_prep_kernel(const uint4* __restrict__ o, const uint4* __restrict__ dout,
                                                       const float* __restrict__ lse, float* __restrict__ nl2,
                                                       float* __restrict__ delta, int N, int npad,
                                                       long long rows_pad) {
  constexpr int VPR = D / 8;  // 16-byte vectors per row
  const int sub = threadIdx.x & 7;
  for (long long r = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 3; r < rows_pad;
       r += (static_cast<long long>(gridDim.x) * blockDim.x) >> 3) {
    const long long bh = r / npad;
    const int n = static_cast<int>(r % npad);
    float acc = 0.0f;
    if (n < N) {
      const long long base = (bh * N + n) * VPR;
      for (int v = sub; v < VPR; v += 8) {
        const uint4 a = o[base + v], b = dout[base + v];
        const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc = fmaf(__uint_as_float(wa[i] << 16), __uint_as_float(wb[i] << 16), acc);
          acc = fmaf(__uint_as_float(wa[i] & 0xFFFF0000u), __uint_as_float(wb[i] & 0xFFFF0000u), acc);
        }
      }
    }
    acc += __shfl_xor_sync(0xFFFFFFFFu, acc, 1);
    acc += __shfl_xor_sync(0xFFFFFFFFu, acc, 2);
    acc += __shfl_xor_sync(0xFFFFFFFFu, acc, 4);
    if (sub == 0) {
      delta[r] = n < N ? acc : 0.0f;
      nl2[r] = n < N ? -__fmul_rn(lse[bh * N + n], 1.4426950408889634f) : -INFINITY;
    }
  }
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 bwd_encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

bool bwd_map(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
             const cuuint32_t* box, CUtensorMapSwizzle swz) {
  auto fn = bwd_encode_fn();
  if (!fn) return false;
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, rank, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// NVFP4 [BH, N, D/2] tiles of 128 rows; MXFP8 rows [BH, N, D] tiles of 128
// rows; sequence-blocked [BH*D, Npad] tiles of D rows x 128 tokens.
bool map_nvfp4(CUtensorMap* m, const void* base, int BH, int N, int D) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D / 2), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D / 2), static_cast<cuuint64_t>(N) * (D / 2)};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(D / 2), 128, 1};
  return bwd_map(m, base, 3, dims, strides, box, D == 128 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B);
}
bool map_rows8(CUtensorMap* m, const void* base, int BH, int N, int D) {
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(N) * D};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(D), 128, 1};
  return bwd_map(m, base, 3, dims, strides, box, D == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B);
}
bool map_t8(CUtensorMap* m, const void* base, int BH, int npad, int D) {
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(npad), static_cast<cuuint64_t>(BH) * D};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(npad)};
  const cuuint32_t box[2] = {128, static_cast<cuuint32_t>(D)};
  return bwd_map(m, base, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

template <int D, bool KV>
int launch_bwd_kernel(const CUtensorMap& a4, const CUtensorMap& b4, const CUtensorMap& a8, const CUtensorMap& b8,
                      const CUtensorMap& t1, const CUtensorMap& t2, const BwdParams& prm, int BH, cudaStream_t stream) {
  using L = BwdLayout<D, KV>;
  auto kern = bwd_kernel<D, KV>;
  static std::once_flag attr_once[64];
  int dev = 0;
  cudaGetDevice(&dev);
  cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once[dev & 63], [&] {
    attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  });
  if (attr_err != cudaSuccess) return FP4ATTN_ERR_CUDA;
  dim3 grid(prm.ntiles, BH);
  kern<<<grid, kBwdThreads, L::kAlloc, stream>>>(a4, b4, a8, b8, t1, t2, prm);
  return cuda_status(cudaGetLastError());
}

template <int D>
int launch_bwd(const fp4attn_nvfp4_t* q, const fp4attn_nvfp4_t* k, const fp4attn_fp8_t* v_rows,
               const fp4attn_fp8_t* do_rows, const fp4attn_fp8_t* do_t, const fp4attn_fp8_t* q_t,
               const fp4attn_fp8_t* k_t, const float* nl2, const float* delta, float* dq, float* dk, float* dv,
               int B, int H, int N, float softmax_scale, cudaStream_t stream, DeviceStatus* status) {
  const int BH = B * H, T = n_row_tiles(N), npad = T * 128;
  CUtensorMap mq, mk, mvr, mdor, mdot, mqt, mkt;
  if (!map_nvfp4(&mq, q->payload, BH, N, D) || !map_nvfp4(&mk, k->payload, BH, N, D) ||
      !map_rows8(&mvr, v_rows->payload, BH, N, D) || !map_rows8(&mdor, do_rows->payload, BH, N, D) ||
      !map_t8(&mdot, do_t->payload, BH, npad, D) || !map_t8(&mqt, q_t->payload, BH, npad, D) ||
      !map_t8(&mkt, k_t->payload, BH, npad, D))
    return FP4ATTN_ERR_CUDA;
  BwdParams kv{};
  kv.sf_a4 = k->sf;
  kv.sf_b4 = q->sf;
  kv.at_a8 = v_rows->sf;
  kv.at_b8 = do_rows->sf;
  kv.at_t1 = do_t->sf;
  kv.at_t2 = q_t->sf;
  kv.nl2 = nl2;
  kv.delta = delta;
  kv.g_q = q->g;
  kv.g_k = k->g;
  kv.out0 = dv;
  kv.out1 = dk;
  kv.status = status;
  kv.N = N;
  kv.ntiles = T;
  kv.softmax_scale = softmax_scale;
  BwdParams qp = kv;
  qp.sf_a4 = q->sf;
  qp.sf_b4 = k->sf;
  qp.at_a8 = do_rows->sf;
  qp.at_b8 = v_rows->sf;
  qp.at_t1 = k_t->sf;
  qp.at_t2 = nullptr;
  qp.out0 = dq;
  qp.out1 = nullptr;
  int st = launch_bwd_kernel<D, true>(mk, mq, mvr, mdor, mdot, mqt, kv, BH, stream);
  if (st != FP4ATTN_OK) return st;
  return launch_bwd_kernel<D, false>(mq, mk, mdor, mvr, mkt, mkt, qp, BH, stream);
}

bool fp8_ok(const fp4attn_fp8_t* t) { return t && t->payload && t->sf && aligned16(t->payload) && aligned16(t->sf); }

}  // namespace
}  // namespace fp4attn

using namespace fp4attn;

extern "C" int fp4attn_bwd_workspace_bytes(int B, int H, int N, int D, size_t* l2_bytes, size_t* delta_bytes) {
  const int st = check_shape(B, H, N, D);
  if (st != FP4ATTN_OK) return st;
  if (!l2_bytes || !delta_bytes) return FP4ATTN_ERR_INVALID_ARG;
  *l2_bytes = *delta_bytes = static_cast<size_t>(B) * H * n_row_tiles(N) * 128 * sizeof(float);
  return FP4ATTN_OK;
}

extern "C" int fp4attn_mxfp8_rows_bytes(int B, int H, int N, int D, size_t* payload_bytes, size_t* sf_bytes) {
  const int st = check_shape(B, H, N, D);
  if (st != FP4ATTN_OK) return st;
  if (!payload_bytes || !sf_bytes) return FP4ATTN_ERR_INVALID_ARG;
  *payload_bytes = static_cast<size_t>(B) * H * N * D;
  *sf_bytes = mxfp4_sf_bytes(B, H, N, D);
  return FP4ATTN_OK;
}

extern "C" int fp4attn_bwd_prep(const void* o, const void* dout, const float* lse, float* nl2, float* delta, int B,
                                int H, int N, int D, void* stream) {
  const int st = check_shape(B, H, N, D);
  if (st != FP4ATTN_OK) return st;
  if (!o || !dout || !lse || !nl2 || !delta) return FP4ATTN_ERR_INVALID_ARG;
  if (!aligned16(o) || !aligned16(dout) || !aligned16(lse) || !aligned16(nl2) || !aligned16(delta))
    return FP4ATTN_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int npad = n_row_tiles(N) * 128;
  const long long rows_pad = static_cast<long long>(B) * H * npad;
  long long want = (rows_pad * 8 + 255) / 256;
  const long long cap = static_cast<long long>(sm_count()) * 8;
  const int grid = static_cast<int>(want < cap ? want : cap);
  if (D == 128)
    bwd_prep_kernel<128><<<grid, 256, 0, s>>>(static_cast<const uint4*>(o), static_cast<const uint4*>(dout), lse,
                                              nl2, delta, N, npad, rows_pad);
  else
    bwd_prep_kernel<64><<<grid, 256, 0, s>>>(static_cast<const uint4*>(o), static_cast<const uint4*>(dout), lse, nl2,
                                             delta, N, npad, rows_pad);
  return cuda_status(cudaGetLastError());
}

extern "C" int fp4attn_bwd_directp_causal(const fp4attn_nvfp4_t* q, const fp4attn_nvfp4_t* k,
                                          const fp4attn_fp8_t* v_rows, const fp4attn_fp8_t* do_rows,
                                          const fp4attn_fp8_t* do_t, const fp4attn_fp8_t* q_t,
                                          const fp4attn_fp8_t* k_t, const float* nl2, const float* delta, float* dq,
                                          float* dk, float* dv, int B, int H, int N, int D, float softmax_scale,
                                          void* stream) {
  const int st = check_shape(B, H, N, D);
  if (st != FP4ATTN_OK) return st;
  if (!q || !k || !q->payload || !q->sf || !q->g || !k->payload || !k->sf || !k->g) return FP4ATTN_ERR_INVALID_ARG;
  if (!aligned16(q->payload) || !aligned16(q->sf) || !aligned16(k->payload) || !aligned16(k->sf))
    return FP4ATTN_ERR_INVALID_ARG;
  if (!fp8_ok(v_rows) || !fp8_ok(do_rows) || !fp8_ok(do_t) || !fp8_ok(q_t) || !fp8_ok(k_t))
    return FP4ATTN_ERR_INVALID_ARG;
  if (!nl2 || !delta || !dq || !dk || !dv || !aligned16(nl2) || !aligned16(delta) || !aligned16(dq) ||
      !aligned16(dk) || !aligned16(dv))
    return FP4ATTN_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.0f) || !std::isfinite(softmax_scale)) return FP4ATTN_ERR_INVALID_ARG;
  DeviceStatus* status = device_status_ptr();
  if (!status) return FP4ATTN_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (D == 128)
    return launch_bwd<128>(q, k, v_rows, do_rows, do_t, q_t, k_t, nl2, delta, dq, dk, dv, B, H, N, softmax_scale, s,
                           status);
  return launch_bwd<64>(q, k, v_rows, do_rows, do_t, q_t, k_t, nl2, delta, dq, dk, dv, B, H, N, softmax_scale, s,
                        status);
}
