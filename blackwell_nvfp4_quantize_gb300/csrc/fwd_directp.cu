// Noncausal Direct-P FP4 attention forward for sm_103a.
//
// Method: "Hardware-Aware FP4 FlashAttention-4" (abstract: Direct-P for
// noncausal inference; "What the paper found": NVFP4 Q/K, log-softmax scores
// mapped directly to MXFP4 E2M1 probability codes with packed FMA and native
// conversion, denominator from the same rounded probabilities that PV
// consumes, LSE saved with O).
//
// One CTA computes two 128-row query tiles of one (b, h) and streams the key /
// value tiles of that head through a TMA ring; both query tiles consume every
// K/V tile.  Roles (352 threads):
//   warps 0-3, 4-7  softmax warpgroups, one per query tile, one thread per
//              query row.  Each reads its S row from TMEM (block maxima come
//              out of tcgen05.ld.red), maps the scores to E2M1 codes (packed
//              fp32 FMA, ex2, hardware e2m1x2 conversion), writes its P tile
//              and E8M0 scale atom to shared memory, rescales its O
//              accumulator when the reference maximum moves, and finally
//              writes O and LSE.
//   warp 8     TMA producer (one elected lane issues).
//   warps 9,10 tcgen05 MMA issuers, one per query tile (one elected lane
//              each; warp 9 also owns the TMEM allocation):
//              S   = Q_t K^T     kind::mxf4nvf4, 16-element UE4M3 scales
//              O_t += P_t V      kind::mxf4, 32-element UE8M0 scales
//              l_t  = P_t 1      the same P operand against a tile of E2M1
//                                ones: the tile's denominator from exactly the
//                                codes and scales the PV product consumes; the
//                                softmax warps add it up in fp32 registers
// TMEM (512 columns): one score bank S shared by the two tiles (a softmax
// warpgroup copies S to registers and releases the bank at once), two output
// banks, two 16-column l banks, and the scale-factor columns.
//
// Causal variant (the causal forward of "What the paper found": forward for
// causal training): key j is seen by query i only when j <= i.  Query tile
// qt needs the key tiles 0 .. qt, the last one masked along its diagonal, and
// no others.  Each of the two slots of a CTA (warpgroup + MMA warp) then runs
// a chain of two query tiles, i and T-1-i (T tiles per head): i+1 key tiles,
// then T-i, T+1 key steps in all, so both slots take every step together
// and the score bank keeps alternating between them.  A slot writes out its
// first tile's O and LSE when it starts on the second.  For odd T the middle
// tile forms a chain alone; the CTA holding it runs its longer slot alone for
// the last steps.  With two query tiles per slot the ring holds one K/V tile
// per slot and stage.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <mutex>

#include "fp8.cuh"
#include "internal.h"

namespace fp4attn {
namespace {

constexpr int kThreads = 352;
constexpr int kWarpTma = 8, kWarpMma0 = 9;  // warps 9 and 10 issue the MMAs of query tiles 0 and 1
// The MMA warp of a slot issues S = Q K(j+1)^T before its PV product of step
// j, so the ring must hold steps j and j+1 at once: at least two stages.
constexpr int kRingStages = 3;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;         // 128 columns: fp32 scores of 128 keys
constexpr uint32_t kColO = 128;       // tile t output at kColO + t * D
constexpr uint32_t kColL = 384;       // tile t denominator at kColL + 16 t
constexpr uint32_t kColSFQ = 416;     // tile t Q scale atoms at kColSFQ + 8 t
constexpr uint32_t kColSFK = 432;     // tile t, KV-step parity q: kColSFK + 16 t + 8 q
constexpr uint32_t kColSFV = 464;     // tile t, KV-step parity q: kColSFV + 8 t + 4 q
constexpr uint32_t kColSFP = 480;     // tile t P scale atom at kColSFP + 4 t
constexpr uint32_t kColSFOnes = 488;  // tile t unit scales of the ones tile at kColSFOnes + 4 t
static_assert(kColSFOnes + 8 <= kTmemCols, "TMEM plan exceeds 512 columns");
constexpr uint32_t kLN = 16;                     // N of the denominator MMA
constexpr float kLog2Six = 2.5849625007211561f;  // log2(6) rounded to fp32
constexpr float kLog2_448 = 8.8073549220576041f;  // log2(448) rounded to fp32 (E4M3 codes)
constexpr double kLog2E = 1.4426950408889634074;
// The reference maximum M of a row moves (and O, l are rescaled by an exact
// power of two) only when a tile's ceil(max score) exceeds it by more than
// this many binades; until then probabilities may exceed 1 by up to 2^8.
constexpr int kRescaleSlack = 8;

// P8: the FP8 P/V variant -- E4M3 probability codes and MXFP8 V, one byte
// per key, so V, P and the ones tile take twice the bytes of the E2M1 form.
// CH: chained slots (causal) -- four query tiles and one K/V tile per slot
// and stage.
template <int D, bool P8 = false, bool CH = false>
struct Layout {
  static constexpr int kRowBytes = D / 2;  // packed E2M1 bytes per Q/K row
  static constexpr int kTileQK = 128 * kRowBytes;
  static constexpr int kKeyBytes = P8 ? 128 : 64;  // bytes of 128 keys of P or V^T
  static constexpr int kTileV = D * kKeyBytes;     // D channels x 128 keys
  static constexpr int kTileP = 128 * kKeyBytes;   // 128 query rows x 128 keys
  static constexpr int kSFAtoms = D / 64;          // NVFP4 scale atoms per 128-row tile
  static constexpr int kNQ = CH ? 4 : 2;           // query tiles held
  static constexpr int kNKV = CH ? 2 : 1;          // K/V tiles per ring stage
  // (the largest form, chained E4M3 with D = 128, fits 227 KB with 2 stages)
  static constexpr int kStages = (CH && P8 && D == 128) ? 2 : kRingStages;
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kNQ * kTileQK;
  static constexpr int kV = kK + kStages * kNKV * kTileQK;
  static constexpr int kP = kV + kStages * kNKV * kTileV;  // two P tiles
  static constexpr int kOnes = kP + 2 * kTileP;             // 16 rows of ones (E2M1 or E4M3)
  static constexpr int kSFQ = kOnes + 16 * kKeyBytes;
  static constexpr int kSFK = kSFQ + kNQ * kSFAtoms * 512;
  static constexpr int kSFV = kSFK + kStages * kNKV * kSFAtoms * 512;
  static constexpr int kSFP = kSFV + kStages * kNKV * 512;
  static constexpr int kSFOnes = kSFP + 2 * 512;
  static constexpr int kBars = kSFOnes + 512;
  static constexpr int kNumBars = 1 + 2 * kStages + 10;  // q, kv full/empty, s_full/s_free/p_full/o_full/drain x2
  static constexpr int kMisc = kBars + kNumBars * 8;
  static constexpr int kBytes = kMisc + 16;
  // Pad the request so that one CTA owns the SM: it allocates all 512 TMEM columns.
  static constexpr int kAlloc = (kBytes + 1024 > 120 * 1024) ? kBytes + 1024 : 120 * 1024;
  static_assert(kStages >= 2, "the K/V ring needs at least two stages");
  static_assert(kTileQK % 1024 == 0 && kTileV % 1024 == 0 && kP % 1024 == 0, "tiles keep 1024-B alignment");
  static_assert(kAlloc <= 227 * 1024, "shared memory of one CTA");
  // ring buffers of stage s for slot t
  __host__ __device__ static constexpr int k_of(int s, int t) { return kK + (s * kNKV + (CH ? t : 0)) * kTileQK; }
  __host__ __device__ static constexpr int v_of(int s, int t) { return kV + (s * kNKV + (CH ? t : 0)) * kTileV; }
  __host__ __device__ static constexpr int sfk_of(int s, int t) { return kSFK + (s * kNKV + (CH ? t : 0)) * kSFAtoms * 512; }
  __host__ __device__ static constexpr int sfv_of(int s, int t) { return kSFV + (s * kNKV + (CH ? t : 0)) * 512; }
  // query tile u (0: first, 1: second of the chain) of slot t
  __host__ __device__ static constexpr int q_of(int t, int u) { return kQ + (CH ? 2 * t + u : t) * kTileQK; }
  __host__ __device__ static constexpr int sfq_of(int t, int u) { return kSFQ + (CH ? 2 * t + u : t) * kSFAtoms * 512; }
};

struct FwdParams {
  const uint8_t* q_sf;
  const uint8_t* k_sf;
  const uint8_t* v_sf;
  const float* g_q;
  const float* g_k;
  __nv_bfloat16* o;
  float* lse;
  DeviceStatus* status;
  int N;
  int ntiles;
  float softmax_scale;
  // debug dump of P (DUMP instantiation only)
  int dump_bh, dump_row0, dump_nrows;
  uint8_t* dump_codes;
  int32_t* dump_kshift;
  float* dump_o;  // fp32 O of the dumped rows, before the bf16 store
};

__device__ __forceinline__ float exp2_int(int e) {  // 2^e, e >= -149
  if (e >= -126) return __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
  if (e >= -149) return __uint_as_float(1u << (e + 149));
  return 0.0f;
}

template <int D, bool DUMP, bool CAUSAL, bool P8>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_directp_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  // Chained slots for the causal E2M1 forward; the causal FP8 P/V forward,
  // whose doubled K/V tiles would not leave room for a three-stage ring,
  // pairs query tiles c and T-1-c instead (one tile per slot).
  constexpr bool kChain = CAUSAL && !P8;
  using L = Layout<D, P8, kChain>;
  constexpr int kStages = L::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBars);
  uint64_t* bar_q_full = bars;
  uint64_t* bar_kv_full = bars + 1;
  uint64_t* bar_kv_empty = bars + 1 + kStages;
  uint64_t* bar_s_full = bars + 1 + 2 * kStages;  // [2]
  uint64_t* bar_s_free = bar_s_full + 2;          // [2]
  uint64_t* bar_p_full = bar_s_full + 4;          // [2]
  uint64_t* bar_o_full = bar_s_full + 6;          // [2]
  uint64_t* bar_drain = bar_s_full + 8;           // [2] the MMA warps' last commit
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.y;
  const int N = p.N;
  // The query tiles of the two slots.  Slot t runs the chain qa[t] (na[t]
  // key steps) then qb[t] (nb[t] steps, 0 when the chain has one tile); its
  // key steps are numbered k = 0 .. n_t-1 across the chain.  Slot 1 never
  // has fewer steps than slot 0.
  const int T = p.ntiles;
  int qa0, na0, qb0 = -1, nb0 = 0, qa1 = -1, na1 = 0, qb1 = -1, nb1 = 0;
  if (!CAUSAL) {
    qa0 = 2 * static_cast<int>(blockIdx.x);
    na0 = T;
    if ((qa0 + 1) * 128 < N) {
      qa1 = qa0 + 1;
      na1 = T;
    }
  } else if (!kChain) {
    // query tiles c (c+1 key tiles) and T-1-c (T-c); the second runs alone
    // once the first is done
    qa0 = static_cast<int>(blockIdx.x);
    na0 = qa0 + 1;
    if (T - 1 - qa0 > qa0) {
      qa1 = T - 1 - qa0;
      na1 = T - qa0;
    }
  } else {
    // chain i: query tiles i and T-1-i; for odd T the middle tile alone
    auto chain = [&](int i, int& qa, int& na, int& qb, int& nb) {
      qa = i;
      na = i + 1;
      if (i < T / 2) {
        qb = T - 1 - i;
        nb = T - i;
      }
    };
    const int nchains = (T + 1) / 2;
    chain(2 * static_cast<int>(blockIdx.x), qa0, na0, qb0, nb0);
    if (2 * static_cast<int>(blockIdx.x) + 1 < nchains) {
      chain(2 * static_cast<int>(blockIdx.x) + 1, qa1, na1, qb1, nb1);
      if (na1 + nb1 < na0 + nb0) {  // the middle tile's short chain goes to slot 0
        int x = qa0;
        qa0 = qa1;
        qa1 = x;
        x = na0;
        na0 = na1;
        na1 = x;
        x = qb0;
        qb0 = qb1;
        qb1 = x;
        x = nb0;
        nb0 = nb1;
        nb1 = x;
      }
    }
  }
  const bool has1 = na1 > 0;  // the second slot has work
  const int nkv0 = na0 + nb0, nkv1 = na1 + nb1;
  const int nkv = has1 ? nkv1 : nkv0;  // key steps streamed through the ring
  // key step k of slot t: query tile, key tile j within that query tile's
  // run, the run's length, and which tile of the chain it is
  struct StepOf {
    int qt, j, len, u;
  };
  auto step_of = [&](int t, int k) -> StepOf {
    if constexpr (!kChain) {
      return StepOf{t ? qa1 : qa0, k, t ? na1 : na0, 0};  // one query tile per slot
    } else {
      const int na = t ? na1 : na0;
      if (k < na) return StepOf{t ? qa1 : qa0, k, na, 0};
      return StepOf{t ? qb1 : qb0, k - na, t ? nb1 : nb0, 1};
    }
  };

  if (threadIdx.x == 0) {
    mbar_init(bar_q_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar_kv_full + s, 1);
      mbar_init(bar_kv_empty + s, has1 ? 2 : 1);  // one commit per MMA warp
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar_s_full + t, 1);
      mbar_init(bar_s_free + t, 4);  // one arrival per softmax warp
      mbar_init(bar_p_full + t, 4);
      mbar_init(bar_o_full + t, 1);
      mbar_init(bar_drain + t, 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  // constant operands of the denominator MMA: E2M1 ones (0x22 = two 1.0 codes)
  // and unit E8M0 scales (0x7F = 2^0)
  // (E4M3 ones are 0x38 bytes in the FP8 P/V variant)
  constexpr uint32_t kOnes4 = P8 ? 0x38383838u : 0x22222222u;
  for (int i = threadIdx.x; i < 16 * L::kKeyBytes / 16; i += kThreads)
    reinterpret_cast<uint4*>(smem + L::kOnes)[i] = make_uint4(kOnes4, kOnes4, kOnes4, kOnes4);
  for (int i = threadIdx.x; i < 512 / 16; i += kThreads)
    reinterpret_cast<uint4*>(smem + L::kSFOnes)[i] = make_uint4(0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
  fence_proxy_async_smem();
  if (warp == kWarpMma0) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // The only CTA on the SM holds all 512 columns, so its allocation starts at
  // lane 0, column 0.  Addressing TMEM from the constant 0 keeps every tcgen05
  // operand a compile-time or warp-uniform value; a different base (which the
  // allocation rules exclude) is reported and the CTA does nothing.
  const uint32_t tmem_base = *tmem_slot;
  constexpr uint32_t tmem = 0;
  if (tmem_base != 0) {
    if (threadIdx.x == 0 && atomicCAS(&p.status->timeout, 0u, 1u) == 0u) p.status->where = 99;
  } else if (warp == kWarpTma) {
    // ------------------------------------------------------------ TMA producer
    // The whole warp runs the loop and waits; one elected lane issues.
    const bool leader = elect_one();
    constexpr uint32_t kSfBytes = L::kSFAtoms * 512;
    if (leader) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      // every query tile of both slots, with its scale atoms
      int nq = has1 ? 2 : 1;
      if constexpr (kChain) {
        nq = 0;
        for (int t = 0; t < 2; ++t)
          for (int u = 0; u < 2; ++u) nq += ((u ? (t ? nb1 : nb0) : (t ? na1 : na0)) > 0) ? 1 : 0;
      }
      mbar_arrive_expect_tx(bar_q_full, nq * (L::kTileQK + kSfBytes));
      for (int t = 0; t < 2; ++t)
        for (int u = 0; u < 2; ++u) {
          if ((u ? (t ? nb1 : nb0) : (t ? na1 : na0)) == 0) continue;
          const int qt = u ? (t ? qb1 : qb0) : (t ? qa1 : qa0);
          tma_load_3d(smem + L::q_of(t, u), &tm_q, bar_q_full, 0, qt * 128, bh);
          bulk_load(smem + L::sfq_of(t, u), p.q_sf + (static_cast<size_t>(bh) * T + qt) * kSfBytes, kSfBytes,
                    bar_q_full);
        }
    }
    int issued = 0;  // key steps whose copies were issued
    for (int k = 0; k < nkv; ++k) {
      const int s = k % kStages;
      if (k >= kStages) {
        const bool ok = mbar_wait(bar_kv_empty + s, ((k / kStages) - 1) & 1, abort_flag, p.status, 1);
        if (!__all_sync(0xFFFFFFFFu, ok)) break;
      }
      if (leader) {
        // the key tile of each slot that takes step k (chained slots: one
        // each; otherwise the slots share one)
        if constexpr (!kChain) {
          mbar_arrive_expect_tx(bar_kv_full + s, L::kTileQK + L::kTileV + kSfBytes + 512);
          tma_load_3d(smem + L::kK + s * L::kTileQK, &tm_k, bar_kv_full + s, 0, k * 128, bh);
          tma_load_2d(smem + L::kV + s * L::kTileV, &tm_v, bar_kv_full + s, k * L::kKeyBytes, bh * D);
          bulk_load(smem + L::kSFK + s * kSfBytes, p.k_sf + (static_cast<size_t>(bh) * T + k) * kSfBytes, kSfBytes,
                    bar_kv_full + s);
          bulk_load(smem + L::kSFV + s * 512, p.v_sf + (static_cast<size_t>(bh) * T + k) * 512, 512, bar_kv_full + s);
        }
        const int nslots = kChain ? ((k < nkv0 ? 1 : 0) + (has1 && k < nkv1 ? 1 : 0)) : 1;
        if (kChain) mbar_arrive_expect_tx(bar_kv_full + s, nslots * (L::kTileQK + L::kTileV + kSfBytes + 512));
        for (int t = 0; t < (kChain ? 2 : 0); ++t) {
          if (kChain && k >= (t ? (has1 ? nkv1 : 0) : nkv0)) continue;
          const int j = kChain ? step_of(t, k).j : k;
          tma_load_3d(smem + L::k_of(s, t), &tm_k, bar_kv_full + s, 0, j * 128, bh);
          tma_load_2d(smem + L::v_of(s, t), &tm_v, bar_kv_full + s, j * L::kKeyBytes, bh * D);
          bulk_load(smem + L::sfk_of(s, t), p.k_sf + (static_cast<size_t>(bh) * T + j) * kSfBytes, kSfBytes,
                    bar_kv_full + s);
          bulk_load(smem + L::sfv_of(s, t), p.v_sf + (static_cast<size_t>(bh) * T + j) * 512, 512,
                    bar_kv_full + s);
        }
      }
      issued = k + 1;
      __syncwarp();
    }
    // Before leaving, make sure no copy into this CTA's shared memory is
    // still in flight, even when the CTA is giving up: wait for the last
    // issued fill of every stage.
    for (int k = issued - kStages < 0 ? 0 : issued - kStages; k < issued; ++k)
      mbar_wait_drain(bar_kv_full + (k % kStages), (k / kStages) & 1, abort_flag, p.status, 2);
    mbar_wait_drain(bar_q_full, 0, abort_flag, p.status, 3);
  } else if (warp == kWarpMma0 || (warp == kWarpMma0 + 1 && has1)) {
    // ------------------------------------------------------------ MMA issuers
    // Warp 9 + t issues everything of query tile t.  The whole warp runs the
    // loop, waits and evaluates every operand (so they stay warp-uniform); one
    // elected lane issues each tcgen05 operation.
    const int t = warp - kWarpMma0;
    const int nkv_t = t ? nkv1 : nkv0;
    constexpr uint32_t kSwizzleQK = (D == 128) ? 4u : 6u;  // 64-B or 32-B rows
    constexpr uint32_t kSbo = 8 * L::kRowBytes;
    constexpr uint32_t idesc_qk = idesc_fp4_block_scaled(128, 128, 0, 0, 0);
    constexpr uint32_t idesc_pv0 = idesc_fp4_block_scaled(128, D, 1, 0, 0);
    constexpr uint32_t idesc_pv1 = idesc_fp4_block_scaled(128, D, 1, 2, 2);
    constexpr uint32_t idesc_l0 = idesc_fp4_block_scaled(128, kLN, 1, 0, 0);
    constexpr uint32_t idesc_l1 = idesc_fp4_block_scaled(128, kLN, 1, 2, 2);
    // P, V^T and the ones tile: K-major rows of 64 bytes (E2M1, 64-byte
    // swizzle) or 128 bytes (E4M3, 128-byte swizzle); 8-row groups apart by SBO.
    constexpr uint32_t kSwizzleKV = P8 ? 2u : 4u;
    constexpr uint32_t kSboKV = 8 * L::kKeyBytes;
    // Descriptors are built once; the start-address field is linear in the
    // shared-memory address (16-byte units), so tiles are reached by adding
    // their offset.
    const uint64_t qdesc_a = smem_desc(smem_u32(smem + L::q_of(t, 0)), 16, kSbo, kSwizzleQK);
    const uint64_t qdesc_b = smem_desc(smem_u32(smem + L::q_of(t, 1)), 16, kSbo, kSwizzleQK);
    const uint64_t kdesc0 = smem_desc(smem_u32(smem + L::k_of(0, t)), 16, kSbo, kSwizzleQK);
    const uint64_t vdesc0 = smem_desc(smem_u32(smem + L::v_of(0, t)), 16, kSboKV, kSwizzleKV);
    const uint64_t pdesc = smem_desc(smem_u32(smem + L::kP + t * L::kTileP), 16, kSboKV, kSwizzleKV);
    const uint64_t ones_desc = smem_desc(smem_u32(smem + L::kOnes), 16, kSboKV, kSwizzleKV);
    // ring stages are kNKV tiles apart
    constexpr uint64_t kQKStep = (L::kNKV * L::kTileQK) >> 4, kVStep = (L::kNKV * L::kTileV) >> 4;
    const uint32_t t_s = tmem + kColS;
    const uint32_t t_o = tmem + kColO + t * D;
    const uint32_t t_l = tmem + kColL + 16 * t;
    const uint32_t t_sfq = tmem + kColSFQ + 8 * t;
    const uint32_t t_sfk = tmem + kColSFK + 16 * t;
    const uint32_t t_sfv = tmem + kColSFV + 8 * t;
    const uint32_t t_sfp = tmem + kColSFP + 4 * t;
    const uint32_t t_sf1 = tmem + kColSFOnes + 4 * t;
    uint64_t* s_full = bar_s_full + t;
    uint64_t* p_full = bar_p_full + t;
    uint64_t* o_full = bar_o_full + t;
    auto wait = [&](uint64_t* bar, uint32_t parity, unsigned site) {
      return __all_sync(0xFFFFFFFFu, mbar_wait(bar, parity, abort_flag, p.status, site));
    };
    // The score bank is free for S_t(j) once the other tile has pulled its
    // previous S into registers (tile 0, step j: tile 1's step j-1; tile 1,
    // step j: tile 0's step j); without a second tile -- or, causal, once
    // tile 0 has run out of key tiles -- once this tile has pulled its own
    // previous S.
    auto bank_free = [&](int j) {  // before S_t(j); j >= 1 for tile 0
      if (t == 1) {
        if (j < nkv0) return wait(bar_s_free, j & 1, 12);
        return wait(bar_s_free + 1, (j - 1) & 1, 16);
      }
      return wait(bar_s_free + (has1 ? 1 : 0), (j - 1) & 1, 13);
    };
    // The whole warp runs each issue; one elected lane issues (inside the asm).
    const uint32_t sfk_src = smem_u32(smem + L::sfk_of(0, t)), sfv_src = smem_u32(smem + L::sfv_of(0, t));
    const uint32_t sfp_src = smem_u32(smem + L::kSFP + t * 512);
    constexpr uint32_t kSfkStep = L::kNKV * L::kSFAtoms * 512, kSfvStep = L::kNKV * 512;
    auto issue_qk = [&](int k) {  // K scale atoms of step k, then S = Q K(j)^T for the step's query tile
      const int s = k % kStages;
      const StepOf st = step_of(t, k);
      if (kChain && k > 0 && st.j == 0) {
        // the chain moves on to its second query tile: its Q scale atoms
        // replace the first tile's (after that tile's products, in issue order)
        for (int a = 0; a < L::kSFAtoms; ++a)
          tc_cp_sf_atom_warp(t_sfq + 4 * a, smem_u32(smem + L::sfq_of(t, 1) + a * 512));
      }
      const uint64_t qdesc = st.u ? qdesc_b : qdesc_a;
      const uint32_t sfk = t_sfk + 8 * (k & 1);
#pragma unroll
      for (int a = 0; a < L::kSFAtoms; ++a) tc_cp_sf_atom_warp(sfk + 4 * a, sfk_src + s * kSfkStep + a * 512);
#pragma unroll
      for (int ks = 0; ks < D / 64; ++ks)
        mma_nvf4_warp(t_s, qdesc + 2 * ks, kdesc0 + s * kQKStep + 2 * ks, idesc_qk, t_sfq + 4 * ks, sfk + 4 * ks,
                      ks > 0);
      tc_commit_warp(s_full);
    };
    auto issue_pv = [&](int k) {  // P and V scale atoms, O_t += P_t V(j), l_t = P_t 1
      const int s = k % kStages;
      const int j = step_of(t, k).j;  // 0: the first product of a query tile overwrites O
      const uint32_t sfv = t_sfv + 4 * (k & 1);
      const uint64_t vd = vdesc0 + s * kVStep;
      tc_cp_sf_atom_warp(t_sfp, sfp_src);
      tc_cp_sf_atom_warp(sfv, sfv_src + s * kSfvStep);
      if constexpr (P8) {
        // E4M3 operands: four K = 32 products per 128 keys, each with the
        // scale byte k of its 32-key block (one scale per row and block)
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_mxf8_warp(t_o, pdesc + 2 * k, vd + 2 * k, idesc_mxf8_block_scaled(128, D, k, k), t_sfp, sfv,
                        j > 0 || k > 0);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_mxf8_warp(t_l, pdesc + 2 * k, ones_desc + 2 * k, idesc_mxf8_block_scaled(128, kLN, k, k), t_sfp,
                        t_sf1, k > 0);
      } else {
        mma_mxf4_warp(t_o, pdesc, vd, idesc_pv0, t_sfp, sfv, j > 0);
        mma_mxf4_warp(t_o, pdesc + 2, vd + 2, idesc_pv1, t_sfp, sfv, true);
        mma_mxf4_warp(t_l, pdesc, ones_desc, idesc_l0, t_sfp, t_sf1, false);
        mma_mxf4_warp(t_l, pdesc + 2, ones_desc + 2, idesc_l1, t_sfp, t_sf1, true);
      }
      tc_commit_warp(o_full);
      tc_commit_warp(bar_kv_empty + s);
      // a stage that slot 0 does not consume still needs both releases
      if (t == 1 && k >= nkv0) tc_commit_warp(bar_kv_empty + s);
    };

    bool ok = wait(bar_q_full, 0, 10);
    if (ok) {
      tc_fence_after();
      for (int a = 0; a < L::kSFAtoms; ++a)
        tc_cp_sf_atom_warp(t_sfq + 4 * a, smem_u32(smem + L::sfq_of(t, 0) + a * 512));
      tc_cp_sf_atom_warp(t_sf1, smem_u32(smem + L::kSFOnes));
      ok = wait(bar_kv_full, 0, 11);
    }
    if (ok && t == 1) ok = wait(bar_s_free, 0, 12);  // tile 0 has pulled S_0(0)
    if (ok) {
      tc_fence_after();
      issue_qk(0);
    }
    // Per key step k: the next scores first (they need only the next key
    // tile and the bank), then this slot's PV product of step k.
    for (int k = 0; ok && k < nkv_t; ++k) {
      if (k + 1 < nkv_t) {
        if (!(ok = wait(bar_kv_full + (k + 1) % kStages, ((k + 1) / kStages) & 1, 14))) break;
        if (!(ok = bank_free(k + 1))) break;
        tc_fence_after();
        issue_qk(k + 1);
      }
      if (!(ok = wait(p_full, k & 1, 15))) break;
      tc_fence_after();
      issue_pv(k);
    }
    // Every MMA and scale copy this warp issued must have completed before
    // TMEM is freed, even when the CTA is giving up.
    tc_commit_warp(bar_drain + t);
    mbar_wait_drain(bar_drain + t, 0, abort_flag, p.status, 17);
  } else if (warp < 8 && (warp < 4 || has1)) {
    // ------------------------------------------------------------ softmax rows
    const int t = warp >> 2;            // slot of this warpgroup
    const int row = threadIdx.x & 127;  // == TMEM lane
    const int nkv_t = t ? nkv1 : nkv0;
    int qrow = (t ? qa1 : qa0) * 128 + row;  // query row of the current tile
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base + kColS;
    const uint32_t tO = tmem + lane_base + kColO + t * D;
    const uint32_t tL = tmem + lane_base + kColL + 16 * t;
    uint64_t* s_full = bar_s_full + t;
    uint64_t* s_free = bar_s_free + t;
    uint64_t* p_full = bar_p_full + t;
    uint64_t* o_full = bar_o_full + t;
    uint8_t* sP = smem + L::kP + t * L::kTileP;
    uint8_t* sSFP = smem + L::kSFP + t * 512;
    const float c = static_cast<float>(((static_cast<double>(p.softmax_scale) * kLog2E) *
                                        static_cast<double>(*p.g_q)) * static_cast<double>(*p.g_k));
    auto is_dump_row = [&](int qr) {
      return DUMP && bh == p.dump_bh && qr >= p.dump_row0 && qr < p.dump_row0 + p.dump_nrows;
    };
    // O / l of the current query tile's row -> bf16 O and the LSE (the whole
    // warp reads the output bank: tcgen05.ld is warp-collective)
    auto write_out = [&](int qr, int m_e, float l_e) {
      const float inv_l = 1.0f / l_e;
      const bool store = qr < N;
      const bool dump = is_dump_row(qr);
      __nv_bfloat16* orow = p.o + (static_cast<size_t>(bh) * N + (store ? qr : 0)) * D;
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        float o[32];
        tmem_ld32(tO + 32 * cc, o);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) o[i] *= inv_l;
        if (store) {
          uint32_t packed[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            __nv_bfloat162 h2 = __floats2bfloat162_rn(o[2 * i], o[2 * i + 1]);
            packed[i] = *reinterpret_cast<uint32_t*>(&h2);
          }
          uint4* dst = reinterpret_cast<uint4*>(orow + 32 * cc);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            dst[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
        }
        if (dump) {
          float* od = p.dump_o + static_cast<size_t>(qr - p.dump_row0) * D + 32 * cc;
#pragma unroll
          for (int i = 0; i < 32; ++i) od[i] = o[i];
        }
      }
      if (store) p.lse[static_cast<size_t>(bh) * N + qr] = 0.69314718055994531f * (static_cast<float>(m_e) + log2f(l_e));
    };
    int m_ref = 0;
    float l_run = 0.0f;  // denominator, relative to 2^m_ref
    bool ok = true;
    // tcgen05.ld / tcgen05.st are warp-collective (.sync.aligned): every
    // branch around them below is made warp-uniform with a vote.
    for (int k = 0; k < nkv_t; ++k) {
      const StepOf st = step_of(t, k);
      const int j = st.j;             // key tile within the current query tile's run
      const int qrow_prev = qrow;     // the previous query tile's row, at a switch
      if (kChain) qrow = st.qt * 128 + row;
      const bool dump_row = is_dump_row(qrow);
      ok = mbar_wait(s_full, k & 1, abort_flag, p.status, 20);
      if (!__all_sync(0xFFFFFFFFu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // S row and its 32-key block maxima, reduced while leaving TMEM; the
      // bank goes back to the MMA warps as soon as the row is in registers.
      float s[128];
      float bm[4];
      bm[0] = tmem_ld32_max(tS + 0, *reinterpret_cast<float(*)[32]>(s + 0));
      bm[1] = tmem_ld32_max(tS + 32, *reinterpret_cast<float(*)[32]>(s + 32));
      bm[2] = tmem_ld32_max(tS + 64, *reinterpret_cast<float(*)[32]>(s + 64));
      bm[3] = tmem_ld32_max(tS + 96, *reinterpret_cast<float(*)[32]>(s + 96));
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_free);

      int valid = N - j * 128;  // keys of this tile that exist (>= 1)
      // causal: on the diagonal tile (the last one) row r sees keys 0 .. r
      if (CAUSAL && j == st.len - 1) valid = min(valid, row + 1);
      if (valid < 128) {
        // partial tile: keys past N (or past the diagonal) are masked and the
        // maxima retaken
#pragma unroll
        for (int i = 0; i < 128; ++i)
          if (i >= valid) s[i] = -INFINITY;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
          float m = fmax3(s[32 * b], s[32 * b + 1], s[32 * b + 2]);
#pragma unroll
          for (int i = 3; i < 31; i += 2) m = fmax3(m, s[32 * b + i], s[32 * b + i + 1]);
          bm[b] = fmaxf(m, s[32 * b + 31]);
        }
      }
      // block maxima of the scaled scores (c > 0, so max(c*s) = c*max(s))
      float xb[4];
      int kb[4];
      float xmax = -INFINITY;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        xb[b] = __fmul_rn(c, bm[b]);
        xmax = fmaxf(xmax, xb[b]);
        kb[b] = (xb[b] == -INFINITY) ? 0 : static_cast<int>(ceilf(__fsub_rn(xb[b], P8 ? kLog2_448 : kLog2Six)));
      }
      const int m_tile = static_cast<int>(ceilf(xmax));
      const int m_old = m_ref;  // also the previous query tile's reference at a switch
      bool rescale = false;
      if (j == 0) {
        m_ref = m_tile;
      } else if (m_tile > m_ref + kRescaleSlack) {
        m_ref = m_tile;
        rescale = true;
      }
      // Direct-P: codes of 2^(X - K_b) = 2^(c*s - K_b), eight E2M1 or four
      // E4M3 codes per word
      constexpr int kWords = L::kKeyBytes / 4;
      uint32_t w[kWords];
      uint32_t sfword = 0;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const float nk = static_cast<float>(-kb[b]);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float* sv = s + 32 * b + 8 * q;
          float x[8];
#pragma unroll
          for (int i = 0; i < 8; i += 2) ffma2(x[i], x[i + 1], c, c, sv[i], sv[i + 1], nk, nk);
#pragma unroll
          for (int i = 0; i < 8; ++i) x[i] = ex2_approx(x[i]);
          if constexpr (P8) {
            w[8 * b + 2 * q] = cvt_e4m3x4(x[0], x[1], x[2], x[3]);
            w[8 * b + 2 * q + 1] = cvt_e4m3x4(x[4], x[5], x[6], x[7]);
          } else {
            w[4 * b + q] = cvt_e2m1x8(x[0], x[1], x[2], x[3], x[4], x[5], x[6], x[7]);
          }
        }
        int e = kb[b] - m_ref;
        e = e < -127 ? -127 : e;
        const uint32_t byte = (xb[b] == -INFINITY) ? 0u : static_cast<uint32_t>(e + 127);
        sfword |= byte << (8 * b);
      }
      // The previous PV product must be done before this tile's P buffer and
      // the O / l banks are touched; it normally finished long ago.  Its tile
      // denominator (relative to the reference it was made with) joins l.
      float l_prev = 0.0f;
      if (k > 0) {
        ok = mbar_wait(o_full, (k - 1) & 1, abort_flag, p.status, 21);
        if (!__all_sync(0xFFFFFFFFu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        l_prev = tmem_ld1(tL);  // completes at a wait below
        if (kChain && j == 0) {
          // the chain has moved on to its second query tile: the first one's
          // products are all complete -- write its O and LSE out before this
          // step's PV product overwrites the output bank
          tmem_wait_ld();
          write_out(qrow_prev, m_old, l_run + l_prev);
          l_run = 0.0f;
          l_prev = 0.0f;
        }
      }
      // Rescale O of the rows whose reference maximum moved; the whole warp
      // takes part in the TMEM round trip, other rows multiply by 1.
      if (__any_sync(0xFFFFFFFFu, rescale)) {
        tmem_wait_ld();
        l_run += l_prev;
        l_prev = 0.0f;
        const float f = rescale ? exp2_int(m_old - m_ref) : 1.0f;
        l_run *= f;
#pragma unroll
        for (int cc = 0; cc < D / 32; ++cc) {
          float o[32];
          tmem_ld32(tO + 32 * cc, o);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= f;
          tmem_st32(tO + 32 * cc, o);
        }
        tmem_wait_st();
      }
      const uint32_t prow = smem_u32(sP + row * L::kKeyBytes);
#pragma unroll
      for (int u = 0; u < kWords / 4; ++u) {
        // 64-byte (E2M1) or 128-byte (E4M3) swizzle of the K-major P tile
        const int chunk = P8 ? (u ^ (row & 7)) : (u ^ ((row >> 1) & 3));
        sts_u4(prow + chunk * 16, w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
      }
      asm volatile("st.shared.u32 [%0], %1;" ::"r"(smem_u32(sSFP + (row & 31) * 16 + (row >> 5) * 4)), "r"(sfword) : "memory");
      if (dump_row) {
        const size_t rr = static_cast<size_t>(qrow - p.dump_row0);
        uint4* dst = reinterpret_cast<uint4*>(p.dump_codes + rr * (T * L::kKeyBytes) + j * L::kKeyBytes);
#pragma unroll
        for (int u = 0; u < kWords / 4; ++u) dst[u] = make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
#pragma unroll
        for (int b = 0; b < 4; ++b) p.dump_kshift[rr * (T * 4) + j * 4 + b] = kb[b];
      }
      tmem_wait_ld();
      l_run += l_prev;
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
    }
    // ------------------------------------------------------------ epilogue
    if (ok) ok = mbar_wait(o_full, (nkv_t - 1) & 1, abort_flag, p.status, 22);
    if (__all_sync(0xFFFFFFFFu, ok)) {
      tc_fence_after();
      const float l = l_run + tmem_ld1(tL);
      tmem_wait_ld();
      write_out(qrow, m_ref, l);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpMma0) {
    __syncwarp();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

bool make_map(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
              const cuuint32_t* box, CUtensorMapSwizzle swz) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, rank, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// v: the V payload and scale atoms -- MXFP4 (E2M1) or, with P8, MXFP8 (E4M3)
// V^T with one byte per key; both use the same atom layout.
// status: the word the kernel's bounded waits report into -- the library's
// per-device status block, or the allocation-free entry point's static word;
// it is never created here.
template <int D, bool DUMP, bool CAUSAL = false, bool P8 = false>
int launch(const fp4attn_nvfp4_t* q, const fp4attn_nvfp4_t* k, const fp4attn_mxfp4_t* v, void* o, float* lse,
           int B, int H, int N, float softmax_scale, int dump_bh, int row0, int nrows, uint8_t* codes,
           int32_t* kshift, float* o_f32, cudaStream_t stream, DeviceStatus* status) {
  using L = Layout<D, P8, CAUSAL && !P8>;
  if (!status) return FP4ATTN_ERR_CUDA;
  const int ntiles = n_row_tiles(N);
  const int BH = B * H;
  CUtensorMap tq, tk, tv;
  const CUtensorMapSwizzle swz_qk = (D == 128) ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B;
  const cuuint64_t qk_dims[3] = {static_cast<cuuint64_t>(D / 2), static_cast<cuuint64_t>(N),
                                 static_cast<cuuint64_t>(BH)};
  const cuuint64_t qk_strides[2] = {static_cast<cuuint64_t>(D / 2), static_cast<cuuint64_t>(N) * (D / 2)};
  const cuuint32_t qk_box[3] = {static_cast<cuuint32_t>(D / 2), 128, 1};
  const cuuint64_t v_dims[2] = {static_cast<cuuint64_t>(ntiles) * L::kKeyBytes, static_cast<cuuint64_t>(BH) * D};
  const cuuint64_t v_strides[1] = {static_cast<cuuint64_t>(ntiles) * L::kKeyBytes};
  const cuuint32_t v_box[2] = {static_cast<cuuint32_t>(L::kKeyBytes), static_cast<cuuint32_t>(D)};
  const CUtensorMapSwizzle swz_v = P8 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  if (!make_map(&tq, q->payload, 3, qk_dims, qk_strides, qk_box, swz_qk) ||
      !make_map(&tk, k->payload, 3, qk_dims, qk_strides, qk_box, swz_qk) ||
      !make_map(&tv, v->payload_t, 2, v_dims, v_strides, v_box, swz_v))
    return FP4ATTN_ERR_CUDA;
  FwdParams prm{};
  prm.q_sf = q->sf;
  prm.k_sf = k->sf;
  prm.v_sf = v->sf;
  prm.g_q = q->g;
  prm.g_k = k->g;
  prm.o = static_cast<__nv_bfloat16*>(o);
  prm.lse = lse;
  prm.status = status;
  prm.N = N;
  prm.ntiles = ntiles;
  prm.softmax_scale = softmax_scale;
  prm.dump_bh = dump_bh;
  prm.dump_row0 = row0;
  prm.dump_nrows = nrows;
  prm.dump_codes = codes;
  prm.dump_kshift = kshift;
  prm.dump_o = o_f32;
  auto kern = fwd_directp_kernel<D, DUMP, CAUSAL, P8>;
  static std::once_flag attr_once[64];
  int dev = 0;
  cudaGetDevice(&dev);
  cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once[dev & 63], [&] {
    attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  });
  if (attr_err != cudaSuccess) return FP4ATTN_ERR_CUDA;
  // two query tiles per CTA: (2c, 2c+1); causal E2M1: two chains of two
  // query tiles (the middle tile of an odd count alone); causal FP8 P/V:
  // (c, ntiles-1-c)
  const int nchains = (ntiles + 1) / 2;
  dim3 grid((CAUSAL && !P8) ? (nchains + 1) / 2 : (ntiles + 1) / 2, BH);
  kern<<<grid, kThreads, L::kAlloc, stream>>>(tq, tk, tv, prm);
  return cuda_status(cudaGetLastError());
}

int check_fwd(const fp4attn_nvfp4_t* q, const fp4attn_nvfp4_t* k, const fp4attn_mxfp4_t* v, void* o, float* lse,
              int B, int H, int N, int D, float softmax_scale) {
  const int st = check_shape(B, H, N, D);
  if (st != FP4ATTN_OK) return st;
  if (!q || !k || !v || !o || !lse) return FP4ATTN_ERR_INVALID_ARG;
  if (!q->payload || !q->sf || !q->g || !k->payload || !k->sf || !k->g || !v->payload_t || !v->sf)
    return FP4ATTN_ERR_INVALID_ARG;
  if (!aligned16(q->payload) || !aligned16(q->sf) || !aligned16(k->payload) || !aligned16(k->sf) ||
      !aligned16(v->payload_t) || !aligned16(v->sf) || !aligned16(o) || !aligned16(lse))
    return FP4ATTN_ERR_INVALID_ARG;
  if (!(softmax_scale > 0.0f) || !std::isfinite(softmax_scale)) return FP4ATTN_ERR_INVALID_ARG;
  return FP4ATTN_OK;
}

}  // namespace
}  // namespace fp4attn

using namespace fp4attn;

extern "C" int fp4attn_fwd_directp(const fp4attn_nvfp4_t* q, const fp4attn_nvfp4_t* k, const fp4attn_mxfp4_t* v,
                                   void* o, float* lse, int B, int H, int N, int D, float softmax_scale,
                                   void* stream) {
  const int st = check_fwd(q, k, v, o, lse, B, H, N, D, softmax_scale);
  if (st != FP4ATTN_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (D == 128) return launch<128, false>(q, k, v, o, lse, B, H, N, softmax_scale, -1, 0, 0, nullptr, nullptr, nullptr, s, device_status_ptr());
  return launch<64, false>(q, k, v, o, lse, B, H, N, softmax_scale, -1, 0, 0, nullptr, nullptr, nullptr, s, device_status_ptr());
}

extern "C" int fp4attn_debug_dump_p(const fp4attn_nvfp4_t* q, const fp4attn_nvfp4_t* k, const fp4attn_mxfp4_t* v,
                                    void* o, float* lse, int B, int H, int N, int D, float softmax_scale, int b,
                                    int h, int row0, int nrows, uint8_t* codes, int32_t* kshift, float* o_f32,
                                    void* stream) {
  const int st = check_fwd(q, k, v, o, lse, B, H, N, D, softmax_scale);
  if (st != FP4ATTN_OK) return st;
  if (b < 0 || b >= B || h < 0 || h >= H || row0 < 0 || nrows <= 0 || row0 + nrows > N || !codes || !kshift ||
      !o_f32 || !aligned16(codes) || !aligned16(kshift) || !aligned16(o_f32))
    return FP4ATTN_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int bh = b * H + h;
  if (D == 128) return launch<128, true>(q, k, v, o, lse, B, H, N, softmax_scale, bh, row0, nrows, codes, kshift, o_f32, s, device_status_ptr());
  return launch<64, true>(q, k, v, o, lse, B, H, N, softmax_scale, bh, row0, nrows, codes, kshift, o_f32, s, device_status_ptr());
}

extern "C" int fp4attn_fwd_directp_causal(const fp4attn_nvfp4_t* q, const fp4attn_nvfp4_t* k,
                                          const fp4attn_mxfp4_t* v, void* o, float* lse, int B, int H, int N, int D,
                                          float softmax_scale, void* stream) {
  const int st = check_fwd(q, k, v, o, lse, B, H, N, D, softmax_scale);
  if (st != FP4ATTN_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (D == 128)
    return launch<128, false, true>(q, k, v, o, lse, B, H, N, softmax_scale, -1, 0, 0, nullptr, nullptr, nullptr, s, device_status_ptr());
  return launch<64, false, true>(q, k, v, o, lse, B, H, N, softmax_scale, -1, 0, 0, nullptr, nullptr, nullptr, s, device_status_ptr());
}

extern "C" int fp4attn_debug_dump_p_causal(const fp4attn_nvfp4_t* q, const fp4attn_nvfp4_t* k,
                                           const fp4attn_mxfp4_t* v, void* o, float* lse, int B, int H, int N, int D,
                                           float softmax_scale, int b, int h, int row0, int nrows, uint8_t* codes,
                                           int32_t* kshift, float* o_f32, void* stream) {
  const int st = check_fwd(q, k, v, o, lse, B, H, N, D, softmax_scale);
  if (st != FP4ATTN_OK) return st;
  if (b < 0 || b >= B || h < 0 || h >= H || row0 < 0 || nrows <= 0 || row0 + nrows > N || !codes || !kshift ||
      !o_f32 || !aligned16(codes) || !aligned16(kshift) || !aligned16(o_f32))
    return FP4ATTN_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // key tiles past a row's diagonal are never visited: their codes and
  // shifts read as zero
  const size_t npad = static_cast<size_t>(n_row_tiles(N)) * 128;
  if (cudaMemsetAsync(codes, 0, static_cast<size_t>(nrows) * (npad / 2), s) != cudaSuccess ||
      cudaMemsetAsync(kshift, 0, static_cast<size_t>(nrows) * (npad / 32) * sizeof(int32_t), s) != cudaSuccess)
    return FP4ATTN_ERR_CUDA;
  const int bh = b * H + h;
  if (D == 128)
    return launch<128, true, true>(q, k, v, o, lse, B, H, N, softmax_scale, bh, row0, nrows, codes, kshift, o_f32, s, device_status_ptr());
  return launch<64, true, true>(q, k, v, o, lse, B, H, N, softmax_scale, bh, row0, nrows, codes, kshift, o_f32, s, device_status_ptr());
}

extern "C" int fp4attn_fwd_directp_causal_save(const void* q, const void* k, const void* v,
                                               const fp4attn_nvfp4_buf_t* q_saved,
                                               const fp4attn_nvfp4_buf_t* k_saved,
                                               const fp4attn_mxfp4_buf_t* v_quant, void* o, float* lse, int B,
                                               int H, int N, int D, float softmax_scale, void* stream) {
  if (!q || !k || !v || !q_saved || !k_saved || !v_quant) return FP4ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v)) return FP4ATTN_ERR_INVALID_ARG;
  const fp4attn_nvfp4_t qn{q_saved->payload, q_saved->sf, q_saved->g};
  const fp4attn_nvfp4_t kn{k_saved->payload, k_saved->sf, k_saved->g};
  const fp4attn_mxfp4_t vm{v_quant->payload_t, v_quant->sf};
  // every argument is checked before anything is launched
  const int st = check_fwd(&qn, &kn, &vm, o, lse, B, H, N, D, softmax_scale);
  if (st != FP4ATTN_OK) return st;
  int r = fp4attn_quant_qk_nvfp4(q, q_saved->payload, q_saved->sf, q_saved->g, B, H, N, D, stream);
  if (r == FP4ATTN_OK) r = fp4attn_quant_qk_nvfp4(k, k_saved->payload, k_saved->sf, k_saved->g, B, H, N, D, stream);
  if (r == FP4ATTN_OK) r = fp4attn_quant_v_mxfp4(v, v_quant->payload_t, v_quant->sf, B, H, N, D, stream);
  if (r == FP4ATTN_OK) r = fp4attn_fwd_directp_causal(&qn, &kn, &vm, o, lse, B, H, N, D, softmax_scale, stream);
  return r;
}

extern "C" int fp4attn_fwd_directp_fp8pv(const fp4attn_nvfp4_t* q, const fp4attn_nvfp4_t* k,
                                         const fp4attn_mxfp8_t* v, void* o, float* lse, int B, int H, int N, int D,
                                         float softmax_scale, int causal, void* stream) {
  if (!v) return FP4ATTN_ERR_INVALID_ARG;
  const fp4attn_mxfp4_t vv{v->payload_t, v->sf};  // same two pointers; one byte per key
  const int st = check_fwd(q, k, &vv, o, lse, B, H, N, D, softmax_scale);
  if (st != FP4ATTN_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (D == 128)
    return causal ? launch<128, false, true, true>(q, k, &vv, o, lse, B, H, N, softmax_scale, -1, 0, 0, nullptr,
                                                   nullptr, nullptr, s, device_status_ptr())
                  : launch<128, false, false, true>(q, k, &vv, o, lse, B, H, N, softmax_scale, -1, 0, 0, nullptr,
                                                    nullptr, nullptr, s, device_status_ptr());
  return causal ? launch<64, false, true, true>(q, k, &vv, o, lse, B, H, N, softmax_scale, -1, 0, 0, nullptr,
                                                nullptr, nullptr, s, device_status_ptr())
                : launch<64, false, false, true>(q, k, &vv, o, lse, B, H, N, softmax_scale, -1, 0, 0, nullptr,
                                                 nullptr, nullptr, s, device_status_ptr());
}

extern "C" int fp4attn_debug_dump_p_fp8pv(const fp4attn_nvfp4_t* q, const fp4attn_nvfp4_t* k,
                                          const fp4attn_mxfp8_t* v, void* o, float* lse, int B, int H, int N, int D,
                                          float softmax_scale, int causal, int b, int h, int row0, int nrows,
                                          uint8_t* codes, int32_t* kshift, float* o_f32, void* stream) {
  if (!v) return FP4ATTN_ERR_INVALID_ARG;
  const fp4attn_mxfp4_t vv{v->payload_t, v->sf};
  const int st = check_fwd(q, k, &vv, o, lse, B, H, N, D, softmax_scale);
  if (st != FP4ATTN_OK) return st;
  if (b < 0 || b >= B || h < 0 || h >= H || row0 < 0 || nrows <= 0 || row0 + nrows > N || !codes || !kshift ||
      !o_f32 || !aligned16(codes) || !aligned16(kshift) || !aligned16(o_f32))
    return FP4ATTN_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // key tiles past a row's diagonal (causal) are never visited: their codes
  // and shifts read as zero
  const size_t npad = static_cast<size_t>(n_row_tiles(N)) * 128;
  if (cudaMemsetAsync(codes, 0, static_cast<size_t>(nrows) * npad, s) != cudaSuccess ||
      cudaMemsetAsync(kshift, 0, static_cast<size_t>(nrows) * (npad / 32) * sizeof(int32_t), s) != cudaSuccess)
    return FP4ATTN_ERR_CUDA;
  const int bh = b * H + h;
  if (D == 128)
    return causal ? launch<128, true, true, true>(q, k, &vv, o, lse, B, H, N, softmax_scale, bh, row0, nrows, codes,
                                                  kshift, o_f32, s, device_status_ptr())
                  : launch<128, true, false, true>(q, k, &vv, o, lse, B, H, N, softmax_scale, bh, row0, nrows,
                                                   codes, kshift, o_f32, s, device_status_ptr());
  return causal ? launch<64, true, true, true>(q, k, &vv, o, lse, B, H, N, softmax_scale, bh, row0, nrows, codes,
                                               kshift, o_f32, s, device_status_ptr())
                : launch<64, true, false, true>(q, k, &vv, o, lse, B, H, N, softmax_scale, bh, row0, nrows, codes,
                                                kshift, o_f32, s, device_status_ptr());
}

// ------------------------------------------------------------------ allocation-free variant
// fp4attn_fwd_directp_noalloc runs the same kernel, but the one piece of
// memory the forward uses beyond its inputs and outputs -- the status word its
// bounded waits report into, normally a block the library cudaMallocs on the
// first call on each device -- lives in the static device array below, which
// exists on every GPU that loads the library for as long as the process runs.
namespace fp4attn {
namespace {

constexpr size_t kNoAllocScratchBytes = 256;  // the array's size; each call uses sizeof(DeviceStatus)
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
DeviceStatus* g_noalloc_status[64] = {};

// Device address of the static scratch on the current device.  The name of a
// __device__ array means nothing to the host, so its address is looked up
// once per device (with that device current) and cached.
DeviceStatus* noalloc_status_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_status[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) return nullptr;
    g_noalloc_status[dev] = static_cast<DeviceStatus*>(ptr);
  }
  return g_noalloc_status[dev];
}

// A caller of the allocation-free entry point has no status word to read, so
// a bounded wait that gave up is made visible in the outputs: every LSE entry
// becomes NaN.  Without a timeout each thread reads one word and returns.
__global__ void noalloc_report_timeout(const DeviceStatus* status, float* lse, long long n) {
  if (status->timeout == 0u) return;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
    lse[i] = __int_as_float(0x7FC00000);
}

// Test support for the NaN report: one warp waits, through the forward's own
// bounded wait, on an mbarrier that nothing arrives at, with a short limit,
// so it gives up and records the timeout in the given status word.
__global__ void __launch_bounds__(32) noalloc_wait_timeout_kernel(uint64_t limit_ns, DeviceStatus* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncwarp();
  mbar_wait(&bar, 0, &abort_flag, status, 92, limit_ns);
}

}  // namespace
}  // namespace fp4attn

extern "C" int fp4attn_fwd_directp_noalloc(const fp4attn_nvfp4_t* q, const fp4attn_nvfp4_t* k,
                                           const fp4attn_mxfp4_t* v, void* o, float* lse, int B, int H, int N, int D,
                                           float softmax_scale, void* stream) {
  const int st = check_fwd(q, k, v, o, lse, B, H, N, D, softmax_scale);
  if (st != FP4ATTN_OK) return st;
  // The scratch this call needs does not grow with the problem: one status
  // word for any supported size.  Anything that needed more would be refused.
  if (sizeof(DeviceStatus) > kNoAllocScratchBytes) return FP4ATTN_ERR_UNSUPPORTED;
  DeviceStatus* status = noalloc_status_word();
  if (!status) return FP4ATTN_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the array keeps the previous call's contents: clear the word first
  if (cudaMemsetAsync(status, 0, sizeof(DeviceStatus), s) != cudaSuccess) return FP4ATTN_ERR_CUDA;
  const int r = (D == 128)
                    ? launch<128, false>(q, k, v, o, lse, B, H, N, softmax_scale, -1, 0, 0, nullptr, nullptr, nullptr, s,
                                         status)
                    : launch<64, false>(q, k, v, o, lse, B, H, N, softmax_scale, -1, 0, 0, nullptr, nullptr, nullptr, s,
                                        status);
  if (r != FP4ATTN_OK) return r;
  noalloc_report_timeout<<<sm_count(), 256, 0, s>>>(status, lse, static_cast<long long>(B) * H * N);
  return cuda_status(cudaGetLastError());
}

extern "C" int fp4attn_debug_noalloc_timeout(float* lse, long long n, int limit_us, void* stream) {
  if (!lse || n <= 0 || !aligned16(lse) || limit_us <= 0 || limit_us > 1000000) return FP4ATTN_ERR_INVALID_ARG;
  DeviceStatus* status = noalloc_status_word();
  if (!status) return FP4ATTN_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(status, 0, sizeof(DeviceStatus), s) != cudaSuccess) return FP4ATTN_ERR_CUDA;
  noalloc_wait_timeout_kernel<<<1, 32, 0, s>>>(static_cast<uint64_t>(limit_us) * 1000u, status);
  noalloc_report_timeout<<<sm_count(), 256, 0, s>>>(status, lse, n);
  return cuda_status(cudaGetLastError());
}
