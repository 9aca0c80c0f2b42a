// Noncausal Direct-P FP4 attention forward for sm_103a.
//
// Method: "Hardware-Aware FP4 FlashAttention-4" (abstract: Direct-P for
// noncausal inference; "What the paper found": NVFP4 Q/K, log-softmax scores
// mapped directly to MXFP4 E2M1 probability codes with packed FMA and native
// conversion, denominator from the same rounded probabilities that PV
// consumes, LSE saved with O).
//
// One CTA computes one 128-row query tile of one (b, h) and streams the key /
// value tiles of that head through a TMA ring.  Roles (192 threads):
//   warps 0-3  softmax: one thread per query row.  Reads its S row from TMEM,
//              takes 32-key block maxima, maps scores to E2M1 codes
//              (fp32 FMA + ex2 + hardware e2m1x2 conversion), sums the decoded
//              codes for the denominator, writes the P tile and its E8M0
//              scales to shared memory, rescales O in TMEM when the reference
//              maximum moves, and finally normalises O and writes O / LSE.
//   warp 4     TMA producer (one elected lane).
//   warp 5     TMEM owner and single-thread tcgen05 MMA issuer:
//              S = Q K^T  (kind::mxf4nvf4, 16-element UE4M3 scales)
//              O += P V   (kind::mxf4, 32-element UE8M0 scales)
// TMEM (512 columns): S [0,128), O [128,128+D), scale factors from 256 on.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <mutex>

#include "internal.h"

namespace fp4attn {
namespace {

constexpr int kThreads = 192;
constexpr int kStages = 3;
// The MMA warp issues S(j+1) = Q K(j+1)^T before O += P(j) V(j), so the ring
// must hold tiles j and j+1 at once.
static_assert(kStages >= 2, "the K/V ring needs at least two stages");
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColO = 128, kColSFQ = 256, kColSFK = 264, kColSFP = 272, kColSFV = 276;
constexpr float kLog2Six = 2.5849625007211561f;  // log2(6) rounded to fp32
constexpr double kLog2E = 1.4426950408889634074;
// The reference maximum M moves (and O is rescaled) only when a new tile's
// ceil(max score) exceeds it by more than this many binades.
constexpr int kRescaleSlack = 0;

template <int D>
struct Layout {
  static constexpr int kRowBytes = D / 2;  // packed E2M1 bytes per Q/K row
  static constexpr int kQ = 0;
  static constexpr int kTileQK = 128 * kRowBytes;
  static constexpr int kTileV = D * 64;  // D channels x 128 keys
  static constexpr int kK = kQ + kTileQK;
  static constexpr int kV = kK + kStages * kTileQK;
  static constexpr int kP = kV + kStages * kTileV;
  static constexpr int kSFQ = kP + 128 * 64;
  static constexpr int kSFAtoms = D / 64;  // NVFP4 scale atoms per 128-row tile
  static constexpr int kSFK = kSFQ + kSFAtoms * 512;
  static constexpr int kSFV = kSFK + kStages * kSFAtoms * 512;
  static constexpr int kSFP = kSFV + kStages * 512;
  static constexpr int kBars = kSFP + 512;
  static constexpr int kNumBars = 1 + 2 * kStages + 4;
  static constexpr int kMisc = kBars + kNumBars * 8;
  static constexpr int kBytes = kMisc + 16;
  // Pad the request so that one CTA owns the SM: it allocates all 512 TMEM columns.
  static constexpr int kAlloc = (kBytes + 1024 > 120 * 1024) ? kBytes + 1024 : 120 * 1024;
  static_assert(kTileQK % 1024 == 0 && kTileV % 1024 == 0, "tiles must keep 1024-B alignment");
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

// Sum of the decoded values of eight non-negative E2M1 codes, in units of 0.5,
// as four byte lanes (each lane <= 24): a byte-permute table lookup.
__device__ __forceinline__ uint32_t e2m1x8_halfsum_lanes(uint32_t w) {
  constexpr uint32_t lo = 0x03020100u;  // 2 x {0, .5, 1, 1.5}
  constexpr uint32_t hi = 0x0C080604u;  // 2 x {2, 3, 4, 6}
  return __byte_perm(lo, hi, w & 0xFFFFu) + __byte_perm(lo, hi, w >> 16);
}

template <int D, bool DUMP>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_directp_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  using L = Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBars);
  uint64_t* bar_q_full = bars;
  uint64_t* bar_kv_full = bars + 1;
  uint64_t* bar_kv_empty = bars + 1 + kStages;
  uint64_t* bar_s_full = bars + 1 + 2 * kStages;
  uint64_t* bar_s_free = bar_s_full + 1;
  uint64_t* bar_p_full = bar_s_full + 2;
  uint64_t* bar_o_full = bar_s_full + 3;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qt = blockIdx.x;
  const int bh = blockIdx.y;
  const int N = p.N;
  const int nkv = p.ntiles;

  if (threadIdx.x == 0) {
    mbar_init(bar_q_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar_kv_full + s, 1);
      mbar_init(bar_kv_empty + s, 1);
    }
    mbar_init(bar_s_full, 1);
    mbar_init(bar_s_free, 128);
    mbar_init(bar_p_full, 128);
    mbar_init(bar_o_full, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      constexpr uint32_t kSfBytes = L::kSFAtoms * 512;
      mbar_arrive_expect_tx(bar_q_full, L::kTileQK + kSfBytes);
      tma_load_3d(smem + L::kQ, &tm_q, bar_q_full, 0, qt * 128, bh);
      bulk_load(smem + L::kSFQ, p.q_sf + (static_cast<size_t>(bh) * p.ntiles + qt) * kSfBytes, kSfBytes, bar_q_full);
      for (int j = 0; j < nkv; ++j) {
        const int s = j % kStages;
        if (j >= kStages && !mbar_wait(bar_kv_empty + s, ((j / kStages) - 1) & 1, abort_flag, p.status, 1)) break;
        mbar_arrive_expect_tx(bar_kv_full + s, L::kTileQK + L::kTileV + kSfBytes + 512);
        tma_load_3d(smem + L::kK + s * L::kTileQK, &tm_k, bar_kv_full + s, 0, j * 128, bh);
        tma_load_2d(smem + L::kV + s * L::kTileV, &tm_v, bar_kv_full + s, j * 64, bh * D);
        bulk_load(smem + L::kSFK + s * kSfBytes, p.k_sf + (static_cast<size_t>(bh) * p.ntiles + j) * kSfBytes,
                  kSfBytes, bar_kv_full + s);
        bulk_load(smem + L::kSFV + s * 512, p.v_sf + (static_cast<size_t>(bh) * p.ntiles + j) * 512, 512,
                  bar_kv_full + s);
      }
      // Before leaving, make sure no copy into this CTA's shared memory is
      // still in flight: wait for the last fill of every stage.
      for (int j = nkv - kStages < 0 ? 0 : nkv - kStages; j < nkv; ++j)
        mbar_wait(bar_kv_full + (j % kStages), (j / kStages) & 1, abort_flag, p.status, 2);
      mbar_wait(bar_q_full, 0, abort_flag, p.status, 3);
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t kSwizzleQK = (D == 128) ? 4u : 6u;  // 64-B or 32-B rows
      constexpr uint32_t kSbo = 8 * L::kRowBytes;
      constexpr uint32_t idesc_qk = idesc_fp4_block_scaled(128, 128, 0, 0, 0);
      constexpr uint32_t idesc_pv0 = idesc_fp4_block_scaled(128, D, 1, 0, 0);
      constexpr uint32_t idesc_pv1 = idesc_fp4_block_scaled(128, D, 1, 2, 2);
      const uint64_t qdesc = smem_desc(smem_u32(smem + L::kQ), 16, kSbo, kSwizzleQK);
      const uint64_t pdesc = smem_desc(smem_u32(smem + L::kP), 16, 512, 4);
      bool ok = mbar_wait(bar_q_full, 0, abort_flag, p.status, 10);
      if (ok) {
        tc_fence_after();
        for (int a = 0; a < L::kSFAtoms; ++a) tc_cp_sf_atom(tmem + kColSFQ + 4 * a, smem + L::kSFQ + a * 512);
      }
      auto issue_qk = [&](int j) {
        const int s = j % kStages;
        for (int a = 0; a < L::kSFAtoms; ++a)
          tc_cp_sf_atom(tmem + kColSFK + 4 * a, smem + L::kSFK + (s * L::kSFAtoms + a) * 512);
        const uint64_t kdesc = smem_desc(smem_u32(smem + L::kK + s * L::kTileQK), 16, kSbo, kSwizzleQK);
        for (int ks = 0; ks < D / 64; ++ks)
          mma_nvf4(tmem + kColS, qdesc + 2 * ks, kdesc + 2 * ks, idesc_qk, tmem + kColSFQ + 4 * ks,
                   tmem + kColSFK + 4 * ks, ks > 0);
        tc_commit(bar_s_full);
      };
      if (ok && (ok = mbar_wait(bar_kv_full, 0, abort_flag, p.status, 11))) {
        tc_fence_after();
        issue_qk(0);
      }
      for (int j = 0; ok && j < nkv; ++j) {
        const int s = j % kStages;
        if (j + 1 < nkv) {
          const int s1 = (j + 1) % kStages;
          if (!(ok = mbar_wait(bar_kv_full + s1, ((j + 1) / kStages) & 1, abort_flag, p.status, 12))) break;
          if (!(ok = mbar_wait(bar_s_free, j & 1, abort_flag, p.status, 13))) break;
          tc_fence_after();
          issue_qk(j + 1);
        }
        if (!(ok = mbar_wait(bar_p_full, j & 1, abort_flag, p.status, 14))) break;
        tc_fence_after();
        tc_cp_sf_atom(tmem + kColSFP, smem + L::kSFP);
        tc_cp_sf_atom(tmem + kColSFV, smem + L::kSFV + s * 512);
        const uint64_t vdesc = smem_desc(smem_u32(smem + L::kV + s * L::kTileV), 16, 512, 4);
        mma_mxf4(tmem + kColO, pdesc, vdesc, idesc_pv0, tmem + kColSFP, tmem + kColSFV, j > 0);
        mma_mxf4(tmem + kColO, pdesc + 2, vdesc + 2, idesc_pv1, tmem + kColSFP, tmem + kColSFV, true);
        tc_commit(bar_o_full);
        tc_commit(bar_kv_empty + s);
      }
    }
  } else {
    // ------------------------------------------------------------ softmax rows
    const int row = threadIdx.x;  // 0..127 == TMEM lane
    const int qrow = qt * 128 + row;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t tS = tmem + lane_base + kColS;
    const uint32_t tO = tmem + lane_base + kColO;
    const float c = static_cast<float>(((static_cast<double>(p.softmax_scale) * kLog2E) *
                                        static_cast<double>(*p.g_q)) * static_cast<double>(*p.g_k));
    const bool dump_row = DUMP && bh == p.dump_bh && qrow >= p.dump_row0 && qrow < p.dump_row0 + p.dump_nrows;
    int m_ref = 0;
    float l_run = 0.0f;
    bool ok = true;
    // tcgen05.ld / tcgen05.st are warp-collective (.sync.aligned): every
    // branch around them below is made warp-uniform with a vote.
    for (int j = 0; j < nkv; ++j) {
      ok = mbar_wait(bar_s_full, j & 1, abort_flag, p.status, 20);
      if (!__all_sync(0xFFFFFFFFu, ok)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float s[128];
      tmem_ld32(tS + 0, *reinterpret_cast<float(*)[32]>(s + 0));
      tmem_ld32(tS + 32, *reinterpret_cast<float(*)[32]>(s + 32));
      tmem_ld32(tS + 64, *reinterpret_cast<float(*)[32]>(s + 64));
      tmem_ld32(tS + 96, *reinterpret_cast<float(*)[32]>(s + 96));
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(bar_s_free);

      const int valid = N - j * 128;  // keys of this tile that exist (>= 1)
      if (valid < 128) {
#pragma unroll
        for (int i = 0; i < 128; ++i)
          if (i >= valid) s[i] = -INFINITY;
      }
      // block maxima of the scaled scores (c > 0, so max(c*s) = c*max(s))
      float xb[4];
      int kb[4];
      float xmax = -INFINITY;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        float m = s[32 * b];
#pragma unroll
        for (int i = 1; i < 32; ++i) m = fmaxf(m, s[32 * b + i]);
        xb[b] = __fmul_rn(c, m);
        xmax = fmaxf(xmax, xb[b]);
        kb[b] = (xb[b] == -INFINITY) ? 0 : static_cast<int>(ceilf(__fsub_rn(xb[b], kLog2Six)));
      }
      const int m_tile = static_cast<int>(ceilf(xmax));
      int m_old = m_ref;
      bool rescale = false;
      if (j == 0) {
        m_ref = m_tile;
      } else if (m_tile > m_ref + kRescaleSlack) {
        m_ref = m_tile;
        rescale = true;
      }
      // Direct-P: codes of 2^(X - K_b), packed 8 per word
      uint32_t w[16];
      float l_tile = 0.0f;
      uint32_t sfword = 0;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const float nk = static_cast<float>(-kb[b]);
        uint32_t lanes = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          float y[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) y[i] = ex2_approx(__fmaf_rn(c, s[32 * b + 8 * q + i], nk));
          w[4 * b + q] = cvt_e2m1x8(y[0], y[1], y[2], y[3], y[4], y[5], y[6], y[7]);
          lanes += e2m1x8_halfsum_lanes(w[4 * b + q]);
        }
        const int halfsum = __dp4a(static_cast<int>(lanes), 0x01010101, 0);
        int e = kb[b] - m_ref;
        e = e < -127 ? -127 : e;
        const uint32_t byte = (xb[b] == -INFINITY) ? 0u : static_cast<uint32_t>(e + 127);
        sfword |= byte << (8 * b);
        l_tile += static_cast<float>(halfsum) * exp2_int(e - 1);
      }
      if (j > 0) {
        // the previous PV product must be done before P and O are touched
        ok = mbar_wait(bar_o_full, (j - 1) & 1, abort_flag, p.status, 21);
        if (!__all_sync(0xFFFFFFFFu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      // Rescale O (and l) of the rows whose reference maximum moved; the whole
      // warp takes part in the TMEM round trip, other rows multiply by 1.
      const float f = rescale ? exp2_int(m_old - m_ref) : 1.0f;
      l_run *= f;
      if (__any_sync(0xFFFFFFFFu, rescale)) {
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
      l_run += l_tile;
      uint8_t* prow = smem + L::kP + row * 64;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int chunk = b ^ ((row >> 1) & 3);  // 64-byte swizzle of the K-major P tile
        *reinterpret_cast<uint4*>(prow + chunk * 16) = make_uint4(w[4 * b], w[4 * b + 1], w[4 * b + 2], w[4 * b + 3]);
      }
      *reinterpret_cast<uint32_t*>(smem + L::kSFP + (row & 31) * 16 + (row >> 5) * 4) = sfword;
      if (dump_row) {
        const size_t rr = static_cast<size_t>(qrow - p.dump_row0);
        uint4* dst = reinterpret_cast<uint4*>(p.dump_codes + rr * (p.ntiles * 64) + j * 64);
#pragma unroll
        for (int b = 0; b < 4; ++b) dst[b] = make_uint4(w[4 * b], w[4 * b + 1], w[4 * b + 2], w[4 * b + 3]);
#pragma unroll
        for (int b = 0; b < 4; ++b) p.dump_kshift[rr * (p.ntiles * 4) + j * 4 + b] = kb[b];
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(bar_p_full);
    }
    // ------------------------------------------------------------ epilogue
    if (ok) ok = mbar_wait(bar_o_full, (nkv - 1) & 1, abort_flag, p.status, 22);
    if (__all_sync(0xFFFFFFFFu, ok)) {
      tc_fence_after();
      const float inv_l = 1.0f / l_run;
      const bool store = qrow < N;
      __nv_bfloat16* orow = p.o + (static_cast<size_t>(bh) * N + (store ? qrow : 0)) * D;
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        float o[32];
        tmem_ld32(tO + 32 * cc, o);
        tmem_wait_ld();
        if (store) {
          uint32_t packed[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            __nv_bfloat162 h2 = __floats2bfloat162_rn(o[2 * i] * inv_l, o[2 * i + 1] * inv_l);
            packed[i] = *reinterpret_cast<uint32_t*>(&h2);
          }
          uint4* dst = reinterpret_cast<uint4*>(orow + 32 * cc);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            dst[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
        }
        if (dump_row) {
          float* od = p.dump_o + static_cast<size_t>(qrow - p.dump_row0) * D + 32 * cc;
#pragma unroll
          for (int i = 0; i < 32; ++i) od[i] = o[i] * inv_l;
        }
      }
      if (store) p.lse[static_cast<size_t>(bh) * N + qrow] = 0.69314718055994531f * (static_cast<float>(m_ref) + log2f(l_run));
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 5) {
    __syncwarp();
    tmem_dealloc(tmem, kTmemCols);
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

template <int D, bool DUMP>
int launch(const fp4attn_nvfp4_t* q, const fp4attn_nvfp4_t* k, const fp4attn_mxfp4_t* v, void* o, float* lse,
           int B, int H, int N, float softmax_scale, int dump_bh, int row0, int nrows, uint8_t* codes,
           int32_t* kshift, float* o_f32, cudaStream_t stream) {
  using L = Layout<D>;
  DeviceStatus* status = device_status_ptr();
  if (!status) return FP4ATTN_ERR_CUDA;
  const int ntiles = n_row_tiles(N);
  const int BH = B * H;
  CUtensorMap tq, tk, tv;
  const CUtensorMapSwizzle swz_qk = (D == 128) ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B;
  const cuuint64_t qk_dims[3] = {static_cast<cuuint64_t>(D / 2), static_cast<cuuint64_t>(N),
                                 static_cast<cuuint64_t>(BH)};
  const cuuint64_t qk_strides[2] = {static_cast<cuuint64_t>(D / 2), static_cast<cuuint64_t>(N) * (D / 2)};
  const cuuint32_t qk_box[3] = {static_cast<cuuint32_t>(D / 2), 128, 1};
  const cuuint64_t v_dims[2] = {static_cast<cuuint64_t>(ntiles) * 64, static_cast<cuuint64_t>(BH) * D};
  const cuuint64_t v_strides[1] = {static_cast<cuuint64_t>(ntiles) * 64};
  const cuuint32_t v_box[2] = {64, static_cast<cuuint32_t>(D)};
  if (!make_map(&tq, q->payload, 3, qk_dims, qk_strides, qk_box, swz_qk) ||
      !make_map(&tk, k->payload, 3, qk_dims, qk_strides, qk_box, swz_qk) ||
      !make_map(&tv, v->payload_t, 2, v_dims, v_strides, v_box, CU_TENSOR_MAP_SWIZZLE_64B))
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
  auto kern = fwd_directp_kernel<D, DUMP>;
  static std::once_flag attr_once[64];
  int dev = 0;
  cudaGetDevice(&dev);
  cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once[dev & 63], [&] {
    attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  });
  if (attr_err != cudaSuccess) return FP4ATTN_ERR_CUDA;
  dim3 grid(ntiles, BH);
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
  if (D == 128) return launch<128, false>(q, k, v, o, lse, B, H, N, softmax_scale, -1, 0, 0, nullptr, nullptr, nullptr, s);
  return launch<64, false>(q, k, v, o, lse, B, H, N, softmax_scale, -1, 0, 0, nullptr, nullptr, nullptr, s);
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
  if (D == 128) return launch<128, true>(q, k, v, o, lse, B, H, N, softmax_scale, bh, row0, nrows, codes, kshift, o_f32, s);
  return launch<64, true>(q, k, v, o, lse, B, H, N, softmax_scale, bh, row0, nrows, codes, kshift, o_f32, s);
}
