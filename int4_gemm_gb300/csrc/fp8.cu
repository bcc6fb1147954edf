// FP8 (E4M3) blockwise quantization and the block-promoted FP8 GEMM.
//
// "Quantization in deployment", section "Fake quantization" (fp8,
// fp8_blockwise): weights carry one FP32 scale per 128 x 128 block,
// activations one per (1, 128) block; s = max(amax, 1e-12) / 448 and the code
// is the E4M3 value of clamp(x / s, -448, 448), the cast rounding to nearest
// even.  Exercise 2 of the same page (the cost of block FP8): the tensor
// cores accumulate the FP8 products of one 128-wide K block, the block's sum
// is multiplied by its activation and weight scales and added into the FP32
// result ("promotion").
//
// GEMM design (one CTA per SM, persistent over 128 x 128 output tiles):
//   warp 0      TMA producer: the A and B tiles of each K block (128 rows x
//               128 bytes each, 128-byte swizzle) into a 6-stage ring;
//   warp 1      MMA issuer: four tcgen05.mma kind::f8f6f4 (128 x 128 x 32)
//               per K block into one of four 128-column TMEM slots, starting
//               from zero, so every slot holds the product of one K block;
//   warps 2..9  promotion: warp w reads lane quarter w % 4, column half
//               (w - 2) / 4 of a slot, hands the slot back to the MMA and
//               adds slot * sa[m, kb] * sb[n / 128, kb] into 64 FP32
//               registers per thread; after the last K block of a tile they
//               store the tile row by row.
// The slot ring runs on across tiles: the MMA starts the next tile while the
// promotion warps store the last one.
#include "common.cuh"
#include "internal.h"

#include <algorithm>

namespace q4 {
namespace {

// ------------------------------------------------------------------ helpers
// E4M3 bytes of two floats, round to nearest even; .satfinite clamps to
// +-448 as the page's clamp does.  lo goes to bits 0..7, hi to bits 8..15.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Four consecutive elements starting at element index e (e % 4 == 0).
template <typename T>
__device__ __forceinline__ void load4(const T* __restrict__ x, int64_t e, float (&v)[4]) {
  if constexpr (sizeof(T) == 4) {
    const float4 w = __ldg(reinterpret_cast<const float4*>(x + e));
    v[0] = w.x; v[1] = w.y; v[2] = w.z; v[3] = w.w;
  } else {
    const uint2 w = __ldg(reinterpret_cast<const uint2*>(x + e));
    const T* h = reinterpret_cast<const T*>(&w);
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = Elem<T>::to_f(h[j]);
  }
}

// The four E4M3 bytes of x_j / s (one IEEE division each), byte j = element j.
__device__ __forceinline__ uint32_t e4m3_codes4(const float (&v)[4], float s) {
  return cvt_e4m3x2(__fdiv_rn(v[0], s), __fdiv_rn(v[1], s)) |
         (cvt_e4m3x2(__fdiv_rn(v[2], s), __fdiv_rn(v[3], s)) << 16);
}

// ------------------------------------------------------------------ quantizers
constexpr int kQThreads = 256;

// Activations, blocks (1, 128): one warp per block, four elements per lane.
// codes [M, K], scales [M, K / 128] row-major.
template <typename T>
__global__ void __launch_bounds__(kQThreads)
    fp8_act_quant_kernel(const T* __restrict__ x, int64_t M, int64_t K, uint8_t* __restrict__ codes,
                         float* __restrict__ scales, int* status) {
  pdl_wait();  // inputs may come from the previous kernel
  const int lane = threadIdx.x & 31;
  const int64_t KB = K / 128, nblk = M * KB;
  const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
  bool bad = false;
  for (int64_t b = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; b < nblk; b += nw) {
    const int64_t row = b / KB, kb = b - row * KB;
    const int64_t e = row * K + kb * 128 + lane * 4;
    float v[4];
    load4<T>(x, e, v);
    float amax = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      bad |= nonfinite(v[j]);
      amax = fmaxf(amax, fabsf(v[j]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float s = __fdiv_rn(fmaxf(amax, 1e-12f), 448.0f);
    *reinterpret_cast<uint32_t*>(codes + e) = e4m3_codes4(v, s);
    if (lane == 0) scales[b] = s;
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) latch_status(status, Q4_ERR_NONFINITE);
}

// Weights, blocks 128 x 128: one CTA per block, thread t holds 64 elements of
// block row t / 2 (half t % 2).  codes [N, K], scales [N / 128, K / 128].
template <typename T>
__global__ void __launch_bounds__(kQThreads)
    fp8_weight_quant_kernel(const T* __restrict__ w, int64_t K, uint8_t* __restrict__ codes,
                            float* __restrict__ scales, int* status) {
  pdl_wait();
  __shared__ float s_max[kQThreads / 32];
  __shared__ int s_bad;
  const int64_t KB = K / 128;
  const int64_t bn = blockIdx.x / KB, kb = blockIdx.x - bn * KB;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int64_t e0 = (bn * 128 + (t >> 1)) * K + kb * 128 + (t & 1) * 64;
  if (t == 0) s_bad = 0;
  float v[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i) load4<T>(w, e0 + 4 * i, v[i]);
  float amax = 0.f;
  bool bad = false;
#pragma unroll
  for (int i = 0; i < 16; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      bad |= nonfinite(v[i][j]);
      amax = fmaxf(amax, fabsf(v[i][j]));
    }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if (lane == 0) s_max[warp] = amax;
  __syncthreads();
  if (bad) s_bad = 1;
  float bmax = 0.f;
#pragma unroll
  for (int i = 0; i < kQThreads / 32; ++i) bmax = fmaxf(bmax, s_max[i]);
  const float s = __fdiv_rn(fmaxf(bmax, 1e-12f), 448.0f);
#pragma unroll
  for (int q = 0; q < 4; ++q)
    reinterpret_cast<uint4*>(codes + e0)[q] =
        make_uint4(e4m3_codes4(v[4 * q], s), e4m3_codes4(v[4 * q + 1], s),
                   e4m3_codes4(v[4 * q + 2], s), e4m3_codes4(v[4 * q + 3], s));
  __syncthreads();
  if (t == 0) {
    scales[blockIdx.x] = s;
    if (s_bad) latch_status(status, Q4_ERR_NONFINITE);
  }
}

// ------------------------------------------------------------------ GEMM
constexpr int GBM = 128, GBN = 128, GBK = 128;  // tile; K block = one promotion unit
constexpr int kGStages = 6;
constexpr int kSlots = 4;                         // TMEM accumulator slots, 128 columns each
constexpr uint32_t kGTileBytes = GBM * GBK;       // one operand tile of one K block (bytes)
constexpr uint32_t kGStageBytes = 2 * kGTileBytes;
constexpr int kPromoWarp0 = 2, kPromoWarps = 8;
constexpr int kBandM = 32;                       // M tiles per band of the tile order
constexpr int kSP = 4;                           // K blocks of scale prefetch in registers
constexpr int kGThreads = (kPromoWarp0 + kPromoWarps) * 32;
constexpr uint32_t kGSmemBytes = kGStages * kGStageBytes + 1024 /*align*/ + 256 /*barriers*/;
static_assert(kGSmemBytes <= 232448, "shared memory");
static_assert(kSlots * GBN <= 512, "TMEM columns");

struct GSmem {
  uint64_t full[kGStages];
  uint64_t empty[kGStages];
  uint64_t slot_full[kSlots];
  uint64_t slot_empty[kSlots];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(GSmem) <= 256, "barrier block");

struct Fp8Params {
  int64_t M, N, K;
  const float* sa;  // [M, K / 128]
  const float* sb;  // [N / 128, K / 128]
  void* C;          // [M, N]
  int c_dtype;
  int num_m, num_n;
  KernelCtl ctl;
};

// Instruction descriptor of tcgen05.mma kind::f8f6f4: FP32 accumulator
// (bits 4-5 = 1), A and B E4M3 (format 0 in bits 7-9 and 10-12), both
// K-major, N / 8 in bits 17-22, M / 16 in bits 24-28.
__host__ __device__ constexpr uint32_t f8_idesc(uint32_t M, uint32_t N) {
  return (1u << 4) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

__device__ __forceinline__ void tc_mma_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__global__ void __launch_bounds__(kGThreads, 1)
    fp8_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a,
                    const __grid_constant__ CUtensorMap tmap_b, const Fp8Params p) {
  extern __shared__ uint8_t smem_raw[];
  pdl_wait();  // operands and scales may come from the previous kernel
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  GSmem* sm = reinterpret_cast<GSmem*>(smem + kGStages * kGStageBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KB = (int)(p.K / GBK);
  const int total_tiles = p.num_m * p.num_n;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kGStages; ++s) {
      mbar_init(smem_u32(&sm->full[s]), 1);
      mbar_init(smem_u32(&sm->empty[s]), 1);
    }
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(smem_u32(&sm->slot_full[s]), 1);
      mbar_init(smem_u32(&sm->slot_empty[s]), kPromoWarps);  // one arrival per promotion warp
    }
    mbar_init(smem_u32(&sm->mma_done), 1);
    sm->abort = 0;
    fence_mbar_init();
    prefetch_tmap(&tmap_a);
    prefetch_tmap(&tmap_b);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&sm->tmem_base), kSlots * GBN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm->tmem_base;
  volatile int* abort_flag = &sm->abort;
  // Tile order: bands of kBandM M tiles (32 x 128 rows of A, 33.5 MB at K = 8192,
  // stay in L2), M fastest inside a band, so the CTAs working at one time share
  // their B tiles and every band reads B from DRAM once.
  auto tile_mn = [&](int t, int& m0, int& n0) {
    const int band_tiles = kBandM * p.num_n;
    const int band = t / band_tiles, r = t - band * band_tiles;
    const int gm = min(kBandM, p.num_m - band * kBandM);
    m0 = (band * kBandM + r % gm) * GBM;
    n0 = (r / gm) * GBN;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    uint32_t stage = 0, phase = 0;
    int issued[kGStages];
    uint32_t issued_phase[kGStages];
    for (int s = 0; s < kGStages; ++s) issued[s] = 0, issued_phase[s] = 0;
    bool alive = true;
    for (int t = blockIdx.x; t < total_tiles && alive; t += gridDim.x) {
      int m0, n0;
      tile_mn(t, m0, n0);
      for (int kb = 0; kb < KB; ++kb) {
        if (!mbar_wait(smem_u32(&sm->empty[stage]), phase ^ 1, p.ctl, abort_flag)) {
          alive = false;
          break;
        }
        uint8_t* st = smem + stage * kGStageBytes;
        const uint32_t full = smem_u32(&sm->full[stage]);
        if (lane == 0) {
          mbar_arrive_expect_tx(full, kGStageBytes);
          tma_load_2d(smem_u32(st), &tmap_a, kb * GBK, m0, full);
          tma_load_2d(smem_u32(st + kGTileBytes), &tmap_b, kb * GBK, n0, full);
        }
        issued[stage] = 1;
        issued_phase[stage] = phase;
        if (++stage == kGStages) stage = 0, phase ^= 1;
      }
    }
    // drain: every copy this warp issued has landed before the CTA exits
    if (lane == 0) {
      KernelCtl drain = p.ctl;
      for (int s = 0; s < kGStages; ++s)
        if (issued[s]) mbar_wait(smem_u32(&sm->full[s]), issued_phase[s], drain, nullptr);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = f8_idesc(GBM, GBN);
      uint32_t stage = 0, phase = 0, gk = 0;  // gk: K blocks issued so far (slot ring position)
      bool alive = true;
      for (int t = blockIdx.x; t < total_tiles && alive; t += gridDim.x) {
        for (int kb = 0; kb < KB; ++kb, ++gk) {
          const uint32_t slot = gk % kSlots, sphase = (gk / kSlots) & 1;
          if (!mbar_wait(smem_u32(&sm->slot_empty[slot]), sphase ^ 1, p.ctl, abort_flag) ||
              !mbar_wait(smem_u32(&sm->full[stage]), phase, p.ctl, abort_flag)) {
            alive = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = smem_u32(smem + stage * kGStageBytes);
          const uint32_t d = tmem + slot * GBN;
#pragma unroll
          for (uint32_t k = 0; k < GBK / 32; ++k) {
            const uint64_t ad = smem_desc(st + 32 * k, 16, 1024, 2);
            const uint64_t bd = smem_desc(st + kGTileBytes + 32 * k, 16, 1024, 2);
            tc_mma_f8(d, ad, bd, idesc, k != 0 ? 1u : 0u);
          }
          tc_commit(smem_u32(&sm->empty[stage]));    // the stage is free once these MMAs are done
          tc_commit(smem_u32(&sm->slot_full[slot]));  // and the slot holds this K block's product
          if (++stage == kGStages) stage = 0, phase ^= 1;
        }
      }
      // all MMAs this thread issued are complete before TMEM is released
      tc_commit(smem_u32(&sm->mma_done));
      KernelCtl drain = p.ctl;
      mbar_wait(smem_u32(&sm->mma_done), 0, drain, nullptr);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ promotion + store
    const int q = warp & 3;                       // TMEM lane quarter this warp may access
    const int h = (warp - kPromoWarp0) >> 2;      // column half of the slot
    const uint32_t t_lane = tmem + ((uint32_t)(q * 32) << 16) + h * 64;
    uint32_t gk = 0;
    bool alive = true;
    for (int t = blockIdx.x; t < total_tiles && alive; t += gridDim.x) {
      int m0, n0;
      tile_mn(t, m0, n0);
      const int64_t row = m0 + q * 32 + lane;
      const bool row_ok = row < p.M;
      const float* sa_row = p.sa + (row_ok ? row : p.M - 1) * KB;
      const float* sb_row = p.sb + (int64_t)(n0 / GBN) * KB;
      float acc[64];
#pragma unroll
      for (int j = 0; j < 64; ++j) acc[j] = 0.f;
      // the scales of K block kb + kSP are requested while block kb is
      // promoted: a K block takes a few hundred ns, an L2 load about a us
      float sa_q[kSP], sb_q[kSP];
#pragma unroll
      for (int i = 0; i < kSP; ++i) {
        sa_q[i] = i < KB ? __ldg(sa_row + i) : 0.f;
        sb_q[i] = i < KB ? __ldg(sb_row + i) : 0.f;
      }
      for (int kb0 = 0; kb0 < KB && alive; kb0 += kSP) {
#pragma unroll
        for (int i = 0; i < kSP; ++i) {
          const int kb = kb0 + i;
          if (kb >= KB || !alive) continue;
          const uint32_t slot = gk % kSlots, sphase = (gk / kSlots) & 1;
          const float sc = sa_q[i] * sb_q[i];
          if (kb + kSP < KB) sa_q[i] = __ldg(sa_row + kb + kSP), sb_q[i] = __ldg(sb_row + kb + kSP);
          if (!mbar_wait(smem_u32(&sm->slot_full[slot]), sphase, p.ctl, abort_flag)) {
            alive = false;
            continue;
          }
          tc_fence_after();
          uint32_t r0[32], r1[32];
          tmem_ld_32x32b_x32(t_lane + slot * GBN, r0);
          tmem_ld_32x32b_x32(t_lane + slot * GBN + 32, r1);
          tmem_ld_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&sm->slot_empty[slot]));
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            acc[j] = fmaf(__uint_as_float(r0[j]), sc, acc[j]);
            acc[32 + j] = fmaf(__uint_as_float(r1[j]), sc, acc[32 + j]);
          }
          ++gk;
        }
      }
      if (!alive || !row_ok) continue;
      const int64_t col0 = n0 + h * 64;
      if (p.c_dtype == Q4_BF16) {
        uint4* out = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.C) + row * p.N + col0);
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          uint32_t w[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[8 * v + 2 * i], acc[8 * v + 2 * i + 1]);
            w[i] = *reinterpret_cast<const uint32_t*>(&b2);
          }
          out[v] = make_uint4(w[0], w[1], w[2], w[3]);
        }
      } else {
        float4* out = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.C) + row * p.N + col0);
#pragma unroll
        for (int v = 0; v < 16; ++v)
          out[v] = make_float4(acc[4 * v], acc[4 * v + 1], acc[4 * v + 2], acc[4 * v + 3]);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kSlots * GBN);
  }
}


// ------------------------------------------------------------------ GEMM, CTA pairs
// For M > 128: a cluster of two CTAs computes one 256 x 256 tile with the
// 2-SM MMA (tcgen05.mma.cta_group::2.kind::f8f6f4, 256 x 256 x 32 per
// instruction).  CTA rank r loads A rows m0 + 128 r .. and B rows n0 + 128 r ..
// of each K block into its own stage; the even CTA issues the MMAs for both
// and each CTA's TMEM receives its 128 rows x 256 columns.  Per CTA and K
// block that is 32 KB of copies for 128 x 256 x 128 products: half the bytes
// per product of the 128 x 128 kernel, and a quarter of the MMA instructions.
//   warp 0      TMA producer (own A rows, own half of B) -> local `full`;
//   warp 1      even CTA: MMA issuer (waits for its own `full` and for the odd
//               CTA's relay on `pair_full`), two 256-column TMEM slots;
//               odd CTA: relay (waits for its `full`, arrives on the even
//               CTA's `pair_full`);
//   warps 2..9  promotion: lane quarter warp % 4, column half (warp - 2) / 4
//               (128 columns, 128 FP32 registers per thread); each reads its
//               slot in eight 16-column loads and arrives on the even CTA's
//               `slot_empty` (16 arrivals: 8 warps x 2 CTAs).
constexpr int kPStages = 6;
constexpr int kPSlots = 2;                          // TMEM slots of 256 columns
constexpr int PBN = 256;                            // pair tile N (128 B rows per CTA)
constexpr uint32_t kPStageBytes = 2 * kGTileBytes;  // A rows + this CTA's half of B
constexpr uint32_t kPSmemBytes = kPStages * kPStageBytes + 1024 /*align*/ + 256 /*barriers*/;
static_assert(kPSmemBytes <= 232448, "shared memory");
static_assert(kPSlots * PBN <= 512, "TMEM columns");

struct PSmem {
  uint64_t full[kPStages];       // this CTA's copies of the stage landed
  uint64_t pair_full[kPStages];  // even CTA: the odd CTA's copies landed (relay)
  uint64_t empty[kPStages];      // the stage's MMAs are done (both CTAs)
  uint64_t slot_full[kPSlots];   // the slot holds one K block's product (both CTAs)
  uint64_t slot_empty[kPSlots];  // even CTA: every promotion warp of the pair read it
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(PSmem) <= 256, "barrier block");

__device__ __forceinline__ void tc_mma_f8_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                               uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__global__ void __launch_bounds__(kGThreads, 1)
    fp8_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmap_a,
                         const __grid_constant__ CUtensorMap tmap_b, const Fp8Params p) {
  extern __shared__ uint8_t smem_raw[];
  pdl_wait();  // operands and scales may come from the previous kernel
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  PSmem* sm = reinterpret_cast<PSmem*>(smem + kPStages * kPStageBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = (int)cluster_ctarank();  // 0: issues the pair's MMAs
  const int cid = blockIdx.x >> 1, ncl = gridDim.x >> 1;
  const int KB = (int)(p.K / GBK);
  const int num_pm = (int)((p.M + 2 * GBM - 1) / (2 * GBM)), num_pn = (int)((p.N + PBN - 1) / PBN);
  const int total_tiles = num_pm * num_pn;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPStages; ++s) {
      mbar_init(smem_u32(&sm->full[s]), 1);
      mbar_init(smem_u32(&sm->pair_full[s]), 1);
      mbar_init(smem_u32(&sm->empty[s]), 1);
    }
    for (int s = 0; s < kPSlots; ++s) {
      mbar_init(smem_u32(&sm->slot_full[s]), 1);
      mbar_init(smem_u32(&sm->slot_empty[s]), 2 * kPromoWarps);
    }
    mbar_init(smem_u32(&sm->mma_done), 1);
    sm->abort = 0;
    fence_mbar_init();
    prefetch_tmap(&tmap_a);
    prefetch_tmap(&tmap_b);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(&sm->tmem_base), kPSlots * PBN);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_barrier_sync();  // the peer's barriers exist before any remote arrival
  tc_fence_after();
  const uint32_t tmem = sm->tmem_base;
  volatile int* abort_flag = &sm->abort;
  // Pair tiles in bands of kBandM / 2 M tiles (the same 32 x 128 rows of A in
  // L2 as the single-CTA kernel), M fastest inside a band.
  auto tile_mn = [&](int t, int& m0, int& n0) {
    constexpr int kBand = kBandM / 2;
    const int band_tiles = kBand * num_pn;
    const int band = t / band_tiles, r = t - band * band_tiles;
    const int gm = min(kBand, num_pm - band * kBand);
    m0 = (band * kBand + r % gm) * 2 * GBM;
    n0 = (r / gm) * PBN;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    uint32_t stage = 0, phase = 0;
    int issued[kPStages];
    uint32_t issued_phase[kPStages];
    for (int s = 0; s < kPStages; ++s) issued[s] = 0, issued_phase[s] = 0;
    bool alive = true;
    for (int t = cid; t < total_tiles && alive; t += ncl) {
      int m0, n0;
      tile_mn(t, m0, n0);
      for (int kb = 0; kb < KB; ++kb) {
        if (!mbar_wait(smem_u32(&sm->empty[stage]), phase ^ 1, p.ctl, abort_flag)) {
          alive = false;
          break;
        }
        uint8_t* st = smem + stage * kPStageBytes;
        const uint32_t full = smem_u32(&sm->full[stage]);
        if (lane == 0) {
          mbar_arrive_expect_tx(full, kPStageBytes);
          tma_load_2d(smem_u32(st), &tmap_a, kb * GBK, m0 + rank * GBM, full);
          tma_load_2d(smem_u32(st + kGTileBytes), &tmap_b, kb * GBK, n0 + rank * (PBN / 2), full);
        }
        issued[stage] = 1;
        issued_phase[stage] = phase;
        if (++stage == kPStages) stage = 0, phase ^= 1;
      }
    }
    // drain: every copy this warp issued has landed before the CTA exits
    if (lane == 0) {
      KernelCtl drain = p.ctl;
      for (int s = 0; s < kPStages; ++s)
        if (issued[s]) mbar_wait(smem_u32(&sm->full[s]), issued_phase[s], drain, nullptr);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ---------------------------------------------------------- MMA issuer
      constexpr uint32_t idesc = f8_idesc(2 * GBM, PBN);
      uint32_t stage = 0, phase = 0, gk = 0;
      bool alive = true;
      for (int t = cid; t < total_tiles && alive; t += ncl) {
        for (int kb = 0; kb < KB; ++kb, ++gk) {
          const uint32_t slot = gk % kPSlots, sphase = (gk / kPSlots) & 1;
          if (!mbar_wait<true>(smem_u32(&sm->slot_empty[slot]), sphase ^ 1, p.ctl, abort_flag) ||
              !mbar_wait(smem_u32(&sm->full[stage]), phase, p.ctl, abort_flag) ||
              !mbar_wait<true>(smem_u32(&sm->pair_full[stage]), phase, p.ctl, abort_flag)) {
            alive = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = smem_u32(smem + stage * kPStageBytes);
          const uint32_t d = tmem + slot * PBN;
#pragma unroll
          for (uint32_t k = 0; k < GBK / 32; ++k) {
            const uint64_t ad = smem_desc(st + 32 * k, 16, 1024, 2);
            const uint64_t bd = smem_desc(st + kGTileBytes + 32 * k, 16, 1024, 2);
            tc_mma_f8_pair(d, ad, bd, idesc, k != 0 ? 1u : 0u);
          }
          tc_commit_pair_mc(smem_u32(&sm->empty[stage]), 3);    // the stage is free in both CTAs
          tc_commit_pair_mc(smem_u32(&sm->slot_full[slot]), 3);  // both halves of the slot are ready
          if (++stage == kPStages) stage = 0, phase ^= 1;
        }
      }
      // all MMAs this thread issued are complete before TMEM is released
      tc_commit_pair_mc(smem_u32(&sm->mma_done), 1);
      KernelCtl drain = p.ctl;
      mbar_wait(smem_u32(&sm->mma_done), 0, drain, nullptr);
    } else if (lane == 0) {
      // ---------------------------------------------------------- relay (odd CTA)
      uint32_t stage = 0, phase = 0;
      const uint32_t leader_pair_full = mapa_shared(smem_u32(&sm->pair_full[0]), 0);
      bool alive = true;
      for (int t = cid; t < total_tiles && alive; t += ncl) {
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait(smem_u32(&sm->full[stage]), phase, p.ctl, abort_flag)) {
            alive = false;
            break;
          }
          mbar_arrive_cluster(leader_pair_full + stage * 8);
          if (++stage == kPStages) stage = 0, phase ^= 1;
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ promotion + store
    const int q = warp & 3;                    // TMEM lane quarter this warp may access
    const int h = (warp - kPromoWarp0) >> 2;   // column half of the 256-column slot
    const uint32_t t_lane = tmem + ((uint32_t)(q * 32) << 16) + h * 128;
    const uint32_t leader_slot_empty = mapa_shared(smem_u32(&sm->slot_empty[0]), 0);
    uint32_t gk = 0;
    bool alive = true;
    for (int t = cid; t < total_tiles && alive; t += ncl) {
      int m0, n0;
      tile_mn(t, m0, n0);
      const int64_t row = m0 + rank * GBM + q * 32 + lane;
      const int64_t col0 = n0 + h * 128;
      const bool row_ok = row < p.M, col_ok = col0 < p.N;
      const float* sa_row = p.sa + (row_ok ? row : p.M - 1) * KB;
      const float* sb_row = p.sb + (col_ok ? col0 / 128 : 0) * KB;
      float acc[128];
#pragma unroll
      for (int j = 0; j < 128; ++j) acc[j] = 0.f;
      // the scales of K block kb + kSP are requested while block kb is promoted
      float sa_q[kSP], sb_q[kSP];
#pragma unroll
      for (int i = 0; i < kSP; ++i) {
        sa_q[i] = i < KB ? __ldg(sa_row + i) : 0.f;
        sb_q[i] = i < KB ? __ldg(sb_row + i) : 0.f;
      }
      for (int kb0 = 0; kb0 < KB && alive; kb0 += kSP) {
#pragma unroll
        for (int i = 0; i < kSP; ++i) {
          const int kb = kb0 + i;
          if (kb >= KB || !alive) continue;
          const uint32_t slot = gk % kPSlots, sphase = (gk / kPSlots) & 1;
          const float sc = sa_q[i] * sb_q[i];
          if (kb + kSP < KB) sa_q[i] = __ldg(sa_row + kb + kSP), sb_q[i] = __ldg(sb_row + kb + kSP);
          if (!mbar_wait(smem_u32(&sm->slot_full[slot]), sphase, p.ctl, abort_flag)) {
            alive = false;
            continue;
          }
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < 8; ++c) {  // 16 columns per load
            uint32_t r[16];
            tmem_ld_32x32b_x16(t_lane + slot * PBN + c * 16, r);
            tmem_ld_wait();
            if (c == 7) {  // the slot's columns of this warp are all in registers
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive_cluster(leader_slot_empty + slot * 8);
            }
#pragma unroll
            for (int j = 0; j < 16; j += 2)  // two columns per instruction
              fma2(acc[16 * c + j], acc[16 * c + j + 1], __uint_as_float(r[j]), __uint_as_float(r[j + 1]), sc, sc);
          }
          ++gk;
        }
      }
      if (!alive || !row_ok || !col_ok) continue;
      if (p.c_dtype == Q4_BF16) {
        uint4* out = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.C) + row * p.N + col0);
#pragma unroll
        for (int v = 0; v < 16; ++v) {
          uint32_t w[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[8 * v + 2 * i], acc[8 * v + 2 * i + 1]);
            w[i] = *reinterpret_cast<const uint32_t*>(&b2);
          }
          out[v] = make_uint4(w[0], w[1], w[2], w[3]);
        }
      } else {
        float4* out = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.C) + row * p.N + col0);
#pragma unroll
        for (int v = 0; v < 32; ++v)
          out[v] = make_float4(acc[4 * v], acc[4 * v + 1], acc[4 * v + 2], acc[4 * v + 3]);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_barrier_sync();  // the pair's MMAs are complete in both CTAs
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kPSlots * PBN);
  }
  // no CTA leaves while its peer may still arrive on its barriers
  cluster_barrier_sync();
}

}  // namespace

q4_status launch_quant_fp8(const void* x, int dtype, int64_t rows, int64_t K, int block_rows,
                           uint8_t* codes, float* scales, cudaStream_t stream) {
  int* status = device_status_ptr();
  if (block_rows == 1) {
    const int64_t nblk = rows * (K / 128);
    const unsigned grid = (unsigned)std::min<int64_t>(ceil_div(nblk, kQThreads / 32),
                                                      (int64_t)num_sms() * 8);
    if (dtype == Q4_F32)
      return launch_pdl(fp8_act_quant_kernel<float>, grid, kQThreads, 0, stream,
                        static_cast<const float*>(x), rows, K, codes, scales, status);
    if (dtype == Q4_BF16)
      return launch_pdl(fp8_act_quant_kernel<__nv_bfloat16>, grid, kQThreads, 0, stream,
                        static_cast<const __nv_bfloat16*>(x), rows, K, codes, scales, status);
    return launch_pdl(fp8_act_quant_kernel<__half>, grid, kQThreads, 0, stream,
                      static_cast<const __half*>(x), rows, K, codes, scales, status);
  }
  const unsigned grid = (unsigned)((rows / 128) * (K / 128));
  if (dtype == Q4_F32)
    return launch_pdl(fp8_weight_quant_kernel<float>, grid, kQThreads, 0, stream,
                      static_cast<const float*>(x), K, codes, scales, status);
  if (dtype == Q4_BF16)
    return launch_pdl(fp8_weight_quant_kernel<__nv_bfloat16>, grid, kQThreads, 0, stream,
                      static_cast<const __nv_bfloat16*>(x), K, codes, scales, status);
  return launch_pdl(fp8_weight_quant_kernel<__half>, grid, kQThreads, 0, stream,
                    static_cast<const __half*>(x), K, codes, scales, status);
}

q4_status launch_fp8_gemm(const uint8_t* qa, const float* sa, const uint8_t* qb, const float* sb,
                          int64_t M, int64_t N, int64_t K, void* C, int c_dtype,
                          cudaStream_t stream) {
  CUtensorMap ta, tb;
  q4_status st;
  if ((st = make_tmap_2d_u8(&ta, qa, K, M, K, GBK, GBM, true)) != Q4_OK) return st;
  if ((st = make_tmap_2d_u8(&tb, qb, K, N, K, GBK, GBN, true)) != Q4_OK) return st;
  static int attr_done[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return Q4_ERR_CUDA;
  if (!attr_done[dev]) {
    Q4_CUDA_TRY(cudaFuncSetAttribute(fp8_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kGSmemBytes));
    attr_done[dev] = 1;
  }
  Fp8Params p;
  p.M = M, p.N = N, p.K = K;
  p.sa = sa, p.sb = sb, p.C = C, p.c_dtype = c_dtype;
  p.num_m = (int)ceil_div(M, GBM), p.num_n = (int)(N / GBN);
  p.ctl = KernelCtl{device_status_ptr(), wait_budget_ns()};
  if (M > GBM) {  // CTA pairs on 256 x 256 tiles
    static int pair_attr[64] = {0};
    static int max_pairs[64] = {0};
    if (!pair_attr[dev]) {
      Q4_CUDA_TRY(cudaFuncSetAttribute(fp8_gemm_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kPSmemBytes));
      pair_attr[dev] = 1;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kGThreads, 1, 1);
    cfg.dynamicSmemBytes = kPSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if (!max_pairs[dev]) {  // persistent: as many pairs as are resident at once
      int n = 0;
      cfg.gridDim = dim3((unsigned)(num_sms() / 2 * 2), 1, 1);
      if (cudaOccupancyMaxActiveClusters(&n, fp8_gemm_pair_kernel, &cfg) != cudaSuccess || n <= 0)
        n = num_sms() / 2;
      max_pairs[dev] = std::min(n, num_sms() / 2);
    }
    const int64_t ptiles = ceil_div(M, 2 * GBM) * ceil_div(N, 256);
    const int pairs = (int)std::max<int64_t>(1, std::min<int64_t>(ptiles, max_pairs[dev]));
    cfg.gridDim = dim3((unsigned)(2 * pairs), 1, 1);
    Q4_CUDA_TRY(cudaLaunchKernelEx(&cfg, fp8_gemm_pair_kernel, ta, tb, p));
    return Q4_OK;
  }
  const int tiles = p.num_m * p.num_n;
  const unsigned grid = (unsigned)std::min(tiles, num_sms());
  return launch_pdl(fp8_gemm_kernel, grid, kGThreads, kGSmemBytes, stream, ta, tb, p);
}

}  // namespace q4
