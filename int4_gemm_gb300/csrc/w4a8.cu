// W4A8: INT4 g128 weights, FP8 (E4M3) activations, FP8 tensor cores.
//
// "Low-bit inference for very large MoE", section "Kernels on different
// hardware", the W4A8 row: the INT4 weights are turned into FP8, the
// activations are quantized to FP8 and the product runs on the FP8 tensor
// cores.  Every INT4 value -8..7 is an E4M3 value, so the conversion is
// exact, and the FP16 group scale (one per 128 along K) lines up with the
// 128-wide K blocks of the block-promoted FP8 product:
//   C[m, n] = sum_kb sa[m, kb] * s16[n, kb] * sum_{k in kb} qa[m, k] * q[n, k]
// (activations from quantize_fp8_blockwise with (1, 128) blocks).
//
// The kernel is the block-promoted FP8 GEMM with the B operand kept 4-bit in
// HBM (one CTA per SM, persistent over 128 x 128 tiles in bands of 32 M tiles):
//   warp 0      TMA producer: the A tile (E4M3, 128-byte swizzle) and the INT4
//               tile (128 rows x 64 bytes, unswizzled) of each K block into a
//               5-stage ring, and the K block's 128 weight scales (FP32, from
//               the [K/128, N] copy made by w4a8_weight_scales) into a 16-deep
//               ring of scale buffers;
//   warps 2, 3  converters: each thread expands eight 16-byte chunks of INT4
//               codes to E4M3 bytes (a 16-entry byte-permute table), a warp
//               reading eight whole rows at a time, and writes them in the
//               128-byte-swizzled layout the MMA reads;
//   warp 1      MMA issuer: four tcgen05.mma kind::f8f6f4 per K block into one
//               of four 128-column TMEM slots;
//   warps 4..11 promotion: slot * s16[n, kb] * sa[m, kb] into 64 FP32 registers
//               per thread; the tile's rows are stored after its last K block.
// A scale buffer is refilled only after the promotion of the K block that last
// used it has finished: the producer of K block g waits for the MMAs of block
// g - 5 to complete, which were issued after the promotion warps read the
// buffers of block g - 9 and released its TMEM slot.
#include "common.cuh"
#include "internal.h"

#include <algorithm>

namespace q4 {
namespace {

constexpr int WBM = 128, WBN = 128, WBK = 128;
constexpr int kWStages = 5;
constexpr int kWSlots = 4;                            // TMEM accumulator slots, 128 columns each
constexpr int kScaleBufs = 16;                        // weight-scale buffers, one K block each
constexpr int kBandM = 32;                            // M tiles per band of the tile order
constexpr int kSP = 4;                                // K blocks of scale prefetch in registers
constexpr uint32_t kATileBytes = WBM * WBK;           // E4M3 A tile
constexpr uint32_t kBTileBytes = WBN * WBK;           // E4M3 B tile after conversion
constexpr uint32_t kBCodeBytes = WBN * WBK / 2;       // INT4 B tile as loaded
constexpr uint32_t kWStageBytes = kATileBytes + kBTileBytes + kBCodeBytes;
constexpr uint32_t kScaleBufBytes = WBN * sizeof(float);
constexpr int kConvWarp0 = 2, kConvWarps = 2;
constexpr int kPromWarp0 = 4, kPromWarps = 8;
constexpr int kWThreads = (kPromWarp0 + kPromWarps) * 32;
constexpr uint32_t kWSmemBytes =
    kWStages * kWStageBytes + kScaleBufs * kScaleBufBytes + 1024 /*align*/ + 512 /*barriers*/;
static_assert(kWStageBytes % 1024 == 0, "stages keep the 1024-byte swizzle alignment");
static_assert(kWSmemBytes <= 232448, "shared memory");
static_assert(kWSlots * WBN <= 512, "TMEM columns");
constexpr int kConvItems = WBN * 4 / (kConvWarps * 32);  // 16-byte code chunks per converter thread
static_assert(kConvItems * kConvWarps * 32 == WBN * 4, "the converters cover the B tile");

struct WSmem {
  uint64_t full[kWStages];      // A tile and INT4 tile landed
  uint64_t b_ready[kWStages];   // B tile converted (one arrival per converter warp)
  uint64_t empty[kWStages];     // the stage's MMAs are done
  uint64_t slot_full[kWSlots];
  uint64_t slot_empty[kWSlots];
  uint64_t sc_full[kScaleBufs];  // a K block's weight scales landed
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(WSmem) <= 512, "barrier block");

struct W4a8Params {
  int64_t M, N, K;
  const float* sa;   // [M, K / 128]
  const float* wsc;  // [K / 128, N]
  void* C;           // [M, N]
  int c_dtype;
  int num_m, num_n;
  KernelCtl ctl;
};

// tcgen05.mma kind::f8f6f4 descriptor: FP32 accumulator (bits 4-5 = 1), A and B
// E4M3 (format 0), both K-major, N / 8 in bits 17-22, M / 16 in bits 24-28.
constexpr uint32_t kIdesc = (1u << 4) | ((uint32_t)(WBN >> 3) << 17) | ((uint32_t)(WBM >> 4) << 24);

__device__ __forceinline__ void mma_e4m3(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(kIdesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// E4M3 bytes of the eight two's complement INT4 nibbles of w (nibble j ->
// byte j of the pair).  The low three bits of a nibble index the byte tables
// of q = 0..7 and of q = -8..-1; a byte permute in sign-replicate mode turns
// each nibble's sign bit into a byte mask that picks between them.
__device__ __forceinline__ uint2 int4x8_to_e4m3(uint32_t w) {
  constexpr uint32_t kPos0 = 0x44403800u;  // 0, 1, 2, 3  -> 0x00 0x38 0x40 0x44
  constexpr uint32_t kPos1 = 0x4E4C4A48u;  // 4, 5, 6, 7  -> 0x48 0x4A 0x4C 0x4E
  constexpr uint32_t kNeg0 = 0xCACCCED0u;  // -8, -7, -6, -5 -> 0xD0 0xCE 0xCC 0xCA
  constexpr uint32_t kNeg1 = 0xB8C0C4C8u;  // -4, -3, -2, -1 -> 0xC8 0xC4 0xC0 0xB8
  const uint32_t wl = w << 4;  // the sign bit of nibble 2i at bit 7 of byte i
  uint2 r;
  uint32_t sel = w & 0x7777u;
  uint32_t msk = prmt(wl, w, 0xD9C8u);  // nibbles 0..3: bytes 0, 4, 1, 5, sign-replicated
  r.x = (prmt(kPos0, kPos1, sel) & ~msk) | (prmt(kNeg0, kNeg1, sel) & msk);
  sel = (w >> 16) & 0x7777u;
  msk = prmt(wl, w, 0xFBEAu);  // nibbles 4..7: bytes 2, 6, 3, 7, sign-replicated
  r.y = (prmt(kPos0, kPos1, sel) & ~msk) | (prmt(kNeg0, kNeg1, sel) & msk);
  return r;
}

__global__ void __launch_bounds__(kWThreads, 1)
    w4a8_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a,
                     const __grid_constant__ CUtensorMap tmap_w, const W4a8Params p) {
  extern __shared__ uint8_t smem_raw[];
  pdl_wait();  // operands and scales may come from the previous kernel
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  float* sbuf = reinterpret_cast<float*>(smem + kWStages * kWStageBytes);
  WSmem* sm = reinterpret_cast<WSmem*>(smem + kWStages * kWStageBytes + kScaleBufs * kScaleBufBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KB = (int)(p.K / WBK);
  const int total_tiles = p.num_m * p.num_n;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kWStages; ++s) {
      mbar_init(smem_u32(&sm->full[s]), 1);
      mbar_init(smem_u32(&sm->b_ready[s]), kConvWarps);
      mbar_init(smem_u32(&sm->empty[s]), 1);
    }
    for (int s = 0; s < kWSlots; ++s) {
      mbar_init(smem_u32(&sm->slot_full[s]), 1);
      mbar_init(smem_u32(&sm->slot_empty[s]), kPromWarps);
    }
    for (int b = 0; b < kScaleBufs; ++b) mbar_init(smem_u32(&sm->sc_full[b]), 1);
    mbar_init(smem_u32(&sm->mma_done), 1);
    sm->abort = 0;
    fence_mbar_init();
    prefetch_tmap(&tmap_a);
    prefetch_tmap(&tmap_w);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&sm->tmem_base), kWSlots * WBN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm->tmem_base;
  volatile int* abort_flag = &sm->abort;
  // bands of kBandM M tiles (a 33.5 MB slice of A at K = 8192 stays in L2), M
  // fastest inside a band
  auto tile_mn = [&](int t, int& m0, int& n0) {
    const int band_tiles = kBandM * p.num_n;
    const int band = t / band_tiles, r = t - band * band_tiles;
    const int gm = min(kBandM, p.num_m - band * kBandM);
    m0 = (band * kBandM + r % gm) * WBM;
    n0 = (r / gm) * WBN;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    uint32_t stage = 0, phase = 0, gk = 0;
    int issued[kWStages];
    uint32_t issued_phase[kWStages];
    for (int s = 0; s < kWStages; ++s) issued[s] = 0, issued_phase[s] = 0;
    bool alive = true;
    for (int t = blockIdx.x; t < total_tiles && alive; t += gridDim.x) {
      int m0, n0;
      tile_mn(t, m0, n0);
      for (int kb = 0; kb < KB; ++kb, ++gk) {
        if (!mbar_wait(smem_u32(&sm->empty[stage]), phase ^ 1, p.ctl, abort_flag)) {
          alive = false;
          break;
        }
        uint8_t* st = smem + stage * kWStageBytes;
        if (lane == 0) {
          const uint32_t full = smem_u32(&sm->full[stage]);
          mbar_arrive_expect_tx(full, kATileBytes + kBCodeBytes);
          tma_load_2d(smem_u32(st), &tmap_a, kb * WBK, m0, full);
          tma_load_2d(smem_u32(st + kATileBytes + kBTileBytes), &tmap_w, kb * (WBK / 2), n0, full);
          const uint32_t b = gk % kScaleBufs;
          const uint32_t scb = smem_u32(&sm->sc_full[b]);
          mbar_arrive_expect_tx(scb, kScaleBufBytes);
          bulk_load(smem_u32(sbuf + b * WBN), p.wsc + (int64_t)kb * p.N + n0, kScaleBufBytes, scb);
        }
        issued[stage] = 1;
        issued_phase[stage] = phase;
        if (++stage == kWStages) stage = 0, phase ^= 1;
      }
    }
    // drain: every copy this warp issued has landed before the CTA exits (the
    // scale copies of the last kScaleBufs K blocks; older ones were waited for
    // by the promotion warps or by this loop's stage waits)
    if (lane == 0) {
      KernelCtl drain = p.ctl;
      for (int s = 0; s < kWStages; ++s)
        if (issued[s]) mbar_wait(smem_u32(&sm->full[s]), issued_phase[s], drain, nullptr);
      for (uint32_t g = gk > (uint32_t)kScaleBufs ? gk - kScaleBufs : 0u; g < gk; ++g)
        mbar_wait(smem_u32(&sm->sc_full[g % kScaleBufs]), (g / kScaleBufs) & 1, drain, nullptr);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, gk = 0;
      bool alive = true;
      for (int t = blockIdx.x; t < total_tiles && alive; t += gridDim.x) {
        for (int kb = 0; kb < KB; ++kb, ++gk) {
          const uint32_t slot = gk % kWSlots, sphase = (gk / kWSlots) & 1;
          // b_ready implies full: the converters waited for the stage's copies
          if (!mbar_wait(smem_u32(&sm->slot_empty[slot]), sphase ^ 1, p.ctl, abort_flag) ||
              !mbar_wait(smem_u32(&sm->b_ready[stage]), phase, p.ctl, abort_flag)) {
            alive = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = smem_u32(smem + stage * kWStageBytes);
          const uint32_t d = tmem + slot * WBN;
#pragma unroll
          for (uint32_t k = 0; k < WBK / 32; ++k)
            mma_e4m3(d, smem_desc(st + 32 * k, 16, 1024, 2),
                     smem_desc(st + kATileBytes + 32 * k, 16, 1024, 2), k != 0 ? 1u : 0u);
          tc_commit(smem_u32(&sm->empty[stage]));
          tc_commit(smem_u32(&sm->slot_full[slot]));
          if (++stage == kWStages) stage = 0, phase ^= 1;
        }
      }
      tc_commit(smem_u32(&sm->mma_done));
      KernelCtl drain = p.ctl;
      mbar_wait(smem_u32(&sm->mma_done), 0, drain, nullptr);
    }
    __syncwarp();
  } else if (warp < kPromWarp0) {
    // ------------------------------------------------------------ converters
    // item it = (row r = it / 4, 16-byte code chunk i = it % 4) of the K block;
    // the converter threads take items it = 64 k + 32 c + lane, so that a
    // warp's 32 loads cover 8 whole rows (512 contiguous bytes: no bank
    // conflict).  Code chunk i becomes output chunks 2i and 2i + 1 of row r,
    // stored at r * 128 + ((j ^ (r % 8)) * 16): the 128-byte swizzle the
    // MMA's shared-memory descriptors describe
    const int cw = warp - kConvWarp0;
    uint32_t stage = 0, phase = 0;
    bool alive = true;
    for (int t = blockIdx.x; t < total_tiles && alive; t += gridDim.x) {
      for (int kb = 0; kb < KB; ++kb) {
        if (!mbar_wait(smem_u32(&sm->full[stage]), phase, p.ctl, abort_flag)) {
          alive = false;
          break;
        }
        uint8_t* st = smem + stage * kWStageBytes;
        const uint8_t* src = st + kATileBytes + kBTileBytes;
        uint8_t* dst = st + kATileBytes;
#pragma unroll
        for (int k = 0; k < kConvItems; ++k) {
          const int it = k * kConvWarps * 32 + cw * 32 + lane;
          const int r = it >> 2, i = it & 3;
          const uint4 w = *reinterpret_cast<const uint4*>(src + r * 64 + i * 16);
          const uint2 e0 = int4x8_to_e4m3(w.x), e1 = int4x8_to_e4m3(w.y);
          const uint2 e2 = int4x8_to_e4m3(w.z), e3 = int4x8_to_e4m3(w.w);
          *reinterpret_cast<uint4*>(dst + r * 128 + (((2 * i) ^ (r & 7)) << 4)) =
              make_uint4(e0.x, e0.y, e1.x, e1.y);
          *reinterpret_cast<uint4*>(dst + r * 128 + (((2 * i + 1) ^ (r & 7)) << 4)) =
              make_uint4(e2.x, e2.y, e3.x, e3.y);
        }
        fence_proxy_async_smem();  // the tensor cores read what these threads wrote
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sm->b_ready[stage]));
        if (++stage == kWStages) stage = 0, phase ^= 1;
      }
    }
  } else {
    // ------------------------------------------------------------ promotion + store
    const int q = warp & 3;                   // TMEM lane quarter this warp may access
    const int h = (warp - kPromWarp0) >> 2;   // column half of the slot
    const uint32_t t_lane = tmem + ((uint32_t)(q * 32) << 16) + h * 64;
    uint32_t gk = 0;
    bool alive = true;
    for (int t = blockIdx.x; t < total_tiles && alive; t += gridDim.x) {
      int m0, n0;
      tile_mn(t, m0, n0);
      const int64_t row = m0 + q * 32 + lane;
      const bool row_ok = row < p.M;
      const float* sa_row = p.sa + (row_ok ? row : p.M - 1) * KB;
      float acc[64];
#pragma unroll
      for (int j = 0; j < 64; ++j) acc[j] = 0.f;
      // the scale of K block kb + kSP is requested while block kb is
      // promoted: a K block takes a few hundred ns, an L2 load about a us
      float sa_q[kSP];
#pragma unroll
      for (int i = 0; i < kSP; ++i) sa_q[i] = i < KB ? __ldg(sa_row + i) : 0.f;
      for (int kb0 = 0; kb0 < KB && alive; kb0 += kSP) {
#pragma unroll
        for (int i = 0; i < kSP; ++i) {
          const int kb = kb0 + i;
          if (kb >= KB || !alive) continue;
          const uint32_t slot = gk % kWSlots, sphase = (gk / kWSlots) & 1;
          const uint32_t b = gk % kScaleBufs;
          const float sa_k = sa_q[i];
          if (kb + kSP < KB) sa_q[i] = __ldg(sa_row + kb + kSP);
          if (!mbar_wait(smem_u32(&sm->slot_full[slot]), sphase, p.ctl, abort_flag) ||
              !mbar_wait(smem_u32(&sm->sc_full[b]), (gk / kScaleBufs) & 1, p.ctl, abort_flag)) {
            alive = false;
            continue;
          }
          tc_fence_after();
          uint32_t r0[32], r1[32];
          tmem_ld_32x32b_x32(t_lane + slot * WBN, r0);
          tmem_ld_32x32b_x32(t_lane + slot * WBN + 32, r1);
          tmem_ld_wait();
          const float4* sw = reinterpret_cast<const float4*>(sbuf + b * WBN + h * 64);
#pragma unroll
          for (int v = 0; v < 8; ++v) {
            const float4 s0 = sw[v], s1 = sw[8 + v];
            acc[4 * v] = fmaf(__uint_as_float(r0[4 * v]) * s0.x, sa_k, acc[4 * v]);
            acc[4 * v + 1] = fmaf(__uint_as_float(r0[4 * v + 1]) * s0.y, sa_k, acc[4 * v + 1]);
            acc[4 * v + 2] = fmaf(__uint_as_float(r0[4 * v + 2]) * s0.z, sa_k, acc[4 * v + 2]);
            acc[4 * v + 3] = fmaf(__uint_as_float(r0[4 * v + 3]) * s0.w, sa_k, acc[4 * v + 3]);
            acc[32 + 4 * v] = fmaf(__uint_as_float(r1[4 * v]) * s1.x, sa_k, acc[32 + 4 * v]);
            acc[32 + 4 * v + 1] = fmaf(__uint_as_float(r1[4 * v + 1]) * s1.y, sa_k, acc[32 + 4 * v + 1]);
            acc[32 + 4 * v + 2] = fmaf(__uint_as_float(r1[4 * v + 2]) * s1.z, sa_k, acc[32 + 4 * v + 2]);
            acc[32 + 4 * v + 3] = fmaf(__uint_as_float(r1[4 * v + 3]) * s1.w, sa_k, acc[32 + 4 * v + 3]);
          }
          // the slot goes back after the scale buffer has been read (its refill
          // waits, through the MMA, for this arrival)
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&sm->slot_empty[slot]));
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
    tmem_dealloc(tmem, kWSlots * WBN);
  }
}

// ------------------------------------------------------------------ CTA pairs
// For M > 128: the same pipeline on 256 x 256 tiles with the 2-SM MMA
// (tcgen05.mma.cta_group::2.kind::f8f6f4, 256 x 256 x 32).  CTA rank r copies
// A rows m0 + 128 r .. and the INT4 codes of B rows n0 + 128 r .. of each K
// block, its converters expand its half of B, and the even CTA issues the
// MMAs once its own converted stage is ready and the odd CTA's relay lane has
// arrived on its `pair_full`.  Both CTAs copy the K block's 256 weight scales
// (the tile's columns); two 256-column TMEM slots; each promotion warp owns a
// lane quarter x 128 columns (128 FP32 registers per thread) and arrives on
// the even CTA's `slot_empty` (16 arrivals) after it has read the slot and the
// scale buffer.  A scale buffer is refilled (K block g, buffer g % 16) after
// the MMAs of block g - 5 completed in both CTAs, which were issued after
// every promotion of block g - 7 had read its buffer.
constexpr int kPStages = 5;
constexpr int kPSlots = 2;
constexpr int PBN = 256;                                   // pair tile N
constexpr uint32_t kPScaleBufBytes = PBN * sizeof(float);  // one K block's tile columns
constexpr uint32_t kPSmemBytes =
    kPStages * kWStageBytes + kScaleBufs * kPScaleBufBytes + 1024 /*align*/ + 512 /*barriers*/;
static_assert(kPSmemBytes <= 232448, "shared memory");
static_assert(kPSlots * PBN <= 512, "TMEM columns");

struct PSmem {
  uint64_t full[kPStages];       // this CTA's A tile and INT4 tile landed
  uint64_t b_ready[kPStages];    // this CTA's half of B converted
  uint64_t pair_full[kPStages];  // even CTA: the odd CTA's stage is converted (relay)
  uint64_t empty[kPStages];      // the stage's MMAs are done (both CTAs)
  uint64_t slot_full[kPSlots];
  uint64_t slot_empty[kPSlots];  // even CTA: every promotion warp of the pair is done
  uint64_t sc_full[kScaleBufs];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(PSmem) <= 512, "barrier block");

constexpr uint32_t kPIdesc = (1u << 4) | ((uint32_t)(PBN >> 3) << 17) | ((uint32_t)((2 * WBM) >> 4) << 24);

__device__ __forceinline__ void mma_e4m3_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                              uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(kPIdesc), "r"(accumulate)
      : "memory");
}

__global__ void __launch_bounds__(kWThreads, 1)
    w4a8_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmap_a,
                          const __grid_constant__ CUtensorMap tmap_w, const W4a8Params p) {
  extern __shared__ uint8_t smem_raw[];
  pdl_wait();  // operands and scales may come from the previous kernel
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  float* sbuf = reinterpret_cast<float*>(smem + kPStages * kWStageBytes);
  PSmem* sm = reinterpret_cast<PSmem*>(smem + kPStages * kWStageBytes + kScaleBufs * kPScaleBufBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = (int)cluster_ctarank();  // 0: issues the pair's MMAs
  const int cid = blockIdx.x >> 1, ncl = gridDim.x >> 1;
  const int KB = (int)(p.K / WBK);
  const int num_pm = (int)((p.M + 2 * WBM - 1) / (2 * WBM)), num_pn = (int)((p.N + PBN - 1) / PBN);
  const int total_tiles = num_pm * num_pn;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPStages; ++s) {
      mbar_init(smem_u32(&sm->full[s]), 1);
      mbar_init(smem_u32(&sm->b_ready[s]), kConvWarps);
      mbar_init(smem_u32(&sm->pair_full[s]), 1);
      mbar_init(smem_u32(&sm->empty[s]), 1);
    }
    for (int s = 0; s < kPSlots; ++s) {
      mbar_init(smem_u32(&sm->slot_full[s]), 1);
      mbar_init(smem_u32(&sm->slot_empty[s]), 2 * kPromWarps);
    }
    for (int b = 0; b < kScaleBufs; ++b) mbar_init(smem_u32(&sm->sc_full[b]), 1);
    mbar_init(smem_u32(&sm->mma_done), 1);
    sm->abort = 0;
    fence_mbar_init();
    prefetch_tmap(&tmap_a);
    prefetch_tmap(&tmap_w);
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
  auto tile_mn = [&](int t, int& m0, int& n0) {  // pair tiles in bands of kBandM / 2
    constexpr int kBand = kBandM / 2;
    const int band_tiles = kBand * num_pn;
    const int band = t / band_tiles, r = t - band * band_tiles;
    const int gm = min(kBand, num_pm - band * kBand);
    m0 = (band * kBand + r % gm) * 2 * WBM;
    n0 = (r / gm) * PBN;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    uint32_t stage = 0, phase = 0, gk = 0;
    int issued[kPStages];
    uint32_t issued_phase[kPStages];
    for (int s = 0; s < kPStages; ++s) issued[s] = 0, issued_phase[s] = 0;
    bool alive = true;
    for (int t = cid; t < total_tiles && alive; t += ncl) {
      int m0, n0;
      tile_mn(t, m0, n0);
      // the tile's weight-scale columns (a tile past N by 128 columns copies 128)
      const uint32_t sc_bytes = (uint32_t)min((int64_t)PBN, p.N - n0) * 4u;
      for (int kb = 0; kb < KB; ++kb, ++gk) {
        if (!mbar_wait(smem_u32(&sm->empty[stage]), phase ^ 1, p.ctl, abort_flag)) {
          alive = false;
          break;
        }
        uint8_t* st = smem + stage * kWStageBytes;
        if (lane == 0) {
          const uint32_t full = smem_u32(&sm->full[stage]);
          mbar_arrive_expect_tx(full, kATileBytes + kBCodeBytes);
          tma_load_2d(smem_u32(st), &tmap_a, kb * WBK, m0 + rank * WBM, full);
          tma_load_2d(smem_u32(st + kATileBytes + kBTileBytes), &tmap_w, kb * (WBK / 2),
                      n0 + rank * (PBN / 2), full);
          const uint32_t b = gk % kScaleBufs;
          const uint32_t scb = smem_u32(&sm->sc_full[b]);
          mbar_arrive_expect_tx(scb, sc_bytes);
          bulk_load(smem_u32(sbuf + b * PBN), p.wsc + (int64_t)kb * p.N + n0, sc_bytes, scb);
        }
        issued[stage] = 1;
        issued_phase[stage] = phase;
        if (++stage == kPStages) stage = 0, phase ^= 1;
      }
    }
    if (lane == 0) {
      KernelCtl drain = p.ctl;
      for (int s = 0; s < kPStages; ++s)
        if (issued[s]) mbar_wait(smem_u32(&sm->full[s]), issued_phase[s], drain, nullptr);
      for (uint32_t g = gk > (uint32_t)kScaleBufs ? gk - kScaleBufs : 0u; g < gk; ++g)
        mbar_wait(smem_u32(&sm->sc_full[g % kScaleBufs]), (g / kScaleBufs) & 1, drain, nullptr);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ---------------------------------------------------------- MMA issuer
      uint32_t stage = 0, phase = 0, gk = 0;
      bool alive = true;
      for (int t = cid; t < total_tiles && alive; t += ncl) {
        for (int kb = 0; kb < KB; ++kb, ++gk) {
          const uint32_t slot = gk % kPSlots, sphase = (gk / kPSlots) & 1;
          // b_ready implies full: the converters waited for the stage's copies
          if (!mbar_wait<true>(smem_u32(&sm->slot_empty[slot]), sphase ^ 1, p.ctl, abort_flag) ||
              !mbar_wait(smem_u32(&sm->b_ready[stage]), phase, p.ctl, abort_flag) ||
              !mbar_wait<true>(smem_u32(&sm->pair_full[stage]), phase, p.ctl, abort_flag)) {
            alive = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = smem_u32(smem + stage * kWStageBytes);
          const uint32_t d = tmem + slot * PBN;
#pragma unroll
          for (uint32_t k = 0; k < WBK / 32; ++k)
            mma_e4m3_pair(d, smem_desc(st + 32 * k, 16, 1024, 2),
                          smem_desc(st + kATileBytes + 32 * k, 16, 1024, 2), k != 0 ? 1u : 0u);
          tc_commit_pair_mc(smem_u32(&sm->empty[stage]), 3);
          tc_commit_pair_mc(smem_u32(&sm->slot_full[slot]), 3);
          if (++stage == kPStages) stage = 0, phase ^= 1;
        }
      }
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
          if (!mbar_wait(smem_u32(&sm->b_ready[stage]), phase, p.ctl, abort_flag)) {
            alive = false;
            break;
          }
          mbar_arrive_cluster(leader_pair_full + stage * 8);
          if (++stage == kPStages) stage = 0, phase ^= 1;
        }
      }
    }
    __syncwarp();
  } else if (warp < kPromWarp0) {
    // ------------------------------------------------------------ converters
    // the same item order and swizzle as the single-CTA kernel, on this CTA's
    // 128 rows of the tile's B
    const int cw = warp - kConvWarp0;
    uint32_t stage = 0, phase = 0;
    bool alive = true;
    for (int t = cid; t < total_tiles && alive; t += ncl) {
      for (int kb = 0; kb < KB; ++kb) {
        if (!mbar_wait(smem_u32(&sm->full[stage]), phase, p.ctl, abort_flag)) {
          alive = false;
          break;
        }
        uint8_t* st = smem + stage * kWStageBytes;
        const uint8_t* src = st + kATileBytes + kBTileBytes;
        uint8_t* dst = st + kATileBytes;
#pragma unroll
        for (int k = 0; k < kConvItems; ++k) {
          const int it = k * kConvWarps * 32 + cw * 32 + lane;
          const int r = it >> 2, i = it & 3;
          const uint4 w = *reinterpret_cast<const uint4*>(src + r * 64 + i * 16);
          const uint2 e0 = int4x8_to_e4m3(w.x), e1 = int4x8_to_e4m3(w.y);
          const uint2 e2 = int4x8_to_e4m3(w.z), e3 = int4x8_to_e4m3(w.w);
          *reinterpret_cast<uint4*>(dst + r * 128 + (((2 * i) ^ (r & 7)) << 4)) =
              make_uint4(e0.x, e0.y, e1.x, e1.y);
          *reinterpret_cast<uint4*>(dst + r * 128 + (((2 * i + 1) ^ (r & 7)) << 4)) =
              make_uint4(e2.x, e2.y, e3.x, e3.y);
        }
        fence_proxy_async_smem();  // the tensor cores read what these threads wrote
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sm->b_ready[stage]));
        if (++stage == kPStages) stage = 0, phase ^= 1;
      }
    }
  } else {
    // ------------------------------------------------------------ promotion + store
    const int q = warp & 3;                   // TMEM lane quarter this warp may access
    const int h = (warp - kPromWarp0) >> 2;   // column half of the 256-column slot
    const uint32_t t_lane = tmem + ((uint32_t)(q * 32) << 16) + h * 128;
    const uint32_t leader_slot_empty = mapa_shared(smem_u32(&sm->slot_empty[0]), 0);
    uint32_t gk = 0;
    bool alive = true;
    for (int t = cid; t < total_tiles && alive; t += ncl) {
      int m0, n0;
      tile_mn(t, m0, n0);
      const int64_t row = m0 + rank * WBM + q * 32 + lane;
      const int64_t col0 = n0 + h * 128;
      const bool row_ok = row < p.M, col_ok = col0 < p.N;
      const float* sa_row = p.sa + (row_ok ? row : p.M - 1) * KB;
      float acc[128];
#pragma unroll
      for (int j = 0; j < 128; ++j) acc[j] = 0.f;
      float sa_q[kSP];
#pragma unroll
      for (int i = 0; i < kSP; ++i) sa_q[i] = i < KB ? __ldg(sa_row + i) : 0.f;
      for (int kb0 = 0; kb0 < KB && alive; kb0 += kSP) {
#pragma unroll
        for (int i = 0; i < kSP; ++i) {
          const int kb = kb0 + i;
          if (kb >= KB || !alive) continue;
          const uint32_t slot = gk % kPSlots, sphase = (gk / kPSlots) & 1;
          const uint32_t b = gk % kScaleBufs;
          const float sa_k = sa_q[i];
          if (kb + kSP < KB) sa_q[i] = __ldg(sa_row + kb + kSP);
          if (!mbar_wait(smem_u32(&sm->slot_full[slot]), sphase, p.ctl, abort_flag) ||
              !mbar_wait(smem_u32(&sm->sc_full[b]), (gk / kScaleBufs) & 1, p.ctl, abort_flag)) {
            alive = false;
            continue;
          }
          tc_fence_after();
          const float4* sw = reinterpret_cast<const float4*>(sbuf + b * PBN + h * 128);
#pragma unroll
          for (int c = 0; c < 16; ++c) {  // 8 columns per load
            uint32_t r[8];
            tmem_ld_32x32b_x8(t_lane + slot * PBN + c * 8, r);
            tmem_ld_wait();
#pragma unroll
            for (int v = 0; v < 2; ++v) {  // two columns per instruction
              const float4 s4 = sw[2 * c + v];  // stale past N (not stored then)
              float t0, t1, t2, t3;
              mul2(t0, t1, __uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]), s4.x, s4.y);
              mul2(t2, t3, __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]), s4.z, s4.w);
              fma2(acc[8 * c + 4 * v], acc[8 * c + 4 * v + 1], t0, t1, sa_k, sa_k);
              fma2(acc[8 * c + 4 * v + 2], acc[8 * c + 4 * v + 3], t2, t3, sa_k, sa_k);
            }
          }
          // the slot and the scale buffer go back together (their refills wait,
          // through the MMA, for this arrival)
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(leader_slot_empty + slot * 8);
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

// FP16 scale bits [N, KB] -> FP32 [KB, N] (the layout whose K-block rows the
// GEMM copies whole).
__global__ void __launch_bounds__(256)
    w4a8_scales_kernel(const uint16_t* __restrict__ s16, int64_t N, int64_t KB, float* __restrict__ out) {
  pdl_wait();
  const int64_t n_all = N * KB;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_all;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t kb = i / N, n = i - kb * N;
    out[i] = __half2float(__ushort_as_half(__ldg(s16 + n * KB + kb)));
  }
}

}  // namespace

q4_status launch_w4a8_scales(const uint16_t* s16, int64_t N, int64_t KB, float* out,
                             cudaStream_t stream) {
  const unsigned grid = (unsigned)std::min<int64_t>(ceil_div(N * KB, 256), (int64_t)num_sms() * 8);
  return launch_pdl(w4a8_scales_kernel, grid, 256, 0, stream, s16, N, KB, out);
}

q4_status launch_w4a8_gemm(const uint8_t* qa, const float* sa, const uint8_t* wq, const float* wsc,
                           int64_t M, int64_t N, int64_t K, void* C, int c_dtype,
                           cudaStream_t stream) {
  CUtensorMap ta, tw;
  q4_status st;
  if ((st = make_tmap_2d_u8(&ta, qa, K, M, K, WBK, WBM, true)) != Q4_OK) return st;
  if ((st = make_tmap_2d_u8(&tw, wq, K / 2, N, K / 2, WBK / 2, WBN, false)) != Q4_OK) return st;
  static int attr_done[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return Q4_ERR_CUDA;
  if (!attr_done[dev]) {
    Q4_CUDA_TRY(cudaFuncSetAttribute(w4a8_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kWSmemBytes));
    attr_done[dev] = 1;
  }
  W4a8Params p;
  p.M = M, p.N = N, p.K = K;
  p.sa = sa, p.wsc = wsc, p.C = C, p.c_dtype = c_dtype;
  p.num_m = (int)ceil_div(M, WBM), p.num_n = (int)(N / WBN);
  p.ctl = KernelCtl{device_status_ptr(), wait_budget_ns()};
  if (M > WBM) {  // CTA pairs on 256 x 256 tiles
    static int pair_attr[64] = {0};
    static int max_pairs[64] = {0};
    if (!pair_attr[dev]) {
      Q4_CUDA_TRY(cudaFuncSetAttribute(w4a8_gemm_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kPSmemBytes));
      pair_attr[dev] = 1;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kWThreads, 1, 1);
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
      if (cudaOccupancyMaxActiveClusters(&n, w4a8_gemm_pair_kernel, &cfg) != cudaSuccess || n <= 0)
        n = num_sms() / 2;
      max_pairs[dev] = std::min(n, num_sms() / 2);
    }
    const int64_t ptiles = ceil_div(M, 2 * WBM) * ceil_div(N, 256);
    const int pairs = (int)std::max<int64_t>(1, std::min<int64_t>(ptiles, max_pairs[dev]));
    cfg.gridDim = dim3((unsigned)(2 * pairs), 1, 1);
    Q4_CUDA_TRY(cudaLaunchKernelEx(&cfg, w4a8_gemm_pair_kernel, ta, tw, p));
    return Q4_OK;
  }
  const int tiles = p.num_m * p.num_n;
  const unsigned grid = (unsigned)std::min(tiles, num_sms());
  return launch_pdl(w4a8_gemm_kernel, grid, kWThreads, kWSmemBytes, stream, ta, tw, p);
}

}  // namespace q4
