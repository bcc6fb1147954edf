// Block-scaled 4-bit quantizers: NVFP4 (tensor amax + per-16 E4M3 scales),
// MXFP4 (per-32 E8M0 scales) and INT4 g128 (per-128 FP16 scales).
//
// Every element is loaded once with 128-bit loads, sixteen per thread; the
// threads that share a scale block reduce its amax with warp shuffles; codes
// leave as packed 64-bit words (16 codes per thread).  The arithmetic follows "Quantization in
// deployment", section "Fake quantization" (fp4, mxfp4, nvfp4) and "Low-bit
// inference for very large MoE", section "Why quantization-aware training"
// (fake_int4): float32, IEEE-rounded divisions, E2M1 ties to the smaller
// magnitude.  The FP4 kernels reach the same codes without a per-element
// division (the argument is at each kernel).
#include "common.cuh"
#include "internal.h"
#include "quant_device.cuh"

#include <algorithm>

namespace q4 {
namespace {

constexpr int kThreads = 256;

// A launch covers rows [row0, row0 + units / nblk) of the tensor, one unit of
// 16 elements per thread (nblk units per row, units < 2^32).  The row of unit
// u comes from a multiply-high by a precomputed constant instead of a
// division (Granlund and Montgomery, "Division by invariant integers using
// multiplication", 1994, unsigned case).
struct UnitMap {
  uint32_t units;  // units in this launch
  uint32_t nblk;   // units per row (K / 16)
  uint32_t magic;  // 2^32 (2^l - nblk) / nblk + 1, l = ceil(log2 nblk)
  uint32_t shift;  // l - 1 (unused when nblk == 1)
  int64_t row0;    // first row of this launch
  __device__ __forceinline__ uint32_t row_of(uint32_t u) const {
    if (nblk == 1) return u;
    const uint32_t t = __umulhi(magic, u);
    return (t + ((u - t) >> 1)) >> shift;
  }
};

UnitMap make_unit_map(uint32_t units, uint32_t nblk, int64_t row0) {
  UnitMap m{units, nblk, 0u, 0u, row0};
  if (nblk > 1) {
    uint32_t l = 0;
    while ((uint64_t(1) << l) < nblk) ++l;
    m.magic = (uint32_t)(((uint64_t(1) << 32) * ((uint64_t(1) << l) - nblk)) / nblk + 1);
    m.shift = l - 1;
  }
  return m;
}

// ------------------------------------------------------------------ amax
// Grid-stride over 8-element units, four independent 16-byte loads in flight
// per thread and iteration.
template <typename T>
__global__ void __launch_bounds__(kThreads) amax_kernel(const T* __restrict__ x, int64_t n8,
                                                        unsigned* amax_bits, int* status) {
  pdl_wait();  // inputs may come from the previous kernel
  float m = 0.f;
  bool bad = false;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t u = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; u + 3 * stride < n8; u += 4 * stride) {
    float v[4][8];
#pragma unroll
    for (int i = 0; i < 4; ++i) load8<T>(x, (u + i * stride) * 8, v[i]);
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        bad |= nonfinite(v[i][j]);
        m = fmaxf(m, fabsf(v[i][j]));
      }
  }
  for (; u < n8; u += stride) {
    float v[8];
    load8<T>(x, u * 8, v);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      bad |= nonfinite(v[j]);
      m = fmaxf(m, fabsf(v[j]));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  __shared__ float warp_max[kThreads / 32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) warp_max[warp] = m;
  bad = __syncthreads_or(bad);
  if (threadIdx.x == 0) {
    float b = 0.f;
    for (int w = 0; w < kThreads / 32; ++w) b = fmaxf(b, warp_max[w]);
    // |x| >= 0, so the float bit patterns order like the values
    atomicMax(amax_bits, __float_as_uint(b));
    if (bad) latch_status(status, Q4_ERR_NONFINITE);
  }
}

// ------------------------------------------------------------------ NVFP4
// One thread per 16-element block.
//
// The pages' rule is y = x / S in float32 (rounded to nearest), clamped to
// [-6, 6], then rounded to the nearest E2M1 value with ties to the smaller
// magnitude.  Here:
//  * y0 = |x| * R, with R within 1 ulp of 1/S, is within 2.5 ulp of |x| / S.  The E2M1 decision
//    points t_k in {0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5} have three
//    significant bits, so when y0 is more than 8 ulp away from every float
//    with three significant bits, RN(|x| / S) and y0 lie strictly inside the
//    same E2M1 rounding cell, and no tie can occur: the hardware RNE convert of
//    y0 gives the pages' code.
//  * Otherwise (rare for real data) y = RN(|x| / S) is computed by an IEEE
//    division.  If y itself has three significant bits it may be a tie; its
//    predecessor lies in the cell that ties-to-smaller selects, and any other
//    three-bit y lies inside its cell, so the predecessor converts correctly.
//    With rne (round half to even on request) y itself is converted: the
//    hardware convert breaks the tie to the even code.
// The sign goes in bit 3 when x < 0, also for codes of magnitude 0; the
// hardware convert keeps the sign of a negative zero.
// Persistent: each CTA walks tiles of 256 units (one per thread), a 4-slot
// ring of bulk copies (one thread issues them) keeping three tiles in flight
// while the threads work on the fourth.  The grid walks the tiles from the
// last to the first: the amax pass before it reads x from the first element to
// the last, so the part of x it read last (up to the size of L2) is still in
// L2 when this pass starts, and the codes are stored with the streaming hint
// so that they do not push it out.
constexpr int kQStages = 4;
constexpr int kQUnits = kThreads;

template <typename T>
__global__ void __launch_bounds__(kThreads, 4)
    nvfp4_kernel(const T* __restrict__ x, const UnitMap um, uint8_t* __restrict__ codes,
                 uint8_t* __restrict__ scales, int layout, int64_t nsf4,
                 const unsigned* __restrict__ amax_bits, float* tensor_scale, KernelCtl ctl,
                 bool rne) {
  pdl_wait();  // inputs may come from the previous kernel
  // x and codes start at row um.row0; scales are indexed by the global row
  constexpr uint32_t kTileBytes = kQUnits * 16 * sizeof(T);
  extern __shared__ __align__(128) uint8_t qring[];  // [kQStages][kTileBytes]
  __shared__ __align__(8) uint64_t full[kQStages];
  __shared__ float s_g, s_c6g;
  __shared__ int s_abort;
  const uint32_t ntiles = (um.units + kQUnits - 1) / kQUnits;
  const uint32_t tid = threadIdx.x;
  // the CTA's i-th tile: index blockIdx.x + i G of the walk, which runs from
  // the last tile down to the first
  auto idx_of = [&](uint32_t i) { return blockIdx.x + i * gridDim.x; };
  auto tile_of = [&](uint32_t i) { return ntiles - 1 - idx_of(i); };
  auto issue = [&](uint32_t i) {  // the CTA's i-th tile into slot i % kQStages
    if (idx_of(i) >= ntiles) return;
    const uint32_t tile = tile_of(i);
    const uint32_t n = min((uint32_t)kQUnits, um.units - tile * kQUnits);
    const uint32_t bar = smem_u32(&full[i % kQStages]);
    mbar_arrive_expect_tx(bar, n * 16 * (uint32_t)sizeof(T));
    bulk_load(smem_u32(qring + (i % kQStages) * kTileBytes), x + (int64_t)tile * kQUnits * 16,
              n * 16 * (uint32_t)sizeof(T), bar);
  };
  if (tid == 0) {
    for (int i = 0; i < kQStages; ++i) mbar_init(smem_u32(&full[i]), 1);
    fence_mbar_init();
    // per-tensor scale g = max(amax_t, 1e-12) / (448 * 6), once per CTA
    s_g = __fdiv_rn(fmaxf(__uint_as_float(*amax_bits), 1e-12f), 2688.0f);
    s_c6g = __frcp_rn(__fmul_rn(6.0f, s_g));  // 1 / (6 g) within 1 ulp
    s_abort = 0;
    for (uint32_t i = 0; i + 1 < kQStages; ++i) issue(i);
  }
  __syncthreads();
  const float g = s_g, c6g = s_c6g;

  uint32_t i = 0;
  for (; idx_of(i) < ntiles; ++i) {
    if (tid == 0 && !mbar_wait(smem_u32(&full[i % kQStages]), (i / kQStages) & 1, ctl, &s_abort))
      s_abort = 1;
    __syncthreads();  // the tile has landed; every thread is done with slot (i - 1) % kQStages
    if (s_abort) break;
    if (tid == 0) issue(i + kQStages - 1);
    const uint32_t u = tile_of(i) * kQUnits + tid;
    if (u >= um.units) continue;
    float v[16];
    {
      const uint4* src = reinterpret_cast<const uint4*>(qring + (i % kQStages) * kTileBytes +
                                                        tid * 16 * sizeof(T));
      if constexpr (sizeof(T) == 4) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 w = src[q];
          v[4 * q] = __uint_as_float(w.x); v[4 * q + 1] = __uint_as_float(w.y);
          v[4 * q + 2] = __uint_as_float(w.z); v[4 * q + 3] = __uint_as_float(w.w);
        }
      } else {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const uint4 w = src[q];
          const T* h = reinterpret_cast<const T*>(&w);
#pragma unroll
          for (int e = 0; e < 8; ++e) v[8 * q + e] = Elem<T>::to_f(h[e]);
        }
      }
    }
    float amax = 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(v[j]));

    // block scale: E4M3 of (amax_b / 6) / g, round to nearest even
    // t = RN(RN(amax / 6) / g) matters only through its E4M3 rounding.  ta =
    // amax * RN(1 / RN(6 g)) is within 5 ulp of t, and the E4M3 rounding cells
    // (normal, subnormal and the saturation edge) are bounded by floats with at
    // most 5 significant bits; unless ta is within 8 ulp of such a float, t and
    // ta round to the same E4M3 value.  Otherwise t is computed as defined.
    float t = __fmul_rn(amax, c6g);
    if (((__float_as_uint(t) + 8u) & 0x7FFF0u) == 0u) t = __fdiv_rn(__fdiv_rn(amax, 6.0f), g);
    const __nv_fp8_storage_t bs = __nv_cvt_float_to_fp8(t, __NV_SATFINITE, __NV_E4M3);
    const float bsf = __half2float(__half(__nv_cvt_fp8_to_halfraw(bs, __NV_E4M3)));
    const float S = __fmul_rn(fmaxf(bsf, 1e-12f), g);

    uint2 packed = make_uint2(0u, 0u);
    if (bs != 0) {
      float R;  // 1 / S within 1 ulp (S is a normal float: e4m3 >= 2^-9, g > 3e-16)
      asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(R) : "f"(S));
      // y = x * R + 0 rounds once like x * R, keeps the sign of a negative x
      // (so its code carries the sign bit even when its magnitude rounds to 0)
      // and turns x = -0 into +0, whose code is 0.
      float y[16];
      bool near = false;
  #pragma unroll
      for (int j = 0; j < 16; ++j) {
        y[j] = __fmaf_rn(v[j], R, 0.0f);
        // |y| in [0.125, 5.5) and within 8 ulp of a float with 3 significant bits
        const uint32_t d = (__float_as_uint(y[j]) & 0x7FFFFFFFu) - 0x3E000000u + 8u;
        near |= ((d & 0x1FFFF0u) == 0u) & (d < 0x02B00008u);
      }
      if (near) {
  #pragma unroll
        for (int j = 0; j < 16; ++j) {
          const uint32_t d = (__float_as_uint(y[j]) & 0x7FFFFFFFu) - 0x3E000000u + 8u;
          if (((d & 0x1FFFF0u) == 0u) & (d < 0x02B00008u)) {
            uint32_t b = __float_as_uint(__fdiv_rn(fabsf(v[j]), S));
            if (!rne && (b & 0x1FFFFFu) == 0u) b -= 1u;  // |y| >= 0.12 here, so b > 0
            y[j] = __uint_as_float(b | (__float_as_uint(y[j]) & 0x80000000u));
          }
        }
      }
  #pragma unroll
      for (int j = 0; j < 4; ++j) {
        packed.x |= cvt_e2m1x2(y[2 * j], y[2 * j + 1]) << (8 * j);
        packed.y |= cvt_e2m1x2(y[8 + 2 * j], y[8 + 2 * j + 1]) << (8 * j);
      }
    }
    __stcs(reinterpret_cast<uint2*>(codes) + u, packed);

    const uint32_t rl = um.row_of(u);
    const int64_t row = um.row0 + rl, blk = u - rl * um.nblk;
    const int64_t off = layout == Q4_SCALES_MMA ? mma_scale_offset(row, blk, nsf4)
                                                : row * um.nblk + blk;
    scales[off] = (uint8_t)bs;
    if (u == 0 && um.row0 == 0 && tensor_scale) *tensor_scale = g;
  }
  // after an abort, copies already issued must land before the CTA exits
  if (tid == 0 && s_abort) {
    KernelCtl drain = ctl;
    for (uint32_t k = i; k < i + kQStages - 1; ++k)
      if (idx_of(k) < ntiles) mbar_wait(smem_u32(&full[k % kQStages]), (k / kQStages) & 1, drain, nullptr);
  }
}

// ------------------------------------------------------------------ MXFP4
// One thread per 16 elements; a thread pair shares one 32-element block (the
// rounding argument is at mxfp4_encode16).
template <typename T>
__global__ void __launch_bounds__(kThreads)
    mxfp4_kernel(const T* __restrict__ x, const UnitMap um, uint8_t* __restrict__ codes,
                 uint8_t* __restrict__ scales, int layout, int64_t nsf4, bool rne) {
  pdl_wait();  // inputs may come from the previous kernel
  const uint32_t u = blockIdx.x * blockDim.x + threadIdx.x;
  const bool live = u < um.units;
  float v[16];
  float amax = 0.f;
  if (live) {
    load16<T>(x, (int64_t)u * 16, v);
#pragma unroll
    for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(v[j]));
  }
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  if (!live) return;

  int e;
  const uint2 packed = mxfp4_encode16(v, amax, rne, e);
  reinterpret_cast<uint2*>(codes)[u] = packed;

  if ((u & 1) == 0) {
    const uint32_t rl = um.row_of(u);
    const int64_t row = um.row0 + rl, blk = (u - rl * um.nblk) >> 1;
    const int64_t off = layout == Q4_SCALES_MMA ? mma_scale_offset(row, blk, nsf4)
                                                : row * (um.nblk / 2) + blk;
    scales[off] = (uint8_t)(e + 127);
  }
}

// ------------------------------------------------------------------ INT4 g128
// One thread per 16 elements; eight threads share one 128-element group.
template <typename T>
__global__ void __launch_bounds__(kThreads)
    int4_kernel(const T* __restrict__ x, const UnitMap um, uint8_t* __restrict__ codes,
                uint16_t* __restrict__ scales) {
  pdl_wait();  // inputs may come from the previous kernel
  const uint32_t u = blockIdx.x * blockDim.x + threadIdx.x;
  const bool live = u < um.units;
  float v[16];
  float amax = 0.f;
  if (live) {
    load16<T>(x, (int64_t)u * 16, v);
#pragma unroll
    for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(v[j]));
  }
#pragma unroll
  for (int o = 1; o < 8; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if (!live) return;

  const __half s16 = __float2half_rn(__fdiv_rn(amax, 7.0f));
  const float sf = __half2float(s16);
  uint2 packed = make_uint2(0u, 0u);
  if (sf != 0.f) {
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      float q = rintf(__fdiv_rn(v[j], sf));
      q = fminf(fmaxf(q, -8.0f), 7.0f);
      const uint32_t c = (uint32_t)(int)q & 0xFu;
      if (j < 8) packed.x |= c << (4 * j);
      else packed.y |= c << (4 * (j - 8));
    }
  }
  reinterpret_cast<uint2*>(codes)[u] = packed;
  if ((u & 7) == 0) {
    const uint32_t rl = um.row_of(u);
    const int64_t grp = (u - rl * um.nblk) >> 3;
    scales[(int64_t)rl * (um.nblk / 8) + grp] = __half_as_ushort(s16);  // scales start at row0
  }
}

// ------------------------------------------------------------------ scale re-layout
__global__ void __launch_bounds__(kThreads)
    scales_to_mma_kernel(const uint8_t* __restrict__ src, int64_t rows, int64_t nsf, int64_t nsf4,
                         uint8_t* __restrict__ dst, int64_t total) {
  pdl_wait();  // inputs may come from the previous kernel
  const int64_t d = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (d >= total) return;
  const int64_t tile = d >> 9, o = d & 511;
  const int64_t r = (tile / nsf4) * 128 + ((o & 15) >> 2) * 32 + (o >> 4);
  const int64_t s = (tile % nsf4) * 4 + (o & 3);
  dst[d] = (r < rows && s < nsf) ? src[r * nsf + s] : (uint8_t)0;
}

inline unsigned blocks_for(int64_t units) { return (unsigned)ceil_div(units, kThreads); }

}  // namespace

q4_status launch_amax(const void* x, int dtype, int64_t n, unsigned* amax_bits,
                      cudaStream_t stream) {
  const int64_t n8 = n / 8;
  if (n8 == 0) return Q4_OK;
  const unsigned grid = (unsigned)std::min<int64_t>(ceil_div(n8, kThreads), (int64_t)num_sms() * 4);
  int* st = device_status_ptr();
  switch (dtype) {
    case Q4_F32: return launch_pdl(amax_kernel<float>, grid, kThreads, 0, stream, (const float*)x, n8, amax_bits, st);
    case Q4_BF16: return launch_pdl(amax_kernel<__nv_bfloat16>, grid, kThreads, 0, stream, (const __nv_bfloat16*)x, n8, amax_bits, st);
    case Q4_F16: return launch_pdl(amax_kernel<__half>, grid, kThreads, 0, stream, (const __half*)x, n8, amax_bits, st);
    default: return Q4_ERR_INVALID_ARG;
  }
}

// Launches `launch(um, grid, row0)` (returning a q4_status) over chunks of
// whole rows (multiples of 128) holding fewer than 2^32 units each.
template <typename F>
q4_status for_row_chunks(int64_t rows, int64_t nblk, F&& launch) {
  const int64_t cap = ((int64_t)0xFFFFFE00 / nblk) / 128 * 128;
  if (cap <= 0) return Q4_ERR_UNSUPPORTED_SHAPE;
  for (int64_t r0 = 0; r0 < rows; r0 += cap) {
    const int64_t nr = std::min(cap, rows - r0);
    const UnitMap um = make_unit_map((uint32_t)(nr * nblk), (uint32_t)nblk, r0);
    if (launch(um, (unsigned)ceil_div(nr * nblk, kThreads), r0) != Q4_OK) return Q4_ERR_CUDA;
  }
  return Q4_OK;
}

template <typename T>
const T* rows_from(const void* x, int64_t r0, int64_t K) {
  return static_cast<const T*>(x) + r0 * K;
}

q4_status launch_quant_nvfp4(const void* x, int dtype, int64_t rows, int64_t K, uint8_t* codes,
                             uint8_t* scales, int layout, const unsigned* amax_bits,
                             float* tensor_scale, cudaStream_t stream, bool rne) {
  const int64_t nblk = K / 16;
  const int64_t nsf4 = ceil_div(nblk, 4);
  // every byte of an unpadded MMA layout is written by the kernel
  if (layout == Q4_SCALES_MMA && (rows % 128 || nblk % 4))
    Q4_CUDA_TRY(cudaMemsetAsync(scales, 0, mma_scales_bytes(rows, nblk), stream));
  if (rows * nblk == 0) return Q4_OK;  // the API reports g of an empty tensor itself
  if (dtype != Q4_F32 && dtype != Q4_BF16 && dtype != Q4_F16) return Q4_ERR_INVALID_ARG;
  const KernelCtl ctl{device_status_ptr(), wait_budget_ns()};
  const size_t ring = (size_t)kQStages * kQUnits * 16 * (dtype == Q4_F32 ? 4 : 2);
  static int attr_done[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return Q4_ERR_CUDA;
  if (!attr_done[dev]) {
    Q4_CUDA_TRY(cudaFuncSetAttribute(nvfp4_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kQStages * kQUnits * 16 * 4));
    attr_done[dev] = 1;
  }
  const int64_t max_ctas = (int64_t)num_sms() * 4;
  return for_row_chunks(rows, nblk, [&](const UnitMap& um, unsigned, int64_t r0) {
    uint8_t* c = codes + r0 * (K / 2);
    const unsigned grid = (unsigned)std::min<int64_t>(ceil_div(um.units, kQUnits), max_ctas);
    if (dtype == Q4_F32)
      return launch_pdl(nvfp4_kernel<float>, grid, kThreads, ring, stream, rows_from<float>(x, r0, K), um, c, scales, layout, nsf4, amax_bits, tensor_scale, ctl, rne);
    else if (dtype == Q4_BF16)
      return launch_pdl(nvfp4_kernel<__nv_bfloat16>, grid, kThreads, ring, stream, rows_from<__nv_bfloat16>(x, r0, K), um, c, scales, layout, nsf4, amax_bits, tensor_scale, ctl, rne);
    else
      return launch_pdl(nvfp4_kernel<__half>, grid, kThreads, ring, stream, rows_from<__half>(x, r0, K), um, c, scales, layout, nsf4, amax_bits, tensor_scale, ctl, rne);
  });
}

q4_status launch_quant_mxfp4(const void* x, int dtype, int64_t rows, int64_t K, uint8_t* codes,
                             uint8_t* scales, int layout, cudaStream_t stream, bool rne) {
  const int64_t nblk = K / 16;
  const int64_t nsf4 = ceil_div(K / 32, 4);
  if (layout == Q4_SCALES_MMA && (rows % 128 || (K / 32) % 4))
    Q4_CUDA_TRY(cudaMemsetAsync(scales, 0, mma_scales_bytes(rows, K / 32), stream));
  if (rows * nblk == 0) return Q4_OK;
  if (dtype != Q4_F32 && dtype != Q4_BF16 && dtype != Q4_F16) return Q4_ERR_INVALID_ARG;
  return for_row_chunks(rows, nblk, [&](const UnitMap& um, unsigned grid, int64_t r0) {
    uint8_t* c = codes + r0 * (K / 2);
    if (dtype == Q4_F32)
      return launch_pdl(mxfp4_kernel<float>, grid, kThreads, 0, stream, rows_from<float>(x, r0, K), um, c, scales, layout, nsf4, rne);
    else if (dtype == Q4_BF16)
      return launch_pdl(mxfp4_kernel<__nv_bfloat16>, grid, kThreads, 0, stream, rows_from<__nv_bfloat16>(x, r0, K), um, c, scales, layout, nsf4, rne);
    else
      return launch_pdl(mxfp4_kernel<__half>, grid, kThreads, 0, stream, rows_from<__half>(x, r0, K), um, c, scales, layout, nsf4, rne);
  });
}

q4_status launch_quant_int4(const void* x, int dtype, int64_t rows, int64_t K, uint8_t* codes,
                            uint16_t* scales, cudaStream_t stream) {
  const int64_t nblk = K / 16;
  if (rows * nblk == 0) return Q4_OK;
  if (dtype != Q4_F32 && dtype != Q4_BF16 && dtype != Q4_F16) return Q4_ERR_INVALID_ARG;
  return for_row_chunks(rows, nblk, [&](const UnitMap& um, unsigned grid, int64_t r0) {
    uint8_t* c = codes + r0 * (K / 2);
    uint16_t* sc = scales + r0 * (K / 128);
    if (dtype == Q4_F32)
      return launch_pdl(int4_kernel<float>, grid, kThreads, 0, stream, rows_from<float>(x, r0, K), um, c, sc);
    else if (dtype == Q4_BF16)
      return launch_pdl(int4_kernel<__nv_bfloat16>, grid, kThreads, 0, stream, rows_from<__nv_bfloat16>(x, r0, K), um, c, sc);
    else
      return launch_pdl(int4_kernel<__half>, grid, kThreads, 0, stream, rows_from<__half>(x, r0, K), um, c, sc);
  });
}

q4_status launch_scales_to_mma(const uint8_t* src, int64_t rows, int64_t nsf, uint8_t* dst,
                               cudaStream_t stream) {
  const int64_t total = (int64_t)mma_scales_bytes(rows, nsf);
  if (total == 0) return Q4_OK;
  return launch_pdl(scales_to_mma_kernel, blocks_for(total), kThreads, 0, stream, src, rows, nsf,
                    ceil_div(nsf, 4), dst, total);
}

}  // namespace q4
