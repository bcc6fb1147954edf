// Device helpers shared by the quantizer kernels and the GEMM prologue that
// quantizes activations in place: 128-bit element loads and the MXFP4 encode
// of 16 elements ("Quantization in deployment", section "Fake quantization",
// mxfp4 and fp4).
#pragma once

#include "common.cuh"

namespace q4 {

// Eight consecutive elements starting at element index e (e % 8 == 0) as
// floats, with 128-bit loads.
template <typename T>
__device__ __forceinline__ void load8(const T* __restrict__ x, int64_t e, float (&v)[8]);

template <>
__device__ __forceinline__ void load8<float>(const float* __restrict__ x, int64_t e,
                                             float (&v)[8]) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(x + e));
  const float4 b = __ldg(reinterpret_cast<const float4*>(x + e + 4));
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

template <typename H>
__device__ __forceinline__ void load8_16bit(const H* __restrict__ x, int64_t e, float (&v)[8]) {
  const uint4 u = __ldg(reinterpret_cast<const uint4*>(x + e));
  const H* h = reinterpret_cast<const H*>(&u);
#pragma unroll
  for (int j = 0; j < 8; ++j) v[j] = Elem<H>::to_f(h[j]);
}
template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16* __restrict__ x, int64_t e,
                                                     float (&v)[8]) {
  load8_16bit(x, e, v);
}
template <>
__device__ __forceinline__ void load8<__half>(const __half* __restrict__ x, int64_t e,
                                              float (&v)[8]) {
  load8_16bit(x, e, v);
}

// Sixteen consecutive elements starting at element index e (e % 16 == 0).
template <typename T>
__device__ __forceinline__ void load16(const T* __restrict__ x, int64_t e, float (&v)[16]) {
  float a[8], b[8];
  load8<T>(x, e, a);
  load8<T>(x, e + 8, b);
#pragma unroll
  for (int j = 0; j < 8; ++j) { v[j] = a[j]; v[j + 8] = b[j]; }
}

// Sixteen consecutive elements kept as raw 128-bit words, so that a thread
// can have several such loads in flight before it converts any of them.
template <typename T>
struct Raw16 {
  uint4 q[sizeof(T)];
};
template <typename T>
__device__ __forceinline__ void load_raw16(const T* __restrict__ x, int64_t e, Raw16<T>& r) {
  const uint4* s = reinterpret_cast<const uint4*>(x + e);
#pragma unroll
  for (int i = 0; i < (int)sizeof(T); ++i) r.q[i] = __ldg(s + i);
}
template <typename T>
__device__ __forceinline__ void unpack16(const Raw16<T>& r, float (&v)[16]) {
  const T* h = reinterpret_cast<const T*>(r.q);
#pragma unroll
  for (int j = 0; j < 16; ++j) v[j] = Elem<T>::to_f(h[j]);
}

// Magnitude-and-sign E2M1 codes of two floats, RNE, saturating at 6: the
// code of lo in bits 0..3, of hi in bits 4..7.
__device__ __forceinline__ uint32_t cvt_e2m1x2(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  return r;
}

// MXFP4 codes of 16 elements of one 32-element block whose amax (over the
// whole block, both halves) is `amax`: the exponent e = floor(log2(max(amax,
// 1e-12))) - 2 (the scale byte is e + 127) and the packed E2M1 codes (element
// j in nibble j of the 64-bit word).
//
// y = x * 2^-e is exactly x / 2^e whenever it is a normal float (e is in
// [-42, 125], so 2^-e is a normal float and |y| < 8), and a subnormal y lies
// far below the smallest midpoint 0.25.  The hardware RNE convert of y is then
// the E2M1 code with ties to even; for the pages' ties to the smaller
// magnitude, a y with at most three significant bits (every midpoint has
// three) is replaced by its predecessor, which lies in the cell that rule
// selects (any other such y -- an E2M1 value, 7, or 0.125 -- stays in its
// cell).  y = x * 2^-e + 0 turns x = -0 into +0 (code 0) and keeps the sign of
// every negative x, as the pages' sign rule asks.
__device__ __forceinline__ uint2 mxfp4_encode16(const float (&v)[16], float amax, bool rne, int& e) {
  amax = fmaxf(amax, 1e-12f);  // normal, so floor(log2) is its exponent field
  e = (int)((__float_as_uint(amax) >> 23) & 0xFFu) - 127 - 2;
  const float rp2 = __uint_as_float((uint32_t)(127 - e) << 23);  // 2^-e
  float y[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    uint32_t b = __float_as_uint(__fmaf_rn(v[j], rp2, 0.0f));
    if (!rne && (b & 0x1FFFFFu) == 0u && (b & 0x7FFFFFFFu) != 0u) b -= 1u;  // magnitude predecessor
    y[j] = __uint_as_float(b);
  }
  uint2 packed = make_uint2(0u, 0u);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    packed.x |= cvt_e2m1x2(y[2 * j], y[2 * j + 1]) << (8 * j);
    packed.y |= cvt_e2m1x2(y[8 + 2 * j], y[8 + 2 * j + 1]) << (8 * j);
  }
  return packed;
}

}  // namespace q4
