// W4A16 decode GEMM: C[m, n] = sum_g s16[n, g] * sum_{k in g} a[m, k] q[n, k]
// ("Low-bit inference for very large MoE", section "Kernels on different
// hardware", the W4A16 row: 4-bit weights, bf16 activations, bound by the
// weight reads in decode).
//
// Design (GB300):
//  * The packed INT4 weights are the only large stream.  Each thread copies
//    its own 16-byte pieces with cp.async into a private slot ring in shared
//    memory (4 groups of 128 in flight) and reads them back in exactly the
//    register shape of the bf16 tensor-core fragment.
//  * Programmatic dependent launch: the first 4 groups of weights are
//    requested before the kernel waits for the previous kernel in the stream
//    (activations and the output come after the wait).  The weights must
//    therefore not be written by a kernel that releases its successor early;
//    this library's quantizers do not.  This kernel itself releases the next
//    one as soon as its own weight loads are issued.
//  * Nibbles become exact bf16 integers with one LOP3 (mask, flip the sign
//    bit, OR the exponent of 128) and one bf16x2 subtraction of 136.
//  * NVFP4 weights: the hardware E2M1 convert gives f16 code pairs, one f16
//    multiply applies the block scale (exact), and the MMAs run in f16 on
//    f16 activations, for every group of 128 columns whose activations are
//    all f16 values; other groups (a value below 2^-17 or above 65504) use
//    bf16 weights built bit by bit, also exact.
//  * The products q * a are exact in the MMA and are summed in FP32; the FP16
//    group scale is applied once per group of 128 in FP32 (per-group
//    promotion), so the only rounding to bf16 is the final store.
//  * The activations of a CTA's K-slice sit in shared memory, permuted so that
//    every B fragment is one conflict-free 16-byte load.
//  * K is split across a thread-block cluster of up to 8 CTAs.  Each CTA
//    pushes the partial sums of the rows that rank q owns into rank q's
//    receive buffer (distributed shared memory stores), one cluster barrier
//    follows, and each owner adds its buffers in rank order: deterministic,
//    and nothing but C goes back to HBM.
#include "common.cuh"
#include "internal.h"

#include <algorithm>

namespace q4 {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kRows = 256;      // weight rows (n) per CTA: 8 warps x 2 tiles x 16
constexpr int kTok = 16;        // tokens per CTA (two n8 MMA tiles)
constexpr int kChunk = 8;       // groups of 128 staged per activation chunk
constexpr int kRing = 4;        // weight groups in flight per thread (cp.async ring)
constexpr int kActBytes = kChunk * 4 * kTok * 4 * 16;   // 32 KiB
constexpr int kRingBytes = kRing * 4 * kThreads * 16;   // 64 KiB: [slot][chunk][thread] x 16 B
constexpr int kSumBytes = kChunk * kTok * 4;            // 512 B: 136 * sum of a per group, token
// receive buffer of the cluster reduction: [source rank][owned row][token] FP32,
// at most 8 ranks x ceil(256 / ranks) rows
__host__ __device__ constexpr int recv_bytes(int tokens) { return (kRows + 7) * tokens * 4; }


__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool pred) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %2, 0;\n\t"
      "@p cp.async.cg.shared.global [%0], [%1], 16;\n\t}" ::"r"(dst),
      "l"(src), "r"((int)pred)
      : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Two nibbles at bits 0..3 and 16..19 of w -> bf16x2 of 136 + q, exactly:
// (n ^ 8) | 0x4300 is the bf16 of 128 + (q + 8).  The offset 136 is removed
// after the MMA, per group and token, as 136 * sum_k a[m, k].
__device__ __forceinline__ uint32_t nib_pair_to_bf16x2(uint32_t w) {
  uint32_t t;
  asm("lop3.b32 %0, %1, 0x000F000F, 0x43084308, 0x6A;" : "=r"(t) : "r"(w));
  return t;
}

// Weight formats of the W4A16 kernel.
constexpr int kInt4 = 0, kNvfp4 = 1, kMxfp4 = 2;

// E2M1 codes at nibbles i and i + 4 of w -> bf16x2 holding code * 2^-126,
// exactly: the three magnitude bits go to bf16 bits 6..8 (the two low bits of
// the exponent field and the top mantissa bit) and the sign bit to bit 15.
// Exponent field 0 is the subnormal range, so code 1 (0.5) becomes
// 0.5 * 2^-126 like every other code.  sgn = w & 0x88888888.
template <int i>
__device__ __forceinline__ uint32_t e2m1_pair_bits(uint32_t w, uint32_t sgn) {
  constexpr int sm = 6 - 4 * i;
  uint32_t m;
  if constexpr (sm >= 0) m = w << sm;
  else m = w >> -sm;
  return (m & 0x01C001C0u) | ((sgn << (12 - 4 * i)) & 0x80008000u);
}

__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// The four E2M1 code pairs of a 32-bit word (byte j = codes 2j, 2j + 1, the
// first in the low nibble) as f16x2 values, the first in the low half: the
// hardware convert, exact.
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t (&h)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\tmov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\tcvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\tcvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
}

__device__ __forceinline__ uint32_t f16x2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// f16x2 of (lo, hi); exact when both are f16 values
__device__ __forceinline__ uint32_t f16x2_of(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// The bf16 value in f16 without rounding (zero, infinities and NaN included)?
__device__ __forceinline__ bool f16_exact(float v) {
  return __half2float(__float2half_rn(v)) == v || v != v;
}

// Scale bytes -> float (exact; finite encodings only).  E4M3: bias 7, three
// mantissa bits, subnormals m * 2^-9.  E8M0: 2^(b - 127), byte 0 = 2^-127.
__device__ __forceinline__ float e4m3_value(uint32_t b) {
  const uint32_t e = (b >> 3) & 15u, m = b & 7u;
  const float mag = e ? __uint_as_float(((e + 120u) << 23) | (m << 20)) : (float)m * 0.001953125f;
  return (b & 0x80u) ? -mag : mag;
}
__device__ __forceinline__ float e8m0_value(uint32_t b) {
  return __uint_as_float(b ? (b << 23) : 0x00400000u);
}
// the bf16x2 with both halves equal to v (exact for the scale values above)
__device__ __forceinline__ uint32_t bf16x2_splat(float v) {
  const __nv_bfloat162 h = __float2bfloat162_rn(v);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t mapa_u32(uint32_t a, uint32_t rank) {
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
  return ra;
}

__device__ __forceinline__ void st_dsmem_f32x2(uint32_t addr, float a, float b) {
  asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" ::"r"(addr), "f"(a), "f"(b) : "memory");
}

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                               uint32_t a2, uint32_t a3, uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1,
                                              uint32_t a2, uint32_t a3, uint32_t b0,
                                              uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pick4(const uint32_t (&a)[4], int i) {
  return i == 0 ? a[0] : i == 1 ? a[1] : i == 2 ? a[2] : a[3];
}

__device__ __forceinline__ uint32_t word(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}


// grid = (CS, ceil(N / 256), ceil(M / 16)), cluster = (CS, 1, 1).  TS = token
// sets of 8 (1 when at most 8 tokens per block, else 2).  FMT: kInt4 (Wsc =
// FP16 scales [N, K/128]), kNvfp4 (E4M3 bytes [N, K/16], tensor scale *wg) or
// kMxfp4 (E8M0 bytes [N, K/32]).
template <int TS, int FMT>
__global__ void __launch_bounds__(kThreads, 2)
    w4a16_kernel(const __nv_bfloat16* __restrict__ A, const uint8_t* __restrict__ Wq,
                 const void* __restrict__ Wsc, const float* __restrict__ wg,
                 __nv_bfloat16* __restrict__ C, int M, int N, int K, int groups_per_cta) {
  const uint16_t* Ws = static_cast<const uint16_t*>(Wsc);
  const uint8_t* Wf = static_cast<const uint8_t*>(Wsc);
  constexpr int kTp = 8 * TS;  // tokens staged per CTA
  extern __shared__ __align__(16) uint8_t smem[];
  uint8_t* ring = smem;                                              // [slot][chunk][thread] x 16 B
  uint4* act = reinterpret_cast<uint4*>(smem + kRingBytes);         // [kChunk][4][kTp][4] x 16 B
  float* csum = reinterpret_cast<float*>(smem + kRingBytes + kActBytes);  // [kChunk][kTok]
  float* recv = reinterpret_cast<float*>(smem + kRingBytes + kActBytes + kSumBytes);  // [cs][per][kTp]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int quad = lane & 3, lrow = lane >> 2;
  const int cs = gridDim.x, rank = blockIdx.x;
  const int n_base = blockIdx.y * kRows;
  const int m0 = blockIdx.z * kTok;
  const int mt = min(M - m0, kTp);  // tokens present in this CTA
  const int ngroups = K / 128;
  const int g_begin = min(ngroups, rank * groups_per_cta);
  const int g_end = min(ngroups, g_begin + groups_per_cta);
  const int ng = g_end - g_begin;
  const int64_t wrow_bytes = K / 2;

  // this thread's four weight rows: tile t (0,1) x half h (0: lrow, 1: lrow + 8)
  int wrow[4];
  bool wok[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    wrow[i] = n_base + warp * 32 + (i >> 1) * 16 + (i & 1) * 8 + lrow;
    wok[i] = wrow[i] < N;
  }
  const uint32_t ring_base = smem_u32(ring);
  // group gi of this CTA's slice -> ring slot gi % kRing; a commit group per call
  auto issue = [&](int gi) {
    const int slot = gi % kRing;
    const bool live = gi < ng;
    const int g = g_begin + (live ? gi : 0);
#pragma unroll
    for (int i = 0; i < 4; ++i)
      cp_async16(ring_base + (uint32_t)(((slot * 4 + i) * kThreads + tid) * 16),
                 Wq + (int64_t)(wok[i] ? wrow[i] : 0) * wrow_bytes + g * 64 + quad * 16,
                 live && wok[i]);
    cp_async_commit();
  };
#pragma unroll
  for (int gi = 0; gi < kRing; ++gi) issue(gi);
  // Weight loads go out before the wait on the previous kernel in the stream
  // (see the note at the top); activations and the output wait for it.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // 16-byte scale loads need 8 groups per row and a 16-byte aligned Ws (the
  // interface only asks for 2-byte alignment)
  const bool s16 = (ngroups & 7) == 0 && (reinterpret_cast<uintptr_t>(Ws) & 15) == 0;

  if constexpr (FMT == kNvfp4) {  // the group mask of the f16 form starts clear
    if (tid == 0) *reinterpret_cast<unsigned*>(csum) = 0u;
    __syncthreads();
  }

  float acc[2][TS][4];  // [tile][token set][fragment]
#pragma unroll
  for (int t = 0; t < 2; ++t)
#pragma unroll
    for (int s = 0; s < TS; ++s)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[t][s][i] = 0.f;

  for (int gi0 = 0; gi0 < ng; gi0 += kChunk) {
    const int gc = min(kChunk, ng - gi0);
    const int c0 = g_begin + gi0;
    // ---- scales of this thread's rows for the chunk.  INT4: the FP16 scale of
    // each of the eight groups.  FP4: per group, the block scales of this
    // thread's 32 columns (NVFP4: the 2 bytes of blocks 2 quad, 2 quad + 1;
    // MXFP4: the byte of block quad), packed in order of the group.
    uint32_t spk[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t row = wok[i] ? wrow[i] : 0;
      if constexpr (FMT == kNvfp4) {
        const uint16_t* src = reinterpret_cast<const uint16_t*>(Wf + row * (K / 16) + (int64_t)c0 * 8) + quad;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint32_t lo = 2 * e < gc ? __ldg(src + 8 * e) : 0u;
          const uint32_t hi = 2 * e + 1 < gc ? __ldg(src + 8 * e + 4) : 0u;
          spk[i][e] = lo | (hi << 16);
        }
        continue;
      } else if constexpr (FMT == kMxfp4) {
        const uint8_t* src = Wf + row * (K / 32) + (int64_t)c0 * 4 + quad;
        spk[i][2] = spk[i][3] = 0u;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          uint32_t v = 0u;
#pragma unroll
          for (int b = 0; b < 4; ++b)
            if (4 * e + b < gc) v |= (uint32_t)__ldg(src + 4 * (4 * e + b)) << (8 * b);
          spk[i][e] = v;
        }
        continue;
      }
      const uint16_t* src = Ws + row * ngroups + c0;
      if (gc == kChunk && s16) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(src));
        spk[i][0] = v.x; spk[i][1] = v.y; spk[i][2] = v.z; spk[i][3] = v.w;
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint32_t lo = 2 * e < gc ? __ldg(src + 2 * e) : 0u;
          const uint32_t hi = 2 * e + 1 < gc ? __ldg(src + 2 * e + 1) : 0u;
          spk[i][e] = lo | (hi << 16);
        }
      }
    }

    // ---- stage the present tokens' activations, permuted per fragment, and
    // 136 * sum of each (group, token) for the INT4 offset.  Columns of absent
    // tokens are left as they are: their results are never stored.
    //  * 16-token blocks: one warp load covers 512 contiguous bytes of one
    //    token's row (two groups): lane l holds 16-byte piece l & 15 of group
    //    2 * pair + (l >> 4), so every sector fetched is used whole (with one
    //    thread per 64 bytes, as below, this staging took 1.1 us longer per
    //    launch).  Warp w takes the (token, group pair) units u * 8 + w, four
    //    loads in flight per lane; the 16 lanes of a (group, token) add their
    //    sums in a fixed shuffle order.
    //  * up to 8 tokens: 4 threads per (group, token), each with 4 pieces of
    //    16 bytes at once (this measured faster than the warp form at M = 4);
    //    partial sums meet in a fixed shuffle order.
    if (gi0 == 0) asm volatile("griddepcontrol.wait;" ::: "memory");
    else __syncthreads();  // every warp is done with the previous chunk
    // {x0,x1 | x2,x3 | x4,x5 | x6,x7} -> {x0,x4 | x1,x5 | x2,x6 | x3,x7}, and
    // the sum of the eight values in a fixed order
    bool exact = true;  // NVFP4: every activation this thread staged is an f16 value
    auto put = [&](const uint4& x, int gi, int w, int tok, int cq, float& sum) {
      if constexpr (FMT == kNvfp4) {
        const uint32_t e[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
          exact = exact && f16_exact(__uint_as_float(e[i] << 16)) &&
                  f16_exact(__uint_as_float(e[i] & 0xFFFF0000u));
      }
      uint4 v;
      v.x = __byte_perm(x.x, x.z, 0x5410);
      v.y = __byte_perm(x.x, x.z, 0x7632);
      v.z = __byte_perm(x.y, x.w, 0x5410);
      v.w = __byte_perm(x.y, x.w, 0x7632);
      act[((gi * 4 + w) * kTp + tok) * 4 + cq] = v;
      if constexpr (FMT == kInt4) {
        const uint32_t e[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
          sum += __uint_as_float(e[i] << 16) + __uint_as_float(e[i] & 0xFFFF0000u);
      }
    };
    if constexpr (TS == 2) {
      const int half = lane >> 4, q = lane & 15, cq = q >> 2, w = q & 3;
#pragma unroll
      for (int u0 = 0; u0 < 8; u0 += 4) {
        uint4 x[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int unit = (u0 + u) * kWarps + warp, tok = unit >> 2, gi = 2 * (unit & 3) + half;
          if (tok < mt && gi < gc)
            x[u] = reinterpret_cast<const uint4*>(A + (int64_t)(m0 + tok) * K + (int64_t)(c0 + gi) * 128)[q];
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int unit = (u0 + u) * kWarps + warp, tok = unit >> 2, gi = 2 * (unit & 3) + half;
          if (tok >= mt) continue;  // the same for the whole warp
          float sum = 0.f;
          if (gi < gc) put(x[u], gi, w, tok, cq, sum);
          if constexpr (FMT == kInt4) {  // FP4 weights have no offset to remove
#pragma unroll
            for (int o = 1; o < 16; o <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
            if (q == 0 && gi < gc) csum[gi * kTok + tok] = 136.0f * sum;
          }
        }
      }
    } else {
      const int pair = tid / 4, part = tid % 4;
      const int gi = pair / kTp, tok = pair % kTp;
      float sum = 0.f;
      if (gi < gc && tok < mt) {
        const uint4* src = reinterpret_cast<const uint4*>(A + (int64_t)(m0 + tok) * K +
                                                          (int64_t)(c0 + gi) * 128) + part * 4;
        uint4 x[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) x[u] = src[u];
#pragma unroll
        for (int u = 0; u < 4; ++u) put(x[u], gi, u, tok, part, sum);  // piece 4 part + u
      }
      if constexpr (FMT == kInt4) {
        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
        sum += __shfl_xor_sync(0xffffffffu, sum, 2);
        if (part == 0 && gi < gc && tok < mt) csum[gi * kTok + tok] = 136.0f * sum;
      }
    }
    // NVFP4, per group of the chunk: when every staged activation of the
    // group is an f16 value, its MMAs run in f16 (the weights come from the
    // hardware E2M1 convert, see below) and its staged slots become f16 pairs
    // in natural order, in place (each 16-byte slot holds the same eight
    // columns in either form); a group with any other value (below 2^-17 in
    // magnitude or above 65504, about 1 in 10^5 of N(0, 1) data) keeps the
    // bf16 form.  Every thread staged values of one group only, so one bit per
    // thread marks the groups that stay bf16.
    unsigned bf16_groups = 0u;
    if constexpr (FMT == kNvfp4) {
      unsigned* s_bad = reinterpret_cast<unsigned*>(csum);  // NVFP4 has no offset sums
      const int my_gi = TS == 2 ? 2 * (warp & 3) + (lane >> 4) : (tid / 4) / kTp;
      const unsigned m = __reduce_or_sync(0xffffffffu, exact ? 0u : 1u << (my_gi & 31));
      if (lane == 0 && m) atomicOr(s_bad, m);
      __syncthreads();
      bf16_groups = *s_bad;
      for (int e = tid; e < kChunk * 4 * kTp * 4; e += kThreads) {
        if ((bf16_groups >> (e / (4 * kTp * 4))) & 1u) continue;
        const uint4 v = act[e];  // {x0,x4 | x1,x5 | x2,x6 | x3,x7} in bf16
        uint4 h;
        h.x = f16x2_of(__uint_as_float(v.x << 16), __uint_as_float(v.y << 16));
        h.y = f16x2_of(__uint_as_float(v.z << 16), __uint_as_float(v.w << 16));
        h.z = f16x2_of(__uint_as_float(v.x & 0xFFFF0000u), __uint_as_float(v.y & 0xFFFF0000u));
        h.w = f16x2_of(__uint_as_float(v.z & 0xFFFF0000u), __uint_as_float(v.w & 0xFFFF0000u));
        act[e] = h;  // {x0,x1 | x2,x3 | x4,x5 | x6,x7} in f16
      }
      __syncthreads();  // every thread has read the mask: the next chunk may set it again
      if (tid == 0) *s_bad = 0u;
    } else {
      __syncthreads();
    }

    auto group = [&](int gl) {
      if (gl < gc) {
        const int gi = gi0 + gl;
        cp_async_wait<kRing - 1>();  // this thread's copies of group gi have landed
        const int slot = gi % kRing;
        uint4 wv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
          wv[i] = *reinterpret_cast<const uint4*>(ring + ((slot * 4 + i) * kThreads + tid) * 16);
        if constexpr (FMT == kNvfp4) {
          if (!((bf16_groups >> gl) & 1u)) {
            // NVFP4, f16 form: code pairs (2j, 2j + 1) by the hardware convert,
            // times the E4M3 scale x 2^-10 in f16 -- exact, subnormals included
            // (at most 6 significant bits, multiples of 2^-20 up to 2.625) --
            // against f16 activations in natural order.  The 2^10 goes back
            // with the tensor scale, as in the bf16 form.
            uint32_t s16[4][2];  // [row][half of this thread's 32 columns]
#pragma unroll
            for (int r = 0; r < 4; ++r) {
              const uint32_t b2 = (pick4(spk[r], gl >> 1) >> ((gl & 1) * 16)) & 0xFFFFu;
              const float lo = e4m3_value(b2 & 0xFFu) * 0x1p-10f, hi = e4m3_value(b2 >> 8) * 0x1p-10f;
              s16[r][0] = f16x2_of(lo, lo);
              s16[r][1] = f16x2_of(hi, hi);
            }
#pragma unroll
            for (int w = 0; w < 4; ++w) {
              uint4 bf[TS];
#pragma unroll
              for (int s = 0; s < TS; ++s) bf[s] = act[((gl * 4 + w) * kTp + lrow + 8 * s) * 4 + quad];
#pragma unroll
              for (int t = 0; t < 2; ++t) {
                uint32_t pl[4], ph[4];
                e2m1x8_to_f16x2(word(wv[2 * t], w), pl);
                e2m1x8_to_f16x2(word(wv[2 * t + 1], w), ph);
                const uint32_t sl = s16[2 * t][w >> 1], sh = s16[2 * t + 1][w >> 1];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  pl[j] = f16x2_mul(pl[j], sl);
                  ph[j] = f16x2_mul(ph[j], sh);
                }
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                  for (int s = 0; s < TS; ++s)
                    mma_f16_16816(acc[t][s], pl[2 * h], ph[2 * h], pl[2 * h + 1], ph[2 * h + 1],
                                  h ? bf[s].z : bf[s].x, h ? bf[s].w : bf[s].y);
              }
            }
            issue(gi + kRing);  // refill the slot just read
            return;
          }
        }
        if constexpr (FMT != kInt4) {
          // FP4: the block scale is folded into each weight, exactly in bf16
          // (e2m1 x E4M3 has at most 6 significant bits; e2m1 x 2^e is exact
          // for the E8M0 bytes a quantizer of finite data writes), so the
          // products with the activations are exact and the MMA accumulates
          // straight into the FP32 sums: no per-group promotion.
          uint32_t s2[4][2];  // [row][half of this thread's 32 columns]
#pragma unroll
          for (int r = 0; r < 4; ++r) {
            if constexpr (FMT == kNvfp4) {
              // E4M3 scale x 2^116 (exact, normal: 2^107 .. 448 * 2^116), so
              // that one multiply gives code * scale * 2^-10; the 2^10 goes
              // back with the tensor scale
              const uint32_t b2 = (pick4(spk[r], gl >> 1) >> ((gl & 1) * 16)) & 0xFFFFu;
              s2[r][0] = bf16x2_splat(e4m3_value(b2 & 0xFFu) * 0x1p116f);
              s2[r][1] = bf16x2_splat(e4m3_value(b2 >> 8) * 0x1p116f);
            } else {
              s2[r][0] = s2[r][1] = bf16x2_splat(e8m0_value((pick4(spk[r], gl >> 2) >> ((gl & 3) * 8)) & 0xFFu));
            }
          }
          constexpr uint32_t kTwo126 = 0x7E807E80u;  // bf16x2 of 2^126
          auto fp4_word = [&](int w) {
            uint4 bf[TS];
#pragma unroll
            for (int s = 0; s < TS; ++s) bf[s] = act[((gl * 4 + w) * kTp + lrow + 8 * s) * 4 + quad];
#pragma unroll
            for (int t = 0; t < 2; ++t) {
              const uint32_t lo = word(wv[2 * t], w), hi = word(wv[2 * t + 1], w);
              const uint32_t ls = lo & 0x88888888u, hs = hi & 0x88888888u;
              const uint32_t sl = (w >> 1) ? s2[2 * t][1] : s2[2 * t][0];
              const uint32_t sh = (w >> 1) ? s2[2 * t + 1][1] : s2[2 * t + 1][0];
              uint32_t pl[4], ph[4];
              if constexpr (FMT == kNvfp4) {  // code * 2^-126 times scale * 2^116
                pl[0] = bf16x2_mul(e2m1_pair_bits<0>(lo, ls), sl);
                pl[1] = bf16x2_mul(e2m1_pair_bits<1>(lo, ls), sl);
                pl[2] = bf16x2_mul(e2m1_pair_bits<2>(lo, ls), sl);
                pl[3] = bf16x2_mul(e2m1_pair_bits<3>(lo, ls), sl);
                ph[0] = bf16x2_mul(e2m1_pair_bits<0>(hi, hs), sh);
                ph[1] = bf16x2_mul(e2m1_pair_bits<1>(hi, hs), sh);
                ph[2] = bf16x2_mul(e2m1_pair_bits<2>(hi, hs), sh);
                ph[3] = bf16x2_mul(e2m1_pair_bits<3>(hi, hs), sh);
              } else {  // E8M0 scales span 2^-127 .. 2^127: times 2^126, then the scale
                pl[0] = bf16x2_mul(bf16x2_mul(e2m1_pair_bits<0>(lo, ls), kTwo126), sl);
                pl[1] = bf16x2_mul(bf16x2_mul(e2m1_pair_bits<1>(lo, ls), kTwo126), sl);
                pl[2] = bf16x2_mul(bf16x2_mul(e2m1_pair_bits<2>(lo, ls), kTwo126), sl);
                pl[3] = bf16x2_mul(bf16x2_mul(e2m1_pair_bits<3>(lo, ls), kTwo126), sl);
                ph[0] = bf16x2_mul(bf16x2_mul(e2m1_pair_bits<0>(hi, hs), kTwo126), sh);
                ph[1] = bf16x2_mul(bf16x2_mul(e2m1_pair_bits<1>(hi, hs), kTwo126), sh);
                ph[2] = bf16x2_mul(bf16x2_mul(e2m1_pair_bits<2>(hi, hs), kTwo126), sh);
                ph[3] = bf16x2_mul(bf16x2_mul(e2m1_pair_bits<3>(hi, hs), kTwo126), sh);
              }
#pragma unroll
              for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int s = 0; s < TS; ++s)
                  mma_bf16_16816(acc[t][s], pl[2 * h], ph[2 * h], pl[2 * h + 1], ph[2 * h + 1],
                                 h ? bf[s].z : bf[s].x, h ? bf[s].w : bf[s].y);
            }
          };
          if constexpr (FMT == kNvfp4) {  // the rare bf16 form: kept short, one word at a time
#pragma unroll 1
            for (int w = 0; w < 4; ++w) fp4_word(w);
          } else {
#pragma unroll
            for (int w = 0; w < 4; ++w) fp4_word(w);
          }
          issue(gi + kRing);  // refill the slot just read
        } else {  // INT4: per-group promotion of the MMA sums
          float part[2][TS][4];
#pragma unroll
          for (int t = 0; t < 2; ++t)
#pragma unroll
            for (int s = 0; s < TS; ++s)
#pragma unroll
              for (int i = 0; i < 4; ++i) part[t][s][i] = 0.f;
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            uint4 bf[TS];
#pragma unroll
            for (int s = 0; s < TS; ++s) bf[s] = act[((gl * 4 + w) * kTp + lrow + 8 * s) * 4 + quad];
#pragma unroll
            for (int t = 0; t < 2; ++t) {
              // nibble pairs (i, i + 4) of the row's word sit at bits 4i.. and 16 + 4i..
              const uint32_t lo = word(wv[2 * t], w), hi = word(wv[2 * t + 1], w);
              uint32_t pl[4], ph[4];
              pl[0] = nib_pair_to_bf16x2(lo);
              pl[1] = nib_pair_to_bf16x2(lo >> 4);
              pl[2] = nib_pair_to_bf16x2(lo >> 8);
              pl[3] = nib_pair_to_bf16x2(lo >> 12);
              ph[0] = nib_pair_to_bf16x2(hi);
              ph[1] = nib_pair_to_bf16x2(hi >> 4);
              ph[2] = nib_pair_to_bf16x2(hi >> 8);
              ph[3] = nib_pair_to_bf16x2(hi >> 12);
#pragma unroll
              for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int s = 0; s < TS; ++s)
                  mma_bf16_16816(part[t][s], pl[2 * h], ph[2 * h], pl[2 * h + 1], ph[2 * h + 1],
                                 h ? bf[s].z : bf[s].x, h ? bf[s].w : bf[s].y);
            }
          }
          issue(gi + kRing);  // refill the slot just read (the registers hold its data)
          // per-group promotion: remove the offset, then one FP32 multiply by the
          // FP16 scale of each row
          float c0v[TS], c1v[TS];
#pragma unroll
          for (int s = 0; s < TS; ++s) {
            const float2 cc = *reinterpret_cast<const float2*>(&csum[gl * kTok + s * 8 + 2 * quad]);
            c0v[s] = cc.x;
            c1v[s] = cc.y;
          }
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            const uint32_t plo = pick4(spk[2 * t], gl >> 1), phi = pick4(spk[2 * t + 1], gl >> 1);
            const float slo = __half2float(__ushort_as_half((uint16_t)((gl & 1) ? plo >> 16 : plo)));
            const float shi = __half2float(__ushort_as_half((uint16_t)((gl & 1) ? phi >> 16 : phi)));
#pragma unroll
            for (int s = 0; s < TS; ++s) {  // pairs of tokens per instruction, same rounding
              float d0, d1, d2, d3;
              sub2(d0, d1, part[t][s][0], part[t][s][1], c0v[s], c1v[s]);
              sub2(d2, d3, part[t][s][2], part[t][s][3], c0v[s], c1v[s]);
              fma2(acc[t][s][0], acc[t][s][1], d0, d1, slo, slo);
              fma2(acc[t][s][2], acc[t][s][3], d2, d3, shi, shi);
            }
          }
        }
      }
    };
    // NVFP4 keeps one copy of the group code (it holds two forms): with the
    // eight groups unrolled, launches of the 8- and 16-token kernels in turn
    // ran 10% slower than either alone (51.6 against 47.3 us per step of
    // three launches rolled).
    if constexpr (FMT == kNvfp4) {
#pragma unroll 1
      for (int gl = 0; gl < kChunk; ++gl) group(gl);
    } else {
#pragma unroll
      for (int gl = 0; gl < kChunk; ++gl) group(gl);
    }
  }
  cp_async_wait<0>();  // no copy may still target this CTA's shared memory at exit
  if (ng == 0) asm volatile("griddepcontrol.wait;" ::: "memory");  // C is written below

  // ---- push the partial sums of each owned row slice to its owner rank:
  // recv[src rank][row - owner * per][token] in the owner's shared memory
  const int per = (kRows + cs - 1) / cs;
  const uint32_t recv_base = smem_u32(recv);
#pragma unroll
  for (int t = 0; t < 2; ++t)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int r = warp * 32 + t * 16 + h * 8 + lrow;
      const int owner = r / per;
      const uint32_t dst = mapa_u32(recv_base, (uint32_t)owner) +
                           (uint32_t)(((rank * per + r - owner * per) * kTp) * 4);
#pragma unroll
      for (int s = 0; s < TS; ++s)
        st_dsmem_f32x2(dst + (uint32_t)((s * 8 + quad * 2) * 4), acc[t][s][2 * h],
                       acc[t][s][2 * h + 1]);
    }
  cluster_sync();  // every push has landed; nothing remote is touched afterwards

  // ---- rank q adds rows [q * per, (q + 1) * per) over the source ranks in order
  // and applies the NVFP4 tensor scale (read after the dependency wait)
  // NVFP4: the tensor scale, times the 2^10 the weights were scaled down by
  // (exact: a power of two)
  const float gsc = FMT == kNvfp4 ? __ldg(wg) * 1024.0f : 1.f;
  const int r_lo = rank * per, r_hi = min(kRows, r_lo + per);
  const int tq = (mt + 3) / 4;  // groups of four tokens
  for (int e = tid; e < (r_hi - r_lo) * tq; e += kThreads) {
    const int t4 = e / (r_hi - r_lo), rl = e % (r_hi - r_lo);
    float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int q = 0; q < cs; ++q) {
      const float4 v = *reinterpret_cast<const float4*>(&recv[((q * per + rl) * kTp) + 4 * t4]);
      sum.x += v.x; sum.y += v.y; sum.z += v.z; sum.w += v.w;
    }
    const int n = n_base + r_lo + rl;
    if (n < N) {
      const float vv[4] = {sum.x, sum.y, sum.z, sum.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (4 * t4 + i < mt) C[(int64_t)(m0 + 4 * t4 + i) * N + n] = __float2bfloat16_rn(vv[i] * gsc);
    }
  }
}

}  // namespace

namespace {
template <int FMT>
q4_status launch_w4a16_fmt(const void* A, const uint8_t* Wq, const void* Wsc, const float* wg,
                           int64_t M, int64_t N, int64_t K, void* C, cudaStream_t stream) {
  if (M == 0 || N == 0) return Q4_OK;
  const int ngroups = (int)(K / 128);
  // split K over a cluster of up to 8 CTAs, at least one group each
  // groups per CTA: a multiple of 8 (aligned 16-byte scale loads), at most 8
  // CTAs per cluster
  int cs = std::max(1, std::min(8, (int)ceil_div(ngroups, 8)));
  const int gpc = (int)(ceil_div(ceil_div(ngroups, cs), 8) * 8);
  cs = (int)ceil_div(ngroups, gpc);
  const size_t smem1 = kRingBytes + kActBytes + kSumBytes + recv_bytes(8);
  const size_t smem2 = kRingBytes + kActBytes + kSumBytes + recv_bytes(16);
  static int attr_done[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return Q4_ERR_CUDA;
  if (!attr_done[dev]) {
    Q4_CUDA_TRY(cudaFuncSetAttribute(w4a16_kernel<1, FMT>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem1));
    Q4_CUDA_TRY(cudaFuncSetAttribute(w4a16_kernel<2, FMT>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem2));
    attr_done[dev] = 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)cs, (unsigned)ceil_div(N, kRows), (unsigned)ceil_div(M, kTok));
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = M <= 8 ? smem1 : smem2;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // programmatic dependent launch: may start while the previous kernel in the
  // stream finishes; the kernel waits for it before touching activations or C
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  // one token set of 8 when every token block has at most 8 tokens
  if (M <= 8)
    Q4_CUDA_TRY(cudaLaunchKernelEx(&cfg, w4a16_kernel<1, FMT>, (const __nv_bfloat16*)A, Wq, Wsc, wg,
                                   (__nv_bfloat16*)C, (int)M, (int)N, (int)K, gpc));
  else
    Q4_CUDA_TRY(cudaLaunchKernelEx(&cfg, w4a16_kernel<2, FMT>, (const __nv_bfloat16*)A, Wq, Wsc, wg,
                                   (__nv_bfloat16*)C, (int)M, (int)N, (int)K, gpc));
  return Q4_OK;
}
}  // namespace

// The decode kernel keeps its partial sums in distributed shared memory: no
// workspace.
size_t w4a16_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  (void)M, (void)N, (void)K;
  return 0;
}

q4_status launch_w4a16(const void* A, const uint8_t* Wq, const uint16_t* Ws, int64_t M, int64_t N,
                       int64_t K, void* C, void* ws, size_t ws_bytes, cudaStream_t stream) {
  (void)ws, (void)ws_bytes;
  return launch_w4a16_fmt<kInt4>(A, Wq, Ws, nullptr, M, N, K, C, stream);
}

q4_status launch_w4a16_fp4(const void* A, const uint8_t* Wq, const uint8_t* Wsf, const float* wg,
                           bool nvfp4, int64_t M, int64_t N, int64_t K, void* C, void* ws,
                           size_t ws_bytes, cudaStream_t stream) {
  (void)ws, (void)ws_bytes;
  return nvfp4 ? launch_w4a16_fmt<kNvfp4>(A, Wq, Wsf, wg, M, N, K, C, stream)
               : launch_w4a16_fmt<kMxfp4>(A, Wq, Wsf, nullptr, M, N, K, C, stream);
}

}  // namespace q4

