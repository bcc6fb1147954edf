// W4A16 decode GEMM: C[m, n] = sum_g s16[n, g] * sum_{k in g} a[m, k] q[n, k]
// ("Low-bit inference for very large MoE", section "Kernels on different
// hardware", the W4A16 row: 4-bit weights, bf16 activations, bound by the
// weight reads in decode).
//
// Design (GB300):
//  * The packed INT4 weights are the only large stream.  Each thread loads its
//    own 16-byte pieces straight from HBM into registers (non-allocating in
//    L1), two groups ahead of use, in exactly the register shape the bf16
//    tensor-core fragment needs -- no shared-memory staging of weights.
//  * Nibbles become exact bf16 integers with one LOP3 (mask, flip the sign
//    bit, OR the exponent of 128) and one bf16x2 subtraction of 136.
//  * The products q * a are exact in the MMA and are summed in FP32; the FP16
//    group scale is applied once per group of 128 in FP32 (per-group
//    promotion), so the only rounding to bf16 is the final store.
//  * The activations of a CTA's K-slice sit in shared memory, permuted so that
//    every B fragment is one conflict-free 16-byte load.
//  * K is split across a thread-block cluster of up to 8 CTAs; their partial
//    sums are reduced through distributed shared memory in rank order, so the
//    result is deterministic and nothing but C goes back to HBM.
#include "common.cuh"
#include "internal.h"

#include <algorithm>

namespace q4 {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kRows = 128;      // weight rows (n) per CTA: 4 warps x 2 tiles x 16
constexpr int kTok = 16;        // tokens per CTA (two n8 MMA tiles)
constexpr int kChunk = 8;       // groups of 128 staged per activation chunk
constexpr int kActBytes = kChunk * 4 * kTok * 4 * 16;  // 32 KiB
constexpr int kRedBytes = kRows * kTok * 4;           // 8 KiB

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Two nibbles at bits 0..3 and 16..19 of w -> bf16x2 holding the signed
// values: (n ^ 8) | 0x4300 is the bf16 of 128 + (q + 8); minus 136 leaves q.
__device__ __forceinline__ uint32_t nib_pair_to_bf16x2(uint32_t w) {
  uint32_t t, r;
  asm("lop3.b32 %0, %1, 0x000F000F, 0x43084308, 0x6A;" : "=r"(t) : "r"(w));
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(t), "r"(0x43084308u));
  return r;
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

__device__ __forceinline__ uint32_t word(const uint4& v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

__device__ __forceinline__ float ld_dsmem_f32(const float* local, uint32_t rank) {
  uint32_t a = smem_u32(local), ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(a), "r"(rank));
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(ra) : "memory");
  return v;
}

// grid = (CS, ceil(N / 128), ceil(M / 16)), cluster = (CS, 1, 1).
__global__ void __launch_bounds__(kThreads)
    w4a16_kernel(const __nv_bfloat16* __restrict__ A, const uint8_t* __restrict__ Wq,
                 const uint16_t* __restrict__ Ws, __nv_bfloat16* __restrict__ C, int M, int N,
                 int K, int groups_per_cta) {
  extern __shared__ __align__(16) uint8_t smem[];
  uint4* act = reinterpret_cast<uint4*>(smem);                    // [kChunk][4][kTok][4] x 16B
  float* red = reinterpret_cast<float*>(smem + kActBytes);       // [kRows][kTok]

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int quad = lane & 3, lrow = lane >> 2;
  const int cs = gridDim.x, rank = blockIdx.x;
  const int n_base = blockIdx.y * kRows;
  const int m0 = blockIdx.z * kTok;
  const int ngroups = K / 128;
  const int g_begin = min(ngroups, rank * groups_per_cta);
  const int g_end = min(ngroups, g_begin + groups_per_cta);
  const int64_t wrow_bytes = K / 2;

  // this thread's four weight rows: tile t (0,1) x half h (0: lrow, 1: lrow + 8)
  int wrow[4];
  bool wok[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    wrow[i] = n_base + warp * 32 + (i >> 1) * 16 + (i & 1) * 8 + lrow;
    wok[i] = wrow[i] < N;
  }

  float acc[2][2][4];  // [tile][token set][fragment]
#pragma unroll
  for (int t = 0; t < 2; ++t)
#pragma unroll
    for (int s = 0; s < 2; ++s)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[t][s][i] = 0.f;

  for (int c0 = g_begin; c0 < g_end; c0 += kChunk) {
    const int gc = min(kChunk, g_end - c0);
    // ---- stage the activations of groups [c0, c0 + gc), permuted per fragment
    __syncthreads();
    const int slots = gc * 16 * kTok;  // 16-byte global chunks
    for (int s = tid; s < slots; s += kThreads) {
      const int tok = s / (gc * 16), q = s % (gc * 16);
      const int gi = q >> 4, cq = (q >> 2) & 3, w = q & 3;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (m0 + tok < M) {
        const uint4 x = *reinterpret_cast<const uint4*>(A + (int64_t)(m0 + tok) * K +
                                                        (int64_t)c0 * 128 + q * 8);
        // {x0,x1 | x2,x3 | x4,x5 | x6,x7} -> {x0,x4 | x1,x5 | x2,x6 | x3,x7}
        v.x = __byte_perm(x.x, x.z, 0x5410);
        v.y = __byte_perm(x.x, x.z, 0x7632);
        v.z = __byte_perm(x.y, x.w, 0x5410);
        v.w = __byte_perm(x.y, x.w, 0x7632);
      }
      act[((gi * 4 + w) * kTok + tok) * 4 + cq] = v;
    }
    __syncthreads();

    // ---- stream the weights: a three-deep register ring, two groups ahead
    uint4 wr[3][4];
    uint16_t sr[3][4];
    auto load_group = [&](int gi, int slot) {
      const int g = c0 + gi;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (gi < gc && wok[i]) {
          wr[slot][i] = ldg_stream(Wq + (int64_t)wrow[i] * wrow_bytes + g * 64 + quad * 16);
          sr[slot][i] = __ldg(Ws + (int64_t)wrow[i] * ngroups + g);
        } else {
          wr[slot][i] = make_uint4(0, 0, 0, 0);
          sr[slot][i] = 0;
        }
      }
    };
    load_group(0, 0);
    load_group(1, 1);
#pragma unroll
    for (int gi = 0; gi < kChunk; ++gi) {
      if (gi + 2 < kChunk) load_group(gi + 2, (gi + 2) % 3);
      if (gi < gc) {
        const int slot = gi % 3;
        float part[2][2][4];
#pragma unroll
        for (int t = 0; t < 2; ++t)
#pragma unroll
          for (int s = 0; s < 2; ++s)
#pragma unroll
            for (int i = 0; i < 4; ++i) part[t][s][i] = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const uint4 b0 = act[((gi * 4 + w) * kTok + lrow) * 4 + quad];
          const uint4 b1 = act[((gi * 4 + w) * kTok + lrow + 8) * 4 + quad];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t bb0 = h ? b0.z : b0.x, bb1 = h ? b0.w : b0.y;
            const uint32_t bc0 = h ? b1.z : b1.x, bc1 = h ? b1.w : b1.y;
#pragma unroll
            for (int t = 0; t < 2; ++t) {
              const uint32_t wlo = word(wr[slot][2 * t], w) >> (8 * h);
              const uint32_t whi = word(wr[slot][2 * t + 1], w) >> (8 * h);
              const uint32_t a0 = nib_pair_to_bf16x2(wlo);
              const uint32_t a1 = nib_pair_to_bf16x2(whi);
              const uint32_t a2 = nib_pair_to_bf16x2(wlo >> 4);
              const uint32_t a3 = nib_pair_to_bf16x2(whi >> 4);
              mma_bf16_16816(part[t][0], a0, a1, a2, a3, bb0, bb1);
              if (M - m0 > 8) mma_bf16_16816(part[t][1], a0, a1, a2, a3, bc0, bc1);
            }
          }
        }
        // per-group promotion: FP32 multiply by the FP16 scale of each row
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const float slo = __half2float(__ushort_as_half(sr[slot][2 * t]));
          const float shi = __half2float(__ushort_as_half(sr[slot][2 * t + 1]));
#pragma unroll
          for (int s = 0; s < 2; ++s) {
            acc[t][s][0] = fmaf(part[t][s][0], slo, acc[t][s][0]);
            acc[t][s][1] = fmaf(part[t][s][1], slo, acc[t][s][1]);
            acc[t][s][2] = fmaf(part[t][s][2], shi, acc[t][s][2]);
            acc[t][s][3] = fmaf(part[t][s][3], shi, acc[t][s][3]);
          }
        }
      }
    }
  }

  // ---- partial sums to shared memory: red[row][token]
#pragma unroll
  for (int t = 0; t < 2; ++t)
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      const int r = warp * 32 + t * 16 + lrow;
      const int tk = s * 8 + quad * 2;
      red[r * kTok + tk] = acc[t][s][0];
      red[r * kTok + tk + 1] = acc[t][s][1];
      red[(r + 8) * kTok + tk] = acc[t][s][2];
      red[(r + 8) * kTok + tk + 1] = acc[t][s][3];
    }
  cluster_sync();

  // ---- rank q reduces rows [q * per, (q + 1) * per) over all ranks, in rank order
  const int per = (kRows + cs - 1) / cs;
  const int r_lo = rank * per, r_hi = min(kRows, r_lo + per);
  for (int e = tid; e < (r_hi - r_lo) * kTok; e += kThreads) {
    const int tk = e % kTok, r = r_lo + e / kTok;
    float s = 0.f;
    for (int q = 0; q < cs; ++q) s += ld_dsmem_f32(&red[r * kTok + tk], (uint32_t)q);
    const int n = n_base + r, m = m0 + tk;
    if (n < N && m < M) C[(int64_t)m * N + n] = __float2bfloat16_rn(s);
  }
  cluster_sync();
}

}  // namespace

q4_status launch_w4a16(const void* A, const uint8_t* Wq, const uint16_t* Ws, int64_t M, int64_t N,
                       int64_t K, void* C, cudaStream_t stream) {
  if (M == 0 || N == 0) return Q4_OK;
  const int ngroups = (int)(K / 128);
  // split K over a cluster of up to 8 CTAs, at least one group each
  const int cs = std::max(1, std::min(8, ngroups));
  const int gpc = (int)ceil_div(ngroups, cs);
  const size_t smem = kActBytes + kRedBytes;
  static int attr_done[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return Q4_ERR_CUDA;
  if (!attr_done[dev]) {
    Q4_CUDA_TRY(cudaFuncSetAttribute(w4a16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)smem));
    attr_done[dev] = 1;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)cs, (unsigned)ceil_div(N, kRows), (unsigned)ceil_div(M, kTok));
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  Q4_CUDA_TRY(cudaLaunchKernelEx(&cfg, w4a16_kernel, (const __nv_bfloat16*)A, Wq, Ws,
                                 (__nv_bfloat16*)C, (int)M, (int)N, (int)K, gpc));
  return Q4_OK;
}

}  // namespace q4
