// Host-side declarations shared by the q4gemm translation units (not part of
// the public C ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/q4gemm.h"

namespace q4 {

struct KernelCtl;

// Library-wide device state (status word) and settings.
int* device_status_ptr();            // device address of this device's status word
unsigned long long wait_budget_ns();  // bound on any kernel-side wait
int num_sms();                        // SM count of the current device

// Error helpers
#define Q4_CUDA_TRY(expr)                         \
  do {                                            \
    cudaError_t e_ = (expr);                      \
    if (e_ != cudaSuccess) return Q4_ERR_CUDA;    \
  } while (0)

// ---------------------------------------------------------------- quantizers
q4_status launch_amax(const void* x, int dtype, int64_t n, unsigned* amax_bits,
                      cudaStream_t stream);
// rne: E2M1 ties to the even code instead of the pages' smaller magnitude
q4_status launch_quant_nvfp4(const void* x, int dtype, int64_t rows, int64_t K, uint8_t* codes,
                             uint8_t* scales, int layout, const unsigned* amax_bits,
                             float* tensor_scale, cudaStream_t stream, bool rne = false);
q4_status launch_quant_mxfp4(const void* x, int dtype, int64_t rows, int64_t K, uint8_t* codes,
                             uint8_t* scales, int layout, cudaStream_t stream, bool rne = false);
q4_status launch_quant_int4(const void* x, int dtype, int64_t rows, int64_t K, uint8_t* codes,
                            uint16_t* scales, cudaStream_t stream);
q4_status launch_scales_to_mma(const uint8_t* src, int64_t rows, int64_t nsf, uint8_t* dst,
                               cudaStream_t stream);

// ---------------------------------------------------------------- GEMMs
// FP4 GEMM on pre-quantized operands with tensor-core scale layouts.
struct Fp4GemmArgs {
  const uint8_t* a_codes;   // [M, K/2]
  const uint8_t* a_scales;  // MMA layout
  const float* a_g;         // NVFP4 tensor scale or nullptr
  const uint8_t* b_codes;   // [N, K/2]
  const uint8_t* b_scales;  // MMA layout
  const float* b_g;
  int64_t M, N, K;
  void* C;
  int c_dtype;
  bool nvfp4;  // true: E4M3 scales per 16; false: E8M0 per 32
  // MXFP4 only: A given raw (a_raw, a_dtype); the GEMM quantizes it in its
  // prologue into a_codes / a_scales (workspace) and counts its CTAs in
  // *gate, which must be zero at launch
  const void* a_raw = nullptr;
  int a_dtype = 0;
  unsigned* gate = nullptr;
  // split-K partial sums (optional): used when at least the launch's need
  void* part_ws = nullptr;
  size_t part_ws_bytes = 0;
};
q4_status launch_fp4_gemm(const Fp4GemmArgs& a, cudaStream_t stream);
size_t fp4_splitk_partial_bytes(int64_t M, int64_t N, int64_t K, int nsms);

// Grouped (routed MoE) NVFP4 GEMM on a pre-quantized token tensor.
struct GroupedArgs {
  const uint8_t* a_routed;   // [R, K/2] quantized codes of the routed rows (copied in routed order)
  const uint8_t* a_sf_rows;  // routed scales, MMA layout, per-expert 128-row padded blocks
  const float* a_g;
  const int32_t* offsets;    // [E+1]
  const int32_t* sched;      // [E+1] tile-row prefix (device, built by the prep kernel)
  int64_t T, R, N, K;
  int E;
  const uint8_t* w_codes;    // [E, N, K/2]
  const uint8_t* w_scales;   // E x mma_scales_bytes(N, K/16)
  const float* w_g;          // [E]
  void* C;                   // [R, N] bf16
};
q4_status launch_grouped_prep(const int32_t* offsets, const int32_t* row_token, int E,
                              const uint8_t* tok_scales_rowmajor, int64_t nsf, int32_t* sched,
                              uint8_t* a_sf_routed, int64_t sf_rows_cap, cudaStream_t stream);
q4_status launch_gather_rows(const uint8_t* codes, const int32_t* row_token, int64_t R,
                             int64_t row_bytes, uint8_t* out, cudaStream_t stream);
q4_status launch_grouped_gemm(const GroupedArgs& a, cudaStream_t stream);

// W4A16 decode GEMMs (w4a16_workspace_bytes is 0: they need no workspace).
size_t w4a16_workspace_bytes(int64_t M, int64_t N, int64_t K);
q4_status launch_w4a16(const void* A, const uint8_t* Wq, const uint16_t* Ws, int64_t M, int64_t N,
                       int64_t K, void* C, void* ws, size_t ws_bytes, cudaStream_t stream);
// FP4 weights: Wsf row-major E4M3 (nvfp4, tensor scale *wg) or E8M0 bytes
q4_status launch_w4a16_fp4(const void* A, const uint8_t* Wq, const uint8_t* Wsf, const float* wg,
                           bool nvfp4, int64_t M, int64_t N, int64_t K, void* C, void* ws,
                           size_t ws_bytes, cudaStream_t stream);

// FP8 blockwise: block_rows 1 (activations, blocks (1, 128)) or 128 (weights,
// 128 x 128); codes [rows, K] E4M3 bytes, scales FP32 row-major per block.
q4_status launch_quant_fp8(const void* x, int dtype, int64_t rows, int64_t K, int block_rows,
                           uint8_t* codes, float* scales, cudaStream_t stream);
// Block-promoted FP8 GEMM: C [M, N] = sum over K blocks of sa * sb * (qa . qb^T).
q4_status launch_fp8_gemm(const uint8_t* qa, const float* sa, const uint8_t* qb, const float* sb,
                          int64_t M, int64_t N, int64_t K, void* C, int c_dtype,
                          cudaStream_t stream);

// W4A8: FP8 activations x INT4 g128 weights on the FP8 tensor cores; wsc is the
// FP32 [K/128, N] copy of the FP16 weight scales (launch_w4a8_scales).
q4_status launch_w4a8_scales(const uint16_t* s16, int64_t N, int64_t KB, float* out,
                             cudaStream_t stream);
q4_status launch_w4a8_gemm(const uint8_t* qa, const float* sa, const uint8_t* wq, const float* wsc,
                           int64_t M, int64_t N, int64_t K, void* C, int c_dtype,
                           cudaStream_t stream);

// TMA descriptor creation through the driver entry point.
q4_status make_tmap_2d_u8(CUtensorMap* map, const void* base, uint64_t inner_bytes, uint64_t rows,
                          uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_rows,
                          bool swizzle128);

// A byte tensor viewed as [d2][d1][d0] (d0 contiguous; s1, s2 the byte
// pitches of d1 and d2), boxes of b0 x b1 x b2.
q4_status make_tmap_3d_u8(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1,
                          uint64_t d2, uint64_t s1, uint64_t s2, uint32_t b0, uint32_t b1,
                          uint32_t b2, bool swizzle128);

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Launch with programmatic dependent launch allowed: the kernel may start once
// the previous kernel's blocks have exited, before that grid has completed;
// it calls pdl_wait() (common.cuh) before its first global-memory access, so
// it sees all of that kernel's writes.
template <typename... KArgs, typename... Args>
q4_status launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                     cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...) == cudaSuccess ? Q4_OK
                                                                                    : Q4_ERR_CUDA;
}
inline size_t mma_scales_bytes(int64_t rows, int64_t nsf) {
  return (size_t)(ceil_div(rows, 128) * 128) * (size_t)(ceil_div(nsf, 4) * 4);
}

}  // namespace q4
