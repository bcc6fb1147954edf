// gemm_w4a4_nvfp4_noalloc: the NVFP4 W4A4 GEMM with the activations given raw
// and quantized on the fly, for callers that cannot hand the library any
// device memory beyond inputs and outputs.
//
// The regular entry point quantizes the activations into a caller-provided
// workspace.  Some callers have no way to provide one: a plugin or custom-op
// interface that passes only input and output buffers, or an engine whose
// memory pool is fully reserved at start-up.  This variant keeps its scratch -- the quantized activations and
// their scales, the amax accumulator and the tensor scale -- in one file-scope
// device array of fixed size, so nothing is allocated per call.
//
// Limits and sharing rules (also stated in include/q4gemm.h):
//  * the scratch is kNoAllocScratchBytes (16 MiB) per GPU that loads the
//    library, held until the process exits; problems whose quantized
//    activations need more are rejected with Q4_ERR_SCRATCH_TOO_SMALL;
//  * every call uses the same array, so calls that overlap on the GPU (other
//    streams, other host threads) race; serialize them;
//  * the first call on each device looks up the array's device address with
//    cudaGetSymbolAddress (once per device, with that device current).
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace q4 {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;
constexpr int kMaxDev = 64;

// Device-side scratch.  In host code this name is only a stand-in for the
// symbol: its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

uint8_t* g_scratch_ptr[kMaxDev] = {nullptr};
std::mutex g_scratch_mu;

inline size_t al256(size_t x) { return (x + 255) & ~size_t(255); }

// Device address of this device's scratch array (looked up once per device).
q4_status scratch_for_current_device(uint8_t** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return Q4_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return Q4_ERR_CUDA;
    g_scratch_ptr[dev] = static_cast<uint8_t*>(p);
  }
  *out = g_scratch_ptr[dev];
  return Q4_OK;
}

}  // namespace
}  // namespace q4

using namespace q4;

extern "C" size_t q4_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

extern "C" size_t q4_noalloc_required_bytes(int64_t M, int64_t K) {
  if (M < 0 || K < 0) return 0;
  return 256 + al256((size_t)M * (size_t)(K / 2)) + al256(mma_scales_bytes(M, K / 16));
}

extern "C" q4_status gemm_w4a4_nvfp4_noalloc(const void* A, int a_dtype, const q4_operand* B,
                                             int64_t M, int64_t N, int64_t K, void* C,
                                             int c_dtype, q4_stream_t stream) {
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (M < 0 || N < 0 || K <= 0) return Q4_ERR_INVALID_ARG;
  if (K % 256) return Q4_ERR_UNSUPPORTED_SHAPE;
  if (M > INT32_MAX / 2 || N > INT32_MAX / 2) return Q4_ERR_UNSUPPORTED_SHAPE;
  if (c_dtype != Q4_F32 && c_dtype != Q4_BF16) return Q4_ERR_INVALID_ARG;
  if (a_dtype != Q4_F32 && a_dtype != Q4_BF16 && a_dtype != Q4_F16) return Q4_ERR_INVALID_ARG;
  if (!B || B->raw || B->scale_layout != Q4_SCALES_MMA) return Q4_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return Q4_OK;
  if (!A || !C || !B->codes || !B->scales || !B->tensor_scale) return Q4_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(C) |
       reinterpret_cast<uintptr_t>(B->codes) | reinterpret_cast<uintptr_t>(B->scales)) & 15)
    return Q4_ERR_INVALID_ARG;
  if (q4_noalloc_required_bytes(M, K) > kNoAllocScratchBytes) return Q4_ERR_SCRATCH_TOO_SMALL;

  uint8_t* base = nullptr;
  q4_status st = scratch_for_current_device(&base);
  if (st != Q4_OK) return st;
  unsigned* amax = reinterpret_cast<unsigned*>(base);
  float* g = reinterpret_cast<float*>(base + 16);
  uint8_t* codes = base + 256;
  uint8_t* sf = codes + al256((size_t)M * (size_t)(K / 2));

  // the amax accumulator keeps the previous call's value: clear it first
  Q4_CUDA_TRY(cudaMemsetAsync(amax, 0, sizeof(unsigned), s));
  if ((st = launch_amax(A, a_dtype, M * K, amax, s)) != Q4_OK) return st;
  if ((st = launch_quant_nvfp4(A, a_dtype, M, K, codes, sf, Q4_SCALES_MMA, amax, g, s)) != Q4_OK)
    return st;
  Fp4GemmArgs a = {};
  a.a_codes = codes; a.a_scales = sf; a.a_g = g;
  a.b_codes = B->codes; a.b_scales = B->scales; a.b_g = B->tensor_scale;
  a.M = M; a.N = N; a.K = K; a.C = C; a.c_dtype = c_dtype; a.nvfp4 = true;
  return launch_fp4_gemm(a, s);
}
