// The C ABI of q4gemm (declared in include/q4gemm.h): host-side argument
// checks, workspace carving, dispatch to the kernels, the device status word
// and TMA descriptor creation.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace q4 {

// First error latched by any kernel on this device (0 = none).
__device__ int g_q4_status = 0;

namespace {
constexpr int kMaxDevices = 64;
std::atomic<int> g_wait_ms{2000};
int* g_status_ptr[kMaxDevices] = {nullptr};
int g_sms[kMaxDevices] = {0};
std::mutex g_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int current_device() {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return -1;
  return d;
}

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Sequential carving of a caller-provided workspace.
struct Carver {
  uint8_t* base;
  size_t cap, used;
  uint8_t* take(size_t bytes) {
    uint8_t* p = base ? base + used : nullptr;
    used += align256(bytes);
    return p;
  }
  bool ok() const { return used <= cap; }
};

bool valid_dtype(int d) { return d == Q4_F32 || d == Q4_BF16 || d == Q4_F16; }
}  // namespace

int* device_status_ptr() {
  const int d = current_device();
  if (d < 0) return nullptr;
  if (!g_status_ptr[d]) {
    std::lock_guard<std::mutex> lk(g_mu);
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_q4_status) != cudaSuccess) return nullptr;
    g_status_ptr[d] = static_cast<int*>(p);
  }
  return g_status_ptr[d];
}

unsigned long long wait_budget_ns() { return (unsigned long long)g_wait_ms.load() * 1000000ull; }

int num_sms() {
  const int d = current_device();
  if (d < 0) return 1;
  if (!g_sms[d]) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d);
    g_sms[d] = n > 0 ? n : 1;
  }
  return g_sms[d];
}

q4_status make_tmap_2d_u8(CUtensorMap* map, const void* base, uint64_t inner_bytes, uint64_t rows,
                          uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_rows,
                          bool swizzle128) {
  if (!g_encode) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                           &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !fn)
        return Q4_ERR_CUDA;
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
  }
  const cuuint64_t dims[2] = {inner_bytes, rows};
  const cuuint64_t strides[1] = {row_stride_bytes};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims,
                              strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? Q4_OK : Q4_ERR_CUDA;
}

// A byte tensor viewed as [d2][d1][d0] with element pitches s1 and s2 for d1
// and d2 (d0 contiguous), boxes of b0 x b1 x b2, optionally 128-byte swizzled.
q4_status make_tmap_3d_u8(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1,
                          uint64_t d2, uint64_t s1, uint64_t s2, uint32_t b0, uint32_t b1,
                          uint32_t b2, bool swizzle128) {
  CUtensorMap dummy;
  q4_status st = make_tmap_2d_u8(&dummy, base, 16, 1, 16, 16, 1, false);  // loads the encoder
  if (st != Q4_OK) return st;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {s1, s2};
  const cuuint32_t box[3] = {b0, b1, b2};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims,
                              strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? Q4_OK : Q4_ERR_CUDA;
}

namespace {

// Workspace plan of one FP4 GEMM operand given raw or with row-major scales.
struct OperandPlan {
  uint8_t* codes;
  uint8_t* sf;
  unsigned* amax;
  float* g;
};

OperandPlan plan_operand(Carver& c, int64_t rows, int64_t K, int block, bool nv) {
  OperandPlan pl;
  pl.codes = c.take((size_t)rows * (size_t)(K / 2));
  pl.sf = c.take(mma_scales_bytes(rows, K / block));
  uint8_t* small = c.take(256);
  pl.amax = reinterpret_cast<unsigned*>(small);
  pl.g = reinterpret_cast<float*>(small + 16);
  (void)nv;
  return pl;
}

q4_status check_operand(const q4_operand* op, int64_t rows, bool nv) {
  if (!op) return Q4_ERR_INVALID_ARG;
  if (rows == 0) return Q4_OK;
  if (op->raw) {
    if (!valid_dtype(op->raw_dtype) || !aligned(op->raw, 16)) return Q4_ERR_INVALID_ARG;
    return Q4_OK;
  }
  if (!op->codes || !op->scales || !aligned(op->codes, 16) || !aligned(op->scales, 16))
    return Q4_ERR_INVALID_ARG;
  if (op->scale_layout != Q4_SCALES_ROWMAJOR && op->scale_layout != Q4_SCALES_MMA)
    return Q4_ERR_INVALID_ARG;
  if (nv && !op->tensor_scale) return Q4_ERR_INVALID_ARG;
  return Q4_OK;
}

// Bring an operand into (codes, MMA-layout scales, tensor scale) form.
q4_status resolve_operand(const q4_operand* op, int64_t rows, int64_t K, bool nv,
                          const OperandPlan& pl, cudaStream_t s, const uint8_t** codes,
                          const uint8_t** sf, const float** g) {
  const int block = nv ? 16 : 32;
  if (rows == 0) {
    *codes = op->codes; *sf = op->scales; *g = op->tensor_scale;
    return Q4_OK;
  }
  q4_status st;
  if (op->raw) {
    if (nv) {
      Q4_CUDA_TRY(cudaMemsetAsync(pl.amax, 0, sizeof(unsigned), s));
      if ((st = launch_amax(op->raw, op->raw_dtype, rows * K, pl.amax, s)) != Q4_OK) return st;
      if ((st = launch_quant_nvfp4(op->raw, op->raw_dtype, rows, K, pl.codes, pl.sf, Q4_SCALES_MMA,
                                   pl.amax, pl.g, s)) != Q4_OK)
        return st;
      *g = pl.g;
    } else {
      if ((st = launch_quant_mxfp4(op->raw, op->raw_dtype, rows, K, pl.codes, pl.sf, Q4_SCALES_MMA,
                                   s)) != Q4_OK)
        return st;
      *g = nullptr;
    }
    *codes = pl.codes;
    *sf = pl.sf;
    return Q4_OK;
  }
  *codes = op->codes;
  *g = nv ? op->tensor_scale : nullptr;
  if (op->scale_layout == Q4_SCALES_MMA) {
    *sf = op->scales;
    return Q4_OK;
  }
  if ((st = launch_scales_to_mma(op->scales, rows, K / block, pl.sf, s)) != Q4_OK) return st;
  *sf = pl.sf;
  return Q4_OK;
}

// The operands' quantized copies, then room for split-K partial sums.
size_t gemm_ws_bytes(int64_t M, int64_t N, int64_t K, int block) {
  Carver c{nullptr, 0, 0};
  plan_operand(c, M, K, block, block == 16);
  plan_operand(c, N, K, block, block == 16);
  c.take(fp4_splitk_partial_bytes(M, N, K, num_sms()));
  return c.used;
}

// The split-K partial region at the end of a carved workspace, when ws holds
// it (otherwise the partial sums meet in distributed shared memory).
void plan_partials(Carver& c, void* ws, int64_t M, int64_t N, int64_t K, Fp4GemmArgs& g) {
  const size_t bytes = fp4_splitk_partial_bytes(M, N, K, num_sms());
  uint8_t* part = c.take(bytes);
  if (bytes && ws && aligned(ws, 256) && c.ok()) {
    g.part_ws = part;
    g.part_ws_bytes = bytes;
  }
}

struct MoePlan {
  uint8_t* tok_codes;
  uint8_t* tok_sf;
  unsigned* amax;
  float* g;
  int32_t* sched;
  uint8_t* routed_sf;
  int64_t cap_rows;
  uint8_t* routed_codes;  // [R, K/2]: the routed rows' codes, in routed order
};

MoePlan plan_moe(Carver& c, int64_t T, int64_t K, int E, int64_t R) {
  MoePlan pl;
  pl.tok_codes = c.take((size_t)T * (size_t)(K / 2));
  pl.tok_sf = c.take((size_t)T * (size_t)(K / 16));
  uint8_t* small = c.take(256);
  pl.amax = reinterpret_cast<unsigned*>(small);
  pl.g = reinterpret_cast<float*>(small + 16);
  pl.sched = reinterpret_cast<int32_t*>(c.take((size_t)(E + 1) * 4));
  pl.cap_rows = (ceil_div(R, 128) + E) * 128;
  pl.routed_sf = c.take(mma_scales_bytes(pl.cap_rows, K / 16));
  pl.routed_codes = c.take((size_t)R * (size_t)(K / 2));
  return pl;
}

q4_status gemm_fp4_common(bool nv, const q4_operand* A, const q4_operand* B, int64_t M, int64_t N,
                          int64_t K, void* C, int c_dtype, void* ws, size_t ws_bytes,
                          q4_stream_t stream) {
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (M < 0 || N < 0 || K <= 0) return Q4_ERR_INVALID_ARG;
  if (K % 256) return Q4_ERR_UNSUPPORTED_SHAPE;
  if (M > INT32_MAX / 2 || N > INT32_MAX / 2) return Q4_ERR_UNSUPPORTED_SHAPE;
  if (c_dtype != Q4_F32 && c_dtype != Q4_BF16) return Q4_ERR_INVALID_ARG;
  q4_status st;
  if ((st = check_operand(A, M, nv)) != Q4_OK) return st;
  if ((st = check_operand(B, N, nv)) != Q4_OK) return st;
  if (M == 0 || N == 0) return Q4_OK;
  if (!C || !aligned(C, 16)) return Q4_ERR_INVALID_ARG;
  const int block = nv ? 16 : 32;
  const bool need_ws = A->raw || B->raw || A->scale_layout == Q4_SCALES_ROWMAJOR ||
                       B->scale_layout == Q4_SCALES_ROWMAJOR;
  Carver c{static_cast<uint8_t*>(ws), ws_bytes, 0};
  const OperandPlan pa = plan_operand(c, M, K, block, nv);
  const OperandPlan pb = plan_operand(c, N, K, block, nv);
  if (need_ws && (!ws || !aligned(ws, 256) || !c.ok())) return Q4_ERR_WORKSPACE;
  Fp4GemmArgs g = {};
  plan_partials(c, ws, M, N, K, g);
  if ((st = resolve_operand(A, M, K, nv, pa, s, &g.a_codes, &g.a_scales, &g.a_g)) != Q4_OK) return st;
  if ((st = resolve_operand(B, N, K, nv, pb, s, &g.b_codes, &g.b_scales, &g.b_g)) != Q4_OK) return st;
  g.M = M; g.N = N; g.K = K; g.C = C; g.c_dtype = c_dtype; g.nvfp4 = nv;
  return launch_fp4_gemm(g, s);
}

}  // namespace
}  // namespace q4

namespace q4 {
namespace {
// One warp waits, through the same bounded wait as every pipeline barrier, on
// an mbarrier that nothing arrives on: the wait gives up after ctl.wait_ns,
// latches Q4_ERR_TIMEOUT and the kernel returns (no trap, nothing left
// pending), so the failure path can be exercised without harming the context.
__global__ void wait_probe_kernel(KernelCtl ctl) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
    abort_flag = 0;
  }
  __syncwarp();
  if (threadIdx.x == 0) mbar_wait(smem_u32(&bar), 0, ctl, &abort_flag);
  __syncwarp();
}
}  // namespace
}  // namespace q4

using namespace q4;

extern "C" {

size_t q4_mma_scales_bytes(int64_t rows, int64_t nsf) {
  if (rows < 0 || nsf < 0) return 0;
  return mma_scales_bytes(rows, nsf);
}

size_t q4_workspace_size(int op, int64_t M, int64_t N, int64_t K) {
  if (M < 0 || N < 0 || K < 0) return 0;
  switch (op) {
    case Q4_OP_QUANTIZE_NVFP4: return 256;
    case Q4_OP_GEMM_W4A4_NVFP4: return gemm_ws_bytes(M, N, K, 16);
    case Q4_OP_GEMM_W4A4_MXFP4: return gemm_ws_bytes(M, N, K, 32);
    case Q4_OP_GEMM_W4A4_MXFP4_FUSED: return 256 + gemm_ws_bytes(M, N, K, 32);
    case Q4_OP_GEMM_W4A16_INT4:
    case Q4_OP_GEMM_W4A16_NVFP4:
    case Q4_OP_GEMM_W4A16_MXFP4: return w4a16_workspace_bytes(M, N, K);
    case Q4_OP_GROUPED_GEMM_MOE: return 0;  // needs E and R: q4_workspace_size_moe
    case Q4_OP_GEMM_FP8_BLOCKWISE:
    case Q4_OP_GEMM_W4A8: return 0;
    default: return 0;
  }
}

size_t q4_workspace_size_moe(int64_t T, int64_t N, int64_t K, int E, int64_t R) {
  (void)N;
  if (T < 0 || K < 0 || E < 0 || R < 0) return 0;
  Carver c{nullptr, 0, 0};
  plan_moe(c, T, K, E, R);
  return c.used;
}

q4_status quantize_nvfp4_ex(const void* x, int x_dtype, int64_t rows, int64_t K, uint8_t* codes,
                            uint8_t* scales, int scale_layout, int rounding, float* tensor_scale,
                            void* ws, size_t ws_bytes, q4_stream_t stream) {
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (rows < 0 || K <= 0 || !valid_dtype(x_dtype)) return Q4_ERR_INVALID_ARG;
  if (rounding != Q4_ROUND_PAGES && rounding != Q4_ROUND_RNE) return Q4_ERR_INVALID_ARG;
  if (K % 16) return Q4_ERR_UNSUPPORTED_SHAPE;
  if (scale_layout != Q4_SCALES_ROWMAJOR && scale_layout != Q4_SCALES_MMA) return Q4_ERR_INVALID_ARG;
  if (!tensor_scale) return Q4_ERR_INVALID_ARG;
  if (!ws || ws_bytes < 256 || !aligned(ws, 256)) return Q4_ERR_WORKSPACE;
  if (rows > 0 && (!x || !codes || !scales || !aligned(x, 16) || !aligned(codes, 16)))
    return Q4_ERR_INVALID_ARG;
  unsigned* amax = static_cast<unsigned*>(ws);
  Q4_CUDA_TRY(cudaMemsetAsync(amax, 0, sizeof(unsigned), s));
  q4_status st;
  if (rows == 0) {
    // g of an empty tensor: max(0, 1e-12) / 2688
    const float g = 1e-12f / 2688.0f;
    Q4_CUDA_TRY(cudaMemcpyAsync(tensor_scale, &g, sizeof(float), cudaMemcpyHostToDevice, s));
    Q4_CUDA_TRY(cudaStreamSynchronize(s));
    return Q4_OK;
  }
  if ((st = launch_amax(x, x_dtype, rows * K, amax, s)) != Q4_OK) return st;
  return launch_quant_nvfp4(x, x_dtype, rows, K, codes, scales, scale_layout, amax, tensor_scale, s,
                            rounding == Q4_ROUND_RNE);
}

q4_status quantize_nvfp4(const void* x, int x_dtype, int64_t rows, int64_t K, uint8_t* codes,
                         uint8_t* scales, int scale_layout, float* tensor_scale, void* ws,
                         size_t ws_bytes, q4_stream_t stream) {
  return quantize_nvfp4_ex(x, x_dtype, rows, K, codes, scales, scale_layout, Q4_ROUND_PAGES,
                           tensor_scale, ws, ws_bytes, stream);
}

q4_status quantize_mxfp4_ex(const void* x, int x_dtype, int64_t rows, int64_t K, uint8_t* codes,
                            uint8_t* scales, int scale_layout, int rounding, q4_stream_t stream) {
  if (rows < 0 || K <= 0 || !valid_dtype(x_dtype)) return Q4_ERR_INVALID_ARG;
  if (rounding != Q4_ROUND_PAGES && rounding != Q4_ROUND_RNE) return Q4_ERR_INVALID_ARG;
  if (K % 32) return Q4_ERR_UNSUPPORTED_SHAPE;
  if (scale_layout != Q4_SCALES_ROWMAJOR && scale_layout != Q4_SCALES_MMA) return Q4_ERR_INVALID_ARG;
  if (rows == 0) return Q4_OK;
  if (!x || !codes || !scales || !aligned(x, 16) || !aligned(codes, 16)) return Q4_ERR_INVALID_ARG;
  return launch_quant_mxfp4(x, x_dtype, rows, K, codes, scales, scale_layout,
                            reinterpret_cast<cudaStream_t>(stream), rounding == Q4_ROUND_RNE);
}

q4_status quantize_mxfp4(const void* x, int x_dtype, int64_t rows, int64_t K, uint8_t* codes,
                         uint8_t* scales, int scale_layout, q4_stream_t stream) {
  return quantize_mxfp4_ex(x, x_dtype, rows, K, codes, scales, scale_layout, Q4_ROUND_PAGES,
                           stream);
}

q4_status quantize_int4_g128(const void* x, int x_dtype, int64_t rows, int64_t K, uint8_t* codes,
                             uint16_t* scales, q4_stream_t stream) {
  if (rows < 0 || K <= 0 || !valid_dtype(x_dtype)) return Q4_ERR_INVALID_ARG;
  if (K % 128) return Q4_ERR_UNSUPPORTED_SHAPE;
  if (rows == 0) return Q4_OK;
  if (!x || !codes || !scales || !aligned(x, 16) || !aligned(codes, 16) || !aligned(scales, 2))
    return Q4_ERR_INVALID_ARG;
  return launch_quant_int4(x, x_dtype, rows, K, codes, scales,
                           reinterpret_cast<cudaStream_t>(stream));
}

q4_status q4_scales_to_mma(const uint8_t* src, int64_t rows, int64_t nsf, uint8_t* dst,
                           q4_stream_t stream) {
  if (rows < 0 || nsf < 0) return Q4_ERR_INVALID_ARG;
  if (rows == 0 || nsf == 0) return Q4_OK;
  if (!src || !dst) return Q4_ERR_INVALID_ARG;
  return launch_scales_to_mma(src, rows, nsf, dst, reinterpret_cast<cudaStream_t>(stream));
}

q4_status gemm_w4a4_nvfp4(const q4_operand* A, const q4_operand* B, int64_t M, int64_t N,
                          int64_t K, void* C, int c_dtype, void* ws, size_t ws_bytes,
                          q4_stream_t stream) {
  return gemm_fp4_common(true, A, B, M, N, K, C, c_dtype, ws, ws_bytes, stream);
}

q4_status gemm_w4a4_mxfp4(const q4_operand* A, const q4_operand* B, int64_t M, int64_t N,
                          int64_t K, void* C, int c_dtype, void* ws, size_t ws_bytes,
                          q4_stream_t stream) {
  return gemm_fp4_common(false, A, B, M, N, K, C, c_dtype, ws, ws_bytes, stream);
}

q4_status gemm_w4a4_mxfp4_fused(const void* A_raw, int a_dtype, const q4_operand* B, int64_t M,
                                int64_t N, int64_t K, void* C, int c_dtype, void* ws,
                                size_t ws_bytes, q4_stream_t stream) {
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (M < 0 || N < 0 || K <= 0) return Q4_ERR_INVALID_ARG;
  if (K % 256) return Q4_ERR_UNSUPPORTED_SHAPE;
  if (M > INT32_MAX / 2 || N > INT32_MAX / 2) return Q4_ERR_UNSUPPORTED_SHAPE;
  if (c_dtype != Q4_F32 && c_dtype != Q4_BF16) return Q4_ERR_INVALID_ARG;
  if (a_dtype != Q4_F32 && a_dtype != Q4_BF16 && a_dtype != Q4_F16) return Q4_ERR_INVALID_ARG;
  q4_status st;
  if ((st = check_operand(B, N, false)) != Q4_OK) return st;
  if (M == 0 || N == 0) return Q4_OK;
  if (!A_raw || !aligned(A_raw, 16)) return Q4_ERR_INVALID_ARG;
  if (!C || !aligned(C, 16)) return Q4_ERR_INVALID_ARG;
  Carver c{static_cast<uint8_t*>(ws), ws_bytes, 0};
  unsigned* gate = reinterpret_cast<unsigned*>(c.take(256));
  const OperandPlan pa = plan_operand(c, M, K, 32, false);
  const OperandPlan pb = plan_operand(c, N, K, 32, false);
  if (!ws || !aligned(ws, 256) || !c.ok()) return Q4_ERR_WORKSPACE;
  Fp4GemmArgs g = {};
  plan_partials(c, ws, M, N, K, g);
  if (M * (K / 16) < ((int64_t)1 << 31)) {  // the prologue's unit indices are 32-bit
    g.a_raw = A_raw;
    g.a_dtype = a_dtype;
    g.a_codes = pa.codes;
    g.a_scales = pa.sf;
    g.gate = gate;
  } else {
    q4_operand a = {A_raw, a_dtype, nullptr, nullptr, Q4_SCALES_MMA, nullptr};
    if ((st = resolve_operand(&a, M, K, false, pa, s, &g.a_codes, &g.a_scales, &g.a_g)) != Q4_OK)
      return st;
  }
  if ((st = resolve_operand(B, N, K, false, pb, s, &g.b_codes, &g.b_scales, &g.b_g)) != Q4_OK)
    return st;
  g.M = M; g.N = N; g.K = K; g.C = C; g.c_dtype = c_dtype; g.nvfp4 = false;
  return launch_fp4_gemm(g, s);
}

namespace {
q4_status w4a16_check(const void* A_bf16, const uint8_t* Wq, const void* Ws, int64_t M, int64_t N,
                      int64_t K, void* C_bf16, void* ws, size_t ws_bytes) {
  if (M < 0 || N < 0 || K <= 0) return Q4_ERR_INVALID_ARG;
  if (K % 128) return Q4_ERR_UNSUPPORTED_SHAPE;
  if (M > INT32_MAX / 2 || N > INT32_MAX / 2 || K > INT32_MAX / 2) return Q4_ERR_UNSUPPORTED_SHAPE;
  if (ceil_div(M, 16) > 65535) return Q4_ERR_UNSUPPORTED_SHAPE;
  if (M == 0 || N == 0) return Q4_OK;
  if (!A_bf16 || !Wq || !Ws || !C_bf16 || !aligned(A_bf16, 16) || !aligned(Wq, 16) ||
      !aligned(C_bf16, 2))
    return Q4_ERR_INVALID_ARG;
  const size_t need = w4a16_workspace_bytes(M, N, K);
  if (need && (!ws || !aligned(ws, 256) || ws_bytes < need)) return Q4_ERR_WORKSPACE;
  return Q4_OK;
}
}  // namespace

q4_status gemm_w4a16_int4(const void* A_bf16, const uint8_t* Wq, const uint16_t* Ws, int64_t M,
                          int64_t N, int64_t K, void* C_bf16, void* ws, size_t ws_bytes,
                          q4_stream_t stream) {
  q4_status st = w4a16_check(A_bf16, Wq, Ws, M, N, K, C_bf16, ws, ws_bytes);
  if (st != Q4_OK || M == 0 || N == 0) return st;
  if (!aligned(Ws, 2)) return Q4_ERR_INVALID_ARG;
  return launch_w4a16(A_bf16, Wq, Ws, M, N, K, C_bf16, ws, ws_bytes,
                      reinterpret_cast<cudaStream_t>(stream));
}

static q4_status w4a16_fp4(const void* A_bf16, const uint8_t* Wq, const uint8_t* Ws,
                           const float* w_g, bool nvfp4, int64_t M, int64_t N, int64_t K,
                           void* C_bf16, void* ws, size_t ws_bytes, q4_stream_t stream) {
  if (nvfp4 && M > 0 && N > 0 && (!w_g || !aligned(w_g, 4) || !aligned(Ws, 2)))
    return Q4_ERR_INVALID_ARG;
  q4_status st = w4a16_check(A_bf16, Wq, Ws, M, N, K, C_bf16, ws, ws_bytes);
  if (st != Q4_OK || M == 0 || N == 0) return st;
  return launch_w4a16_fp4(A_bf16, Wq, Ws, w_g, nvfp4, M, N, K, C_bf16, ws, ws_bytes,
                          reinterpret_cast<cudaStream_t>(stream));
}

q4_status gemm_w4a16_nvfp4(const void* A_bf16, const uint8_t* Wq, const uint8_t* Ws,
                           const float* w_tensor_scale, int64_t M, int64_t N, int64_t K,
                           void* C_bf16, void* ws, size_t ws_bytes, q4_stream_t stream) {
  return w4a16_fp4(A_bf16, Wq, Ws, w_tensor_scale, true, M, N, K, C_bf16, ws, ws_bytes, stream);
}

q4_status gemm_w4a16_mxfp4(const void* A_bf16, const uint8_t* Wq, const uint8_t* Ws, int64_t M,
                           int64_t N, int64_t K, void* C_bf16, void* ws, size_t ws_bytes,
                           q4_stream_t stream) {
  return w4a16_fp4(A_bf16, Wq, Ws, nullptr, false, M, N, K, C_bf16, ws, ws_bytes, stream);
}

q4_status quantize_fp8_blockwise(const void* x, int x_dtype, int64_t rows, int64_t K,
                                 int block_rows, uint8_t* codes, float* scales,
                                 q4_stream_t stream) {
  if (rows < 0 || K <= 0 || !valid_dtype(x_dtype) || (block_rows != 1 && block_rows != 128))
    return Q4_ERR_INVALID_ARG;
  if (K % 128 || rows % block_rows) return Q4_ERR_UNSUPPORTED_SHAPE;
  if ((rows / block_rows) * (K / 128) > INT32_MAX / 2) return Q4_ERR_UNSUPPORTED_SHAPE;
  if (rows == 0) return Q4_OK;
  if (!x || !codes || !scales || !aligned(x, 16) || !aligned(codes, 16) || !aligned(scales, 4))
    return Q4_ERR_INVALID_ARG;
  return launch_quant_fp8(x, x_dtype, rows, K, block_rows, codes, scales,
                          reinterpret_cast<cudaStream_t>(stream));
}

q4_status gemm_fp8_blockwise(const uint8_t* qa, const float* sa, const uint8_t* qb,
                             const float* sb, int64_t M, int64_t N, int64_t K, void* C,
                             int c_dtype, void* ws, size_t ws_bytes, q4_stream_t stream) {
  (void)ws;  // needs no workspace (q4_workspace_size gives 0)
  (void)ws_bytes;
  if (M < 0 || N < 0 || K <= 0 || (c_dtype != Q4_F32 && c_dtype != Q4_BF16))
    return Q4_ERR_INVALID_ARG;
  if (K % 128 || N % 128) return Q4_ERR_UNSUPPORTED_SHAPE;
  if (M > INT32_MAX / 2 || N > INT32_MAX / 2 || K > INT32_MAX / 2 ||
      ceil_div(M, 128) * (N / 128) > INT32_MAX / 2)
    return Q4_ERR_UNSUPPORTED_SHAPE;
  if (M == 0 || N == 0) return Q4_OK;
  if (!qa || !sa || !qb || !sb || !C || !aligned(qa, 16) || !aligned(qb, 16) || !aligned(C, 16) ||
      !aligned(sa, 4) || !aligned(sb, 4))
    return Q4_ERR_INVALID_ARG;
  return launch_fp8_gemm(qa, sa, qb, sb, M, N, K, C, c_dtype, reinterpret_cast<cudaStream_t>(stream));
}

q4_status w4a8_weight_scales(const uint16_t* w_scales, int64_t N, int64_t K, float* w_scales_kn,
                             q4_stream_t stream) {
  if (N < 0 || K <= 0) return Q4_ERR_INVALID_ARG;
  if (K % 128 || N > INT32_MAX / 2 || K > INT32_MAX / 2) return Q4_ERR_UNSUPPORTED_SHAPE;
  if (N == 0) return Q4_OK;
  if (!w_scales || !w_scales_kn || !aligned(w_scales, 2) || !aligned(w_scales_kn, 4))
    return Q4_ERR_INVALID_ARG;
  return launch_w4a8_scales(w_scales, N, K / 128, w_scales_kn, reinterpret_cast<cudaStream_t>(stream));
}

q4_status gemm_w4a8(const uint8_t* qa, const float* sa, const uint8_t* w_codes,
                    const float* w_scales_kn, int64_t M, int64_t N, int64_t K, void* C,
                    int c_dtype, void* ws, size_t ws_bytes, q4_stream_t stream) {
  (void)ws;  // needs no workspace (q4_workspace_size gives 0)
  (void)ws_bytes;
  if (M < 0 || N < 0 || K <= 0 || (c_dtype != Q4_F32 && c_dtype != Q4_BF16))
    return Q4_ERR_INVALID_ARG;
  if (K % 128 || N % 128) return Q4_ERR_UNSUPPORTED_SHAPE;
  if (M > INT32_MAX / 2 || N > INT32_MAX / 2 || K > INT32_MAX / 2 ||
      ceil_div(M, 128) * (N / 128) > INT32_MAX / 2)
    return Q4_ERR_UNSUPPORTED_SHAPE;
  if (M == 0 || N == 0) return Q4_OK;
  if (!qa || !sa || !w_codes || !w_scales_kn || !C || !aligned(qa, 16) || !aligned(w_codes, 16) ||
      !aligned(w_scales_kn, 16) || !aligned(C, 16) || !aligned(sa, 4))
    return Q4_ERR_INVALID_ARG;
  return launch_w4a8_gemm(qa, sa, w_codes, w_scales_kn, M, N, K, C, c_dtype,
                          reinterpret_cast<cudaStream_t>(stream));
}

q4_status grouped_gemm_moe(const void* tokens_bf16, int64_t T, int64_t K,
                           const int32_t* expert_offsets, const int32_t* row_token, int64_t R,
                           int E, const q4_operand* W, int64_t N, void* C_bf16, void* ws,
                           size_t ws_bytes, q4_stream_t stream) {
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (T < 0 || K <= 0 || R < 0 || E < 0 || N < 0) return Q4_ERR_INVALID_ARG;
  if (!W || W->raw) return Q4_ERR_INVALID_ARG;  // the experts' weights come quantized
  if (W->scale_layout != Q4_SCALES_MMA && W->scale_layout != Q4_SCALES_ROWMAJOR) return Q4_ERR_INVALID_ARG;
  const uint8_t* W_codes = W->codes;
  const uint8_t* W_scales = W->scales;
  const float* W_tensor_scales = W->tensor_scale;
  if (K % 256) return Q4_ERR_UNSUPPORTED_SHAPE;
  if (E > 1024 || T > INT32_MAX / 2 || R > INT32_MAX / 2 || (int64_t)E * N > INT32_MAX / 2)
    return Q4_ERR_UNSUPPORTED_SHAPE;
  if (R == 0 || N == 0 || E == 0) return Q4_OK;
  if (T == 0) return Q4_ERR_INVALID_ARG;  // routed rows need tokens
  if (!tokens_bf16 || !expert_offsets || !row_token || !W_codes || !W_scales ||
      !W_tensor_scales || !C_bf16)
    return Q4_ERR_INVALID_ARG;
  if (!aligned(tokens_bf16, 16) || !aligned(W_codes, 16) || !aligned(W_scales, 16) ||
      !aligned(C_bf16, 16) || !aligned(expert_offsets, 4) || !aligned(row_token, 4))
    return Q4_ERR_INVALID_ARG;
  Carver c{static_cast<uint8_t*>(ws), ws_bytes, 0};
  const MoePlan pl = plan_moe(c, T, K, E, R);
  const bool w_rowmajor = W->scale_layout == Q4_SCALES_ROWMAJOR;
  const size_t w_sf_bytes = mma_scales_bytes(N, K / 16);  // one expert, tensor-core layout
  uint8_t* w_sf_mma = w_rowmajor ? c.take((size_t)E * w_sf_bytes) : nullptr;
  if (!ws || !aligned(ws, 256) || !c.ok()) return Q4_ERR_WORKSPACE;
  q4_status st;
  if (w_rowmajor) {  // [E, N, K/16] row-major -> E tensor-core-layout tensors
    if (N % 128 == 0) {  // whole 128-row blocks: the E experts form one tensor of E N rows
      if ((st = launch_scales_to_mma(W_scales, (int64_t)E * N, K / 16, w_sf_mma, s)) != Q4_OK) return st;
    } else {
      for (int e = 0; e < E; ++e)
        if ((st = launch_scales_to_mma(W_scales + (int64_t)e * N * (K / 16), N, K / 16,
                                       w_sf_mma + (size_t)e * w_sf_bytes, s)) != Q4_OK)
          return st;
    }
    W_scales = w_sf_mma;
  }
  // the tokens are quantized once, as one tensor with one tensor scale
  Q4_CUDA_TRY(cudaMemsetAsync(pl.amax, 0, sizeof(unsigned), s));
  if ((st = launch_amax(tokens_bf16, Q4_BF16, T * K, pl.amax, s)) != Q4_OK) return st;
  if ((st = launch_quant_nvfp4(tokens_bf16, Q4_BF16, T, K, pl.tok_codes, pl.tok_sf,
                               Q4_SCALES_ROWMAJOR, pl.amax, pl.g, s)) != Q4_OK)
    return st;
  if ((st = launch_grouped_prep(expert_offsets, row_token, E, pl.tok_sf, K / 16, pl.sched,
                                pl.routed_sf, pl.cap_rows, s)) != Q4_OK)
    return st;
  if ((st = launch_gather_rows(pl.tok_codes, row_token, R, K / 2, pl.routed_codes, s)) != Q4_OK)
    return st;
  GroupedArgs g = {};
  g.a_routed = pl.routed_codes; g.a_sf_rows = pl.routed_sf; g.a_g = pl.g;
  g.offsets = expert_offsets; g.sched = pl.sched;
  g.T = T; g.R = R; g.N = N; g.K = K; g.E = E;
  g.w_codes = W_codes; g.w_scales = W_scales; g.w_g = W_tensor_scales; g.C = C_bf16;
  return launch_grouped_gemm(g, s);
}

q4_status q4_sync_status(q4_stream_t stream) {
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return Q4_ERR_CUDA;
  int* d = device_status_ptr();
  if (!d) return Q4_ERR_CUDA;
  int h = 0;
  if (cudaMemcpyAsync(&h, d, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess) return Q4_ERR_CUDA;
  if (cudaMemsetAsync(d, 0, sizeof(int), s) != cudaSuccess) return Q4_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return Q4_ERR_CUDA;
  return h;
}

const char* q4_status_string(q4_status s) {
  switch (s) {
    case Q4_OK: return "ok";
    case Q4_ERR_INVALID_ARG: return "invalid argument";
    case Q4_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case Q4_ERR_CUDA: return "CUDA error";
    case Q4_ERR_TIMEOUT: return "kernel wait timed out";
    case Q4_ERR_NONFINITE: return "non-finite input";
    case Q4_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
    case Q4_ERR_SCRATCH_TOO_SMALL:
      return "problem larger than the fixed scratch of the no-allocation entry point";
    default: return "unknown status";
  }
}

int q4_set_wait_timeout_ms(int ms) {
  if (ms <= 0) return g_wait_ms.load();
  return g_wait_ms.exchange(ms);
}

q4_status q4_selftest_wait_timeout(q4_stream_t stream) {
  const KernelCtl ctl{device_status_ptr(), wait_budget_ns()};
  if (!ctl.status) return Q4_ERR_CUDA;
  wait_probe_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(ctl);
  return cudaGetLastError() == cudaSuccess ? Q4_OK : Q4_ERR_CUDA;
}

}  // extern "C"
