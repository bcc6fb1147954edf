/*
 * q4gemm: block-scaled 4-bit quantization and the GEMMs that consume it, for
 * one NVIDIA GB300 (sm_103a).
 *
 * Formats (all codes are packed two per byte: element 2j of a row in the low
 * nibble of byte j, element 2j+1 in the high nibble):
 *
 *  NVFP4   E2M1 codes, one E4M3 scale per 16 elements along K, one FP32 scale
 *          per tensor.  "Quantization in deployment" (anrans.github.io AI-infra
 *          handbook), section "Fake quantization" (nvfp4, fp4) and the format
 *          cheat sheet; "Quantization chains" (inferenceinterviews.com),
 *          section "Bits per weight, scales included".
 *  MXFP4   E2M1 codes, one E8M0 (power-of-two) scale per 32.  Same page,
 *          "Fake quantization" (mxfp4).
 *  INT4    symmetric integers in [-8, 7] (two's complement nibbles), one FP16
 *          scale per 128.  "Low-bit inference for very large MoE", section
 *          "Why quantization-aware training" (fake_int4), with the group of
 *          128 and FP16 scale of "Quantization chains", "Bits per weight".
 *  FP8     E4M3 bytes (one per element), one FP32 scale per 128 x 128 weight
 *          block or per (1, 128) activation block.  "Quantization in
 *          deployment", "Fake quantization" (fp8_blockwise) and exercise 2.
 *
 * The E2M1 code of a value y = clamp(x / S, -6, 6) is the nearest of
 * 0, 0.5, 1, 1.5, 2, 3, 4, 6 with ties going to the smaller magnitude; its
 * sign bit (bit 3) is set when x < 0.  Bit-exact definitions of every step
 * are in the documentation of each call below.
 *
 * Conventions for every call:
 *  - All data pointers are DEVICE pointers to caller-owned memory unless a
 *    parameter says otherwise.  The library never allocates device memory;
 *    calls that need scratch take a caller-provided workspace whose size is
 *    given by q4_workspace_size().  Workspaces must be 256-byte aligned.
 *  - Every call is asynchronous on the given CUDA stream (0 = legacy default
 *    stream).  Argument errors are detected on the host and returned before
 *    anything is launched.  Errors found by a kernel (a non-finite input, a
 *    pipeline wait that timed out) are latched in a device status word and
 *    returned by q4_sync_status().
 *  - Matrices are row-major.  GEMMs compute C = A . B^T with A [M, K] and B
 *    [N, K] (B is in the weight layout).
 *  - Block-scale tensors exist in two layouts:
 *      Q4_SCALES_ROWMAJOR  [rows, K / block], one byte per block;
 *      Q4_SCALES_MMA       the tensor-core layout: rows are grouped by 128
 *                          and scale columns by 4; the 512-byte tile of
 *                          row group R and column group J starts at
 *                          (R * ceil(nsf / 4) + J) * 512 and holds the scale
 *                          of row r, column s at
 *                          (r % 32) * 16 + ((r % 128) / 32) * 4 + s % 4.
 *                          Its size is ceil(rows / 128) * 128 * ceil(nsf / 4)
 *                          * 4 bytes (nsf = K / block); padding is zero.
 */
#ifndef Q4GEMM_H_
#define Q4GEMM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* q4_stream_t; /* the same type as cudaStream_t */

typedef int q4_status;
#define Q4_OK 0
#define Q4_ERR_INVALID_ARG (-1)       /* null pointer, negative size, bad enum, misalignment */
#define Q4_ERR_UNSUPPORTED_SHAPE (-2) /* K not a multiple of the required block, sizes too large */
#define Q4_ERR_CUDA (-3)              /* a CUDA runtime or driver call failed */
#define Q4_ERR_TIMEOUT (-4)           /* a kernel's bounded pipeline wait ran out */
#define Q4_ERR_NONFINITE (-5)         /* a quantizer saw a NaN or infinite input */
#define Q4_ERR_WORKSPACE (-6)         /* workspace missing, too small or misaligned */
#define Q4_ERR_SCRATCH_TOO_SMALL (-7) /* problem exceeds the fixed scratch of a no-allocation call */

typedef enum { Q4_F32 = 0, Q4_BF16 = 1, Q4_F16 = 2 } q4_dtype;
typedef enum { Q4_SCALES_ROWMAJOR = 0, Q4_SCALES_MMA = 1 } q4_scale_layout;
/* Tie rule of the E2M1 rounding step: the pages' (a value halfway between two
 * E2M1 magnitudes takes the smaller one) or IEEE round half to even (the even
 * code, mantissa bit 0).  Everything else is identical in both modes. */
typedef enum { Q4_ROUND_PAGES = 0, Q4_ROUND_RNE = 1 } q4_rounding;

/* Operation codes for q4_workspace_size(). */
typedef enum {
  Q4_OP_QUANTIZE_NVFP4 = 0,
  Q4_OP_GEMM_W4A4_NVFP4 = 1, /* M, N, K; both operands given raw (the largest case) */
  Q4_OP_GEMM_W4A4_MXFP4 = 2,
  Q4_OP_GEMM_W4A16_INT4 = 3,
  Q4_OP_GROUPED_GEMM_MOE = 4, /* M = number of tokens T, N, K; E and R via q4_workspace_size_moe */
  Q4_OP_GEMM_W4A16_NVFP4 = 5,
  Q4_OP_GEMM_W4A16_MXFP4 = 6,
  Q4_OP_GEMM_FP8_BLOCKWISE = 7, /* needs none today: 0 */
  Q4_OP_GEMM_W4A8 = 8,          /* needs none today: 0 */
  Q4_OP_GEMM_W4A4_MXFP4_FUSED = 9
} q4_op;

/*
 * One FP4 GEMM operand [rows, K].
 *  raw != NULL: the operand is given unquantized ([rows, K] in raw_dtype) and
 *               the GEMM call quantizes it into the workspace first (NVFP4:
 *               with its own per-tensor scale).  codes/scales/tensor_scale
 *               are then ignored.
 *  raw == NULL: codes [rows, K/2], scales in scale_layout and (NVFP4 only)
 *               tensor_scale, a device pointer to one float, as written by
 *               quantize_nvfp4 / quantize_mxfp4.
 */
typedef struct {
  const void* raw;
  int raw_dtype; /* q4_dtype */
  const uint8_t* codes;
  const uint8_t* scales;
  int scale_layout; /* q4_scale_layout */
  const float* tensor_scale;
} q4_operand;

/* Bytes of workspace the operation needs for these sizes (0 if none). */
size_t q4_workspace_size(int op, int64_t M, int64_t N, int64_t K);
size_t q4_workspace_size_moe(int64_t T, int64_t N, int64_t K, int E, int64_t R);

/* Size in bytes of a Q4_SCALES_MMA scale tensor for rows x nsf scales. */
size_t q4_mma_scales_bytes(int64_t rows, int64_t nsf);

/*
 * NVFP4 quantization of x [rows, K] (K % 16 == 0), "Quantization in
 * deployment", "Fake quantization" (nvfp4 then fp4).  In float32 with IEEE
 * rounding:
 *   g  = max(max|x|, 1e-12) / 2688                     (written to *tensor_scale)
 *   per block of 16 along K:
 *     t  = (amax_b / 6) / g;  bs = E4M3(t), round to nearest even
 *     S  = max(e4m3(bs), 1e-12) * g
 *     code = E2M1(clamp(x / S, -6, 6))   (ties to the smaller magnitude)
 *   a block whose scale byte is 0 gets all-zero codes.
 * codes: [rows, K/2]; scales: E4M3 bytes in scale_layout; tensor_scale: one
 * device float.  ws: q4_workspace_size(Q4_OP_QUANTIZE_NVFP4, rows, 0, K)
 * bytes (the amax accumulator).  Two kernels are launched (amax, quantize).
 */
q4_status quantize_nvfp4(const void* x, int x_dtype, int64_t rows, int64_t K, uint8_t* codes,
                         uint8_t* scales, int scale_layout, float* tensor_scale, void* ws,
                         size_t ws_bytes, q4_stream_t stream);

/*
 * MXFP4 quantization of x [rows, K] (K % 32 == 0), "Quantization in
 * deployment", "Fake quantization" (mxfp4).  Per block of 32:
 *   e = floor(log2(max(amax_b, 1e-12))) - 2  (exact, from the float bits)
 *   scale byte = e + 127 (E8M0);  code = E2M1(clamp(x / 2^e, -6, 6)).
 */
q4_status quantize_mxfp4(const void* x, int x_dtype, int64_t rows, int64_t K, uint8_t* codes,
                         uint8_t* scales, int scale_layout, q4_stream_t stream);

/*
 * The two FP4 quantizers with a choice of E2M1 tie rule (q4_rounding).
 * quantize_nvfp4 / quantize_mxfp4 are these with Q4_ROUND_PAGES.  With
 * Q4_ROUND_RNE an element whose quotient x / S (float32) lies exactly halfway
 * between two E2M1 magnitudes gets the even code (0.25 -> 0, 0.75 -> 1,
 * 1.25 -> 1, 1.75 -> 2, 2.5 -> 2, 3.5 -> 4, 5 -> 4); scales, tensor scale,
 * signs, layouts, workspace and errors are as in the calls above (an unknown
 * rounding value is Q4_ERR_INVALID_ARG).
 */
q4_status quantize_nvfp4_ex(const void* x, int x_dtype, int64_t rows, int64_t K, uint8_t* codes,
                            uint8_t* scales, int scale_layout, int rounding, float* tensor_scale,
                            void* ws, size_t ws_bytes, q4_stream_t stream);
q4_status quantize_mxfp4_ex(const void* x, int x_dtype, int64_t rows, int64_t K, uint8_t* codes,
                            uint8_t* scales, int scale_layout, int rounding, q4_stream_t stream);

/*
 * Symmetric INT4 quantization with one FP16 scale per 128 (K % 128 == 0),
 * "Low-bit inference for very large MoE", "Why quantization-aware training"
 * (fake_int4) with groups of 128:
 *   s16 = fp16_rne(amax_g / 7);  q = clamp(rint(x / float(s16)), -8, 7)
 *   (q = 0 where s16 == 0).  codes [rows, K/2]; scales [rows, K/128] FP16 bits.
 */
q4_status quantize_int4_g128(const void* x, int x_dtype, int64_t rows, int64_t K, uint8_t* codes,
                             uint16_t* scales, q4_stream_t stream);

/*
 * Scale re-layout: src [rows, nsf] row-major bytes -> dst in Q4_SCALES_MMA
 * layout (q4_mma_scales_bytes(rows, nsf) bytes, padding zeroed).  No page
 * prints this layout; it is the order in which the GB300 tensor cores read
 * block scales.
 */
q4_status q4_scales_to_mma(const uint8_t* src, int64_t rows, int64_t nsf, uint8_t* dst,
                           q4_stream_t stream);

/*
 * W4A4 GEMMs on the FP4 tensor cores ("Low-bit inference for very large
 * MoE", "Kernels on different hardware": activations quantized to FP4 too,
 * both operands enter the FP4 tensor cores).  C [M, N] = A_hat . B_hat^T
 * with FP32 accumulation, where
 *   NVFP4: x_hat = e2m1(code) * e4m3(scale) * g   (the product of the two
 *          tensor scales gA * gB is applied in the FP32 epilogue)
 *   MXFP4: x_hat = e2m1(code) * 2^(scale - 127)
 * c_dtype is Q4_F32 or Q4_BF16 (round to nearest even).  K % 256 == 0; M and
 * N are arbitrary (M, N >= 0).  Raw operands are quantized on the fly (see
 * q4_operand).  ws: q4_workspace_size(op, M, N, K) bytes.  For shapes with
 * few output tiles the GEMM splits K over a cluster of CTAs; with a
 * workspace of that full size their partial sums meet in it (through L2),
 * otherwise (ws NULL or smaller, allowed when both operands come quantized
 * with Q4_SCALES_MMA scales) in distributed shared memory, with the same
 * result bit for bit.
 */
q4_status gemm_w4a4_nvfp4(const q4_operand* A, const q4_operand* B, int64_t M, int64_t N,
                          int64_t K, void* C, int c_dtype, void* ws, size_t ws_bytes,
                          q4_stream_t stream);
q4_status gemm_w4a4_mxfp4(const q4_operand* A, const q4_operand* B, int64_t M, int64_t N,
                          int64_t K, void* C, int c_dtype, void* ws, size_t ws_bytes,
                          q4_stream_t stream);

/*
 * gemm_w4a4_mxfp4 with the activation quantization fused into the GEMM
 * ("Low-bit inference for very large MoE", "Kernels on different hardware":
 * the activations are quantized on the fly in the GEMM's prologue; the MXFP4
 * encode of "Quantization in deployment", "Fake quantization", mxfp4).  One
 * launch: every CTA first encodes its share of A's 32-element blocks into the
 * workspace, all CTAs meet at a grid-wide gate, then the main loop runs as in
 * gemm_w4a4_mxfp4 (results are bit-identical to it with A->raw = A_raw).
 * A_raw: [M, K] in a_dtype (Q4_F32, Q4_BF16 or Q4_F16), 16-byte aligned.
 * B, C, c_dtype, K, M, N: as for gemm_w4a4_mxfp4.
 * ws: q4_workspace_size(Q4_OP_GEMM_W4A4_MXFP4_FUSED, M, N, K) bytes, 256-byte
 *     aligned.  Its first 256 bytes hold the gate's counters: they must be
 *     zero before the first call on this workspace (e.g. one cudaMemsetAsync
 *     when it is allocated), and every call whose kernel finishes without an
 *     error leaves them zero again, so no reset is needed between calls.
 *     After a call that latched an error status, zero them again.  Calls
 *     that share a workspace must be ordered (the same stream).
 * Where the grid cannot be resident all at once (the gate needs every CTA
 * running), or M * K / 16 >= 2^31, the call quantizes A in a separate pass
 * first, with the same results.
 */
q4_status gemm_w4a4_mxfp4_fused(const void* A_raw, int a_dtype, const q4_operand* B, int64_t M,
                                int64_t N, int64_t K, void* C, int c_dtype, void* ws,
                                size_t ws_bytes, q4_stream_t stream);

/*
 * W4A16 decode GEMM ("Low-bit inference for very large MoE", "Kernels on
 * different hardware", W4A16 row: weights stay 4-bit in memory, activations
 * bf16; decode is bound by weight reads):
 *   C[m, n] = sum_g s16[n, g] * sum_{k in g} a[m, k] * q[n, k]
 * A_bf16 [M, K]; Wq [N, K/2] INT4 codes; Ws [N, K/128] FP16 bits (as written
 * by quantize_int4_g128); C_bf16 [M, N].  FP32 accumulation, one FP32
 * multiply by the scale per group of 128.  K % 128 == 0; any M >= 0 (tuned
 * for M <= 16).  Alignment: A and Wq 16 bytes, Ws and C 2 bytes.
 * ws/ws_bytes: q4_workspace_size(Q4_OP_GEMM_W4A16_INT4, ...) is 0 today (the
 * K-split partial sums meet in distributed shared memory), so ws may be NULL;
 * the pair keeps every GEMM call alike.
 * Launched with programmatic dependent launch: it starts reading Wq and Ws
 * before the previous kernel in the stream has finished (A and C wait for
 * it).  Wq and Ws must not be written by a preceding kernel that releases its
 * successor early (griddepcontrol.launch_dependents); kernels that do not do
 * this, copies, and this library's quantizers are safe.
 */
q4_status gemm_w4a16_int4(const void* A_bf16, const uint8_t* Wq, const uint16_t* Ws, int64_t M,
                          int64_t N, int64_t K, void* C_bf16, void* ws, size_t ws_bytes,
                          q4_stream_t stream);

/*
 * W4A16 with FP4 weights ("Low-bit inference for very large MoE", "Kernels on
 * different hardware": the W4A16 row lists INT4 or FP4 weights with 16-bit
 * activations): C[m, n] = sum_k a[m, k] * w[n, k] with
 *   NVFP4: w = e2m1(code) * e4m3(Ws[n, k / 16]) * g,   g = *w_tensor_scale
 *   MXFP4: w = e2m1(code) * 2^(Ws[n, k / 32] - 127)
 * A_bf16 [M, K]; Wq [N, K/2] E2M1 codes; Ws row-major scale bytes
 * (Q4_SCALES_ROWMAJOR, as quantize_nvfp4 / quantize_mxfp4 write them);
 * C_bf16 [M, N].  The block scale is folded into each weight, which is
 * exact (e2m1 x E4M3 has at most 6 significant bits; e2m1 x 2^e for scale
 * bytes up to 252, all that a quantizer of finite data writes), so every
 * product with an activation is exact; the sums are FP32, g is applied once
 * in FP32, and the only rounding to bf16 is the final store.  NVFP4 weights
 * meet the activations in f16 (weights x 2^-10, exact) for every group of
 * 128 columns whose activations are all f16 values (every bf16 value from
 * 2^-17 to 65504 in magnitude is one, as are zero and the infinities; NaN
 * stays NaN), in bf16 otherwise: the same exact products either way.
 * K % 128 == 0; any M >= 0 (tuned for M <= 16).  Alignment: A, Wq 16 bytes;
 * NVFP4 Ws 2 bytes, w_tensor_scale 4 bytes.  ws/ws_bytes as for
 * gemm_w4a16_int4 (q4_workspace_size(Q4_OP_GEMM_W4A16_NVFP4 or _MXFP4, ...)
 * is 0 today; ws may be NULL).  Launched like gemm_w4a16_int4 (programmatic
 * dependent launch; Wq and Ws are read before the previous kernel in the
 * stream has finished, under the same rule as there).
 */
q4_status gemm_w4a16_nvfp4(const void* A_bf16, const uint8_t* Wq, const uint8_t* Ws,
                           const float* w_tensor_scale, int64_t M, int64_t N, int64_t K,
                           void* C_bf16, void* ws, size_t ws_bytes, q4_stream_t stream);
q4_status gemm_w4a16_mxfp4(const void* A_bf16, const uint8_t* Wq, const uint8_t* Ws, int64_t M,
                           int64_t N, int64_t K, void* C_bf16, void* ws, size_t ws_bytes,
                           q4_stream_t stream);

/*
 * Grouped routed-MoE NVFP4 GEMM ("Low-bit inference for very large MoE",
 * "Kernels on different hardware": one low-bit weight matrix per expert,
 * grouped by routing).  The T tokens [T, K] bf16 are NVFP4-quantized once as
 * one tensor (one per-tensor scale), then for every expert e
 *   C[r, :] = A_hat[row_token[r], :] . W_hat_e^T   for r in
 *   [expert_offsets[e], expert_offsets[e+1])
 * expert_offsets: device int32 [E+1], non-decreasing, expert_offsets[0] = 0,
 * expert_offsets[E] = R.  row_token: device int32 [R], values in [0, T).
 * W: the E experts' NVFP4 weights as one operand (raw must be NULL): codes
 * [E, N, K/2]; scales in W->scale_layout, either E consecutive
 * Q4_SCALES_MMA tensors of q4_mma_scales_bytes(N, K/16) bytes each or
 * Q4_SCALES_ROWMAJOR [E, N, K/16] bytes (re-laid out into the workspace on
 * every call: pre-convert with q4_scales_to_mma for speed); tensor_scale:
 * device float [E], one per expert.
 * C_bf16: [R, N].  K % 256 == 0.  An expert with no rows is legal.
 * ws: q4_workspace_size_moe(T, N, K, E, R) bytes, plus
 * E * q4_mma_scales_bytes(N, K/16) more with row-major weight scales; it
 * holds the quantized tokens, their codes copied in routed order (R * K/2
 * bytes), the routed scales, the expert schedule (and the re-laid-out weight
 * scales).
 */
q4_status grouped_gemm_moe(const void* tokens_bf16, int64_t T, int64_t K,
                           const int32_t* expert_offsets, const int32_t* row_token, int64_t R,
                           int E, const q4_operand* W, int64_t N, void* C_bf16, void* ws,
                           size_t ws_bytes, q4_stream_t stream);

/*
 * FP8 blockwise quantization ("Quantization in deployment", "Fake
 * quantization", fp8 and fp8_blockwise): E4M3 codes, one FP32 scale per
 * block of block_rows x 128 elements, block_rows = 128 for weights
 * (128 x 128 blocks) or 1 for activations (one scale per row and 128
 * columns).  For every block, in float32 with IEEE rounding:
 *   s = max(amax_block, 1e-12) / 448;  code = e4m3_rne(clamp(x / s, -448, 448))
 * where an E4M3 byte keeps the sign of x / s, also when it rounds to zero.
 * codes: [rows, K] bytes (one per element, 16-byte aligned); scales: float
 * [rows / block_rows, K / 128] row-major.  K % 128 == 0; rows % 128 == 0
 * when block_rows == 128.  x: [rows, K] of x_dtype, 16-byte aligned.  A
 * non-finite input latches Q4_ERR_NONFINITE (see q4_sync_status()).
 */
q4_status quantize_fp8_blockwise(const void* x, int x_dtype, int64_t rows, int64_t K,
                                 int block_rows, uint8_t* codes, float* scales,
                                 q4_stream_t stream);

/*
 * Block-promoted FP8 GEMM ("Quantization in deployment", exercise 2, the cost
 * of block FP8): the tensor cores sum the FP8 products of each 128-wide K
 * block in FP32, and each block's sum is multiplied by its activation and
 * weight scales and added into the FP32 result:
 *   C[m, n] = sum_kb sa[m, kb] * sb[n / 128, kb] * sum_{k in kb} qa[m, k] * qb[n, k]
 * qa: E4M3 [M, K] with sa float [M, K / 128] (quantize_fp8_blockwise with
 * block_rows 1); qb: E4M3 [N, K] with sb float [N / 128, K / 128] (block_rows
 * 128).  C: [M, N] in c_dtype (Q4_F32, or Q4_BF16 rounded to nearest even),
 * 16-byte aligned.  K % 128 == 0, N % 128 == 0; any M.  qa and qb 16-byte
 * aligned.  ws/ws_bytes: q4_workspace_size(Q4_OP_GEMM_FP8_BLOCKWISE, ...) is 0
 * today, so ws may be NULL (the pair keeps every GEMM call alike).
 * Asynchronous; operands may come from the previous kernel in the stream
 * (programmatic dependent launch, read only after it has finished).
 */
q4_status gemm_fp8_blockwise(const uint8_t* qa, const float* sa, const uint8_t* qb,
                             const float* sb, int64_t M, int64_t N, int64_t K, void* C,
                             int c_dtype, void* ws, size_t ws_bytes, q4_stream_t stream);

/*
 * W4A8 ("Low-bit inference for very large MoE", "Kernels on different
 * hardware", the W4A8 row: INT4 weights turned into FP8, activations quantized
 * to FP8, the product on FP8 tensor cores).  Every INT4 value -8..7 is an
 * E4M3 value, so the weight codes convert exactly; the FP16 group scale (one
 * per 128 along K) joins the activation scale in the per-K-block promotion:
 *   C[m, n] = sum_kb sa[m, kb] * s16[n, kb] * sum_{k in kb} qa[m, k] * q[n, k]
 * qa, sa: FP8 activations from quantize_fp8_blockwise with block_rows 1.
 * w_codes: [N, K/2] INT4 codes as quantize_int4_g128 writes them (16-byte
 * aligned).  w_scales_kn: float [K/128, N], the weight scales converted once
 * by w4a8_weight_scales (16-byte aligned).  C: [M, N] in c_dtype (Q4_F32 or
 * Q4_BF16), 16-byte aligned.  K % 128 == 0, N % 128 == 0; any M.  ws/ws_bytes:
 * q4_workspace_size(Q4_OP_GEMM_W4A8, ...) is 0 today, so ws may be NULL.
 */
q4_status w4a8_weight_scales(const uint16_t* w_scales, int64_t N, int64_t K, float* w_scales_kn,
                             q4_stream_t stream);
q4_status gemm_w4a8(const uint8_t* qa, const float* sa, const uint8_t* w_codes,
                    const float* w_scales_kn, int64_t M, int64_t N, int64_t K, void* C,
                    int c_dtype, void* ws, size_t ws_bytes, q4_stream_t stream);

/*
 * gemm_w4a4_nvfp4 without a workspace, for callers that cannot give the
 * library any device memory beyond inputs and outputs: a plugin or custom-op
 * interface that passes only input and output buffers, or an engine whose
 * memory pool is fully reserved at start-up.  The pages have no counterpart:
 * this is a deployment convenience, not a step of the method.
 *
 * Computes exactly what gemm_w4a4_nvfp4 computes with A given raw (A [M, K]
 * in a_dtype, NVFP4-quantized on the fly with its own tensor scale) and B
 * pre-quantized with Q4_SCALES_MMA scales and a tensor scale.  The quantized
 * activations live in one file-scope device array of
 * q4_noalloc_scratch_bytes() (16 MiB) per GPU that loads the library, held
 * until the process exits; a problem needing more (q4_noalloc_required_bytes(M,
 * K): M * K / 2 code bytes plus its scales) returns Q4_ERR_SCRATCH_TOO_SMALL
 * before anything is launched.  Nothing is allocated: no cudaMalloc, no
 * cudaFree, no allocating library call.
 *
 * All calls share that array and it keeps the last call's contents, so calls
 * that overlap on the GPU (several streams or host threads) race: serialize
 * them.  The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress, once per device, with that device current).
 */
q4_status gemm_w4a4_nvfp4_noalloc(const void* A, int a_dtype, const q4_operand* B, int64_t M,
                                  int64_t N, int64_t K, void* C, int c_dtype, q4_stream_t stream);
size_t q4_noalloc_scratch_bytes(void);
size_t q4_noalloc_required_bytes(int64_t M, int64_t K);

/*
 * Synchronizes the stream, then returns (and clears) the first error a kernel
 * latched since the last call: Q4_OK, Q4_ERR_TIMEOUT or Q4_ERR_NONFINITE; or
 * Q4_ERR_CUDA if the synchronization itself failed.
 */
q4_status q4_sync_status(q4_stream_t stream);

/* Static description of a status code. */
const char* q4_status_string(q4_status s);

/* Upper bound, in milliseconds, of every bounded wait inside the kernels
 * (default 2000).  Returns the previous value.  Host-side setting, read at
 * launch. */
int q4_set_wait_timeout_ms(int ms);

/* Diagnostic: launch one warp that waits, through the kernels' own bounded
 * wait, on a barrier that nothing completes.  After the timeout set above it
 * gives up and latches Q4_ERR_TIMEOUT, which q4_sync_status() then returns;
 * the context stays usable.  Exercises the failure path of the pipelines
 * without faulting or hanging the GPU. */
q4_status q4_selftest_wait_timeout(q4_stream_t stream);

/*
 * Measurement aid (not a step of the method): read-bandwidth probe.  Streams
 * `bytes` from src once with 16-byte loads (8 CTAs of 256 threads per SM,
 * four loads in flight per thread) and XORs what it reads into sink[0 ..
 * q4_read_probe_sink_words()) so that the loads are kept.  Timed over the
 * same bytes per launch and launch pattern as an HBM-bound kernel, it gives
 * the rate a bare read of that size reaches.  src: device, 16-byte aligned;
 * bytes % 16 == 0 (0: no-op); sink: device, 4-byte aligned, written with
 * atomic XOR (contents meaningless).  Q4_ERR_INVALID_ARG otherwise.
 */
size_t q4_read_probe_sink_words(void);
q4_status q4_read_probe(const void* src, size_t bytes, unsigned* sink, q4_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* Q4GEMM_H_ */
