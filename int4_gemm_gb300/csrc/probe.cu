// Read-bandwidth probe: a measurement aid beside the method's kernels, not a
// step of the method.  It streams a buffer once with 16-byte loads (8 CTAs of
// 256 threads per SM, grid-stride, four loads in flight per thread, evict-
// first) and folds what it reads with XOR into one word per CTA, so the loads
// cannot be dropped.  Timed over the same bytes per launch and in the same
// back-to-back launch pattern as an HBM-bound kernel of the library, it gives
// the rate a bare read of that size reaches: below the long-copy peak, since
// one launch of a few tens of MB spends part of its time filling and
// draining the memory pipeline.
#include "common.cuh"
#include "internal.h"

namespace q4 {
namespace {

constexpr int kProbeThreads = 256;
constexpr int kProbeCtasPerSm = 8;

__global__ void __launch_bounds__(kProbeThreads)
    read_probe_kernel(const uint4* __restrict__ p, size_t n16, unsigned* __restrict__ sink) {
  const size_t stride = (size_t)gridDim.x * kProbeThreads;
  unsigned acc = 0u;
  for (size_t i = (size_t)blockIdx.x * kProbeThreads + threadIdx.x; i < n16; i += 4 * stride) {
    uint4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const size_t j = i + u * stride;
      v[u] = j < n16 ? __ldcs(p + j) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) acc ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
  }
  acc = __reduce_xor_sync(0xffffffffu, acc);
  if ((threadIdx.x & 31) == 0) atomicXor(sink + blockIdx.x, acc);
}

}  // namespace

size_t read_probe_sink_words() { return (size_t)kProbeCtasPerSm * num_sms(); }

}  // namespace q4

size_t q4_read_probe_sink_words(void) { return q4::read_probe_sink_words(); }

q4_status q4_read_probe(const void* src, size_t bytes, unsigned* sink, q4_stream_t stream) {
  if (bytes == 0) return Q4_OK;
  if (!src || !sink || (reinterpret_cast<uintptr_t>(src) & 15) || (bytes & 15) ||
      (reinterpret_cast<uintptr_t>(sink) & 3))
    return Q4_ERR_INVALID_ARG;
  const int grid = (int)q4::read_probe_sink_words();
  q4::read_probe_kernel<<<grid, q4::kProbeThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(src), bytes / 16, sink);
  return cudaGetLastError() == cudaSuccess ? Q4_OK : Q4_ERR_CUDA;
}
