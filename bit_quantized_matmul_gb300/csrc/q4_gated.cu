// q4_gated.cu — the elementwise step of a gated MLP, h = SiLU(g) * u, for the
// calls whose gate and up outputs are not fused into the matmul (tensor-core
// path, batch-invariant mode): one pass over g and u written by a grouped
// call.  The streaming path computes the same expression in the matmul's
// epilogue (q4mm_mma.cu) and writes only h.
#include <cuda_runtime.h>

#include "q4mm_internal.h"

namespace q4 {
namespace {

__global__ void __launch_bounds__(256) silu_mul_kernel(const float* __restrict__ g, const float* __restrict__ u,
                                                       float* __restrict__ h, int64_t n) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const float gv = g[i];
    h[i] = gv / (1.0f + expf(-gv)) * u[i];
  }
}

}  // namespace

int launch_silu_mul(const float* g, const float* u, float* h, int64_t n, cudaStream_t s) {
  if (n <= 0) return Q4_OK;
  const int64_t blocks64 = (n + 255) / 256;
  const unsigned blocks = (unsigned)(blocks64 < 4096 ? blocks64 : 4096);
  silu_mul_kernel<<<blocks, 256, 0, s>>>(g, u, h, n);
  return cudaGetLastError() == cudaSuccess ? Q4_OK : Q4_ERR_CUDA;
}

}  // namespace q4
