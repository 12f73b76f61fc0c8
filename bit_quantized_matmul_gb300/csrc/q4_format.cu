// q4_format.cu — Q4_0 quantization and conversion between the canonical
// 18-byte blocks and the library's tiled device layout.
//
// Block rule (the pages say only "4-bit quantized Qwen2.5 7B" — "Why
// Continuous Batching Slowed Down My LLM Inference Engine", intro — so the
// library fixes the usual Q4_0 definition): per 32 weights along K,
// m = first element of largest |w|, d = m / -8, q = clamp(round(w/d)+8, 0, 15)
// with IEEE division and round-half-away-from-zero, d stored as binary16
// (round to nearest even).  All-zero blocks get d = 0, q = 8.
#include <cuda_fp16.h>

#include "q4mm_internal.h"

namespace q4 {
namespace {

constexpr unsigned FLAG_NONFINITE = 1u;
constexpr unsigned FLAG_RANGE = 2u;

// Device nibble order (see q4mm_internal.h): word i, nibble at bit 4p holds
// k = 8i+2p, nibble at bit 16+4p holds k = 8i+2p+1.
__device__ __forceinline__ uint4 pack_device_order(const uint8_t (&q)[32]) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t v = 0;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      v |= (uint32_t)q[8 * i + 2 * p] << (4 * p);
      v |= (uint32_t)q[8 * i + 2 * p + 1] << (16 + 4 * p);
    }
    w[i] = v;
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ void unpack_device_order(uint4 v, uint8_t (&q)[32]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      q[8 * i + 2 * p] = (w[i] >> (4 * p)) & 0xFu;
      q[8 * i + 2 * p + 1] = (w[i] >> (16 + 4 * p)) & 0xFu;
    }
}

// One thread per (row, block); blockDim = 128 rows of one tile.
__global__ void __launch_bounds__(TILE_N) quantize_kernel(const float* __restrict__ w, int64_t N,
                                                          int64_t K, int64_t KB,
                                                          uint8_t* __restrict__ nib,
                                                          uint16_t* __restrict__ dsc,
                                                          unsigned int* flag) {
  const int r = threadIdx.x;
  const int64_t t = blockIdx.x, b = blockIdx.y;
  const int64_t n = t * TILE_N + r;
  const int64_t o = (t * KB + b) * TILE_N + r;
  uint4 out = make_uint4(0x88888888u, 0x88888888u, 0x88888888u, 0x88888888u);
  uint16_t d16 = 0;
  if (n < N) {
    const float4* src = reinterpret_cast<const float4*>(w + n * K + b * BLOCK_K);
    float v[32];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 f = src[i];
      v[4 * i] = f.x;
      v[4 * i + 1] = f.y;
      v[4 * i + 2] = f.z;
      v[4 * i + 3] = f.w;
    }
    bool finite = true;
#pragma unroll
    for (int i = 0; i < 32; ++i) finite = finite && isfinite(v[i]);
    float amax = fabsf(v[0]);
    int im = 0;
#pragma unroll
    for (int i = 1; i < 32; ++i) {
      if (fabsf(v[i]) > amax) {  // strict: the first of equal magnitudes wins
        amax = fabsf(v[i]);
        im = i;
      }
    }
    float m = v[0];
#pragma unroll
    for (int i = 1; i < 32; ++i)
      if (i == im) m = v[i];
    const float d = __fdiv_rn(m, -8.0f);
    d16 = __half_as_ushort(__float2half_rn(d));
    if (!finite) {
      atomicOr(flag, FLAG_NONFINITE);
    } else if ((d16 & 0x7C00u) == 0x7C00u) {
      atomicOr(flag, FLAG_RANGE);
    }
    uint8_t q[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      int qi = 8;
      if (d != 0.0f) {
        qi = (int)roundf(__fdiv_rn(v[i], d)) + 8;  // roundf: half away from zero
        qi = qi < 0 ? 0 : (qi > 15 ? 15 : qi);
      }
      q[i] = (uint8_t)qi;
    }
    out = pack_device_order(q);
  }
  reinterpret_cast<uint4*>(nib)[o] = out;
  dsc[o] = d16;
}

// Canonical blocks [N][KB][18] (device staging copy) -> device layout.
__global__ void __launch_bounds__(TILE_N) import_kernel(const uint8_t* __restrict__ canon,
                                                        int64_t N, int64_t KB,
                                                        uint8_t* __restrict__ nib,
                                                        uint16_t* __restrict__ dsc,
                                                        unsigned int* flag) {
  const int r = threadIdx.x;
  const int64_t t = blockIdx.x, b = blockIdx.y;
  const int64_t n = t * TILE_N + r;
  const int64_t o = (t * KB + b) * TILE_N + r;
  uint4 out = make_uint4(0x88888888u, 0x88888888u, 0x88888888u, 0x88888888u);
  uint16_t d16 = 0;
  if (n < N) {
    const uint8_t* blk = canon + (n * KB + b) * CANON_BLOCK_BYTES;
    d16 = (uint16_t)(blk[0] | (blk[1] << 8));
    if ((d16 & 0x7C00u) == 0x7C00u) atomicOr(flag, FLAG_NONFINITE);
    uint8_t q[32];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const uint8_t byte = blk[2 + j];
      q[j] = byte & 0xFu;
      q[j + 16] = byte >> 4;
    }
    out = pack_device_order(q);
  }
  reinterpret_cast<uint4*>(nib)[o] = out;
  dsc[o] = d16;
}

// Device layout -> canonical blocks [N][KB][18].
__global__ void __launch_bounds__(TILE_N) export_kernel(const uint8_t* __restrict__ nib,
                                                        const uint16_t* __restrict__ dsc,
                                                        int64_t N, int64_t KB,
                                                        uint8_t* __restrict__ canon) {
  const int r = threadIdx.x;
  const int64_t t = blockIdx.x, b = blockIdx.y;
  const int64_t n = t * TILE_N + r;
  if (n >= N) return;
  const int64_t o = (t * KB + b) * TILE_N + r;
  uint8_t q[32];
  unpack_device_order(reinterpret_cast<const uint4*>(nib)[o], q);
  const uint16_t d16 = dsc[o];
  uint8_t* blk = canon + (n * KB + b) * CANON_BLOCK_BYTES;
  blk[0] = (uint8_t)(d16 & 0xFFu);
  blk[1] = (uint8_t)(d16 >> 8);
#pragma unroll
  for (int j = 0; j < 16; ++j) blk[2 + j] = (uint8_t)(q[j] | (q[j + 16] << 4));
}

int flag_to_status(unsigned f) {
  if (f & FLAG_NONFINITE) return Q4_ERR_NONFINITE;
  if (f & FLAG_RANGE) return Q4_ERR_RANGE;
  return Q4_OK;
}

}  // namespace

int launch_quantize(const float* w, int64_t N, int64_t K, Weight* W, unsigned int* flag,
                    cudaStream_t s) {
  dim3 grid((unsigned)W->tiles, (unsigned)W->KB);
  quantize_kernel<<<grid, TILE_N, 0, s>>>(w, N, K, W->KB, W->nib, W->d, flag);
  return cudaGetLastError() == cudaSuccess ? Q4_OK : Q4_ERR_CUDA;
}

int launch_import(const uint8_t* canon_dev, Weight* W, unsigned int* flag, cudaStream_t s) {
  dim3 grid((unsigned)W->tiles, (unsigned)W->KB);
  import_kernel<<<grid, TILE_N, 0, s>>>(canon_dev, W->N, W->KB, W->nib, W->d, flag);
  return cudaGetLastError() == cudaSuccess ? Q4_OK : Q4_ERR_CUDA;
}

int launch_export(const Weight* W, uint8_t* canon_dev, cudaStream_t s) {
  dim3 grid((unsigned)W->tiles, (unsigned)W->KB);
  export_kernel<<<grid, TILE_N, 0, s>>>(W->nib, W->d, W->N, W->KB, canon_dev);
  return cudaGetLastError() == cudaSuccess ? Q4_OK : Q4_ERR_CUDA;
}

int quantize_flag_status(unsigned f) { return flag_to_status(f); }

}  // namespace q4
