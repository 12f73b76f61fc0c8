// q4_format.cu — Q4_0 quantization and conversion between the canonical
// 18-byte blocks and the library's fragment device layout.
//
// Block rule (the pages say only "4-bit quantized Qwen2.5 7B" — "Why
// Continuous Batching Slowed Down My LLM Inference Engine", intro — so the
// library fixes the usual Q4_0 definition): per 32 weights along K,
// m = first element of largest |w|, d = m / -8, q = clamp(round(w/d)+8, 0, 15)
// with IEEE division and round-half-away-from-zero, d stored as binary16
// (round to nearest even).  All-zero blocks get d = 0, q = 8.
//
// Quantization writes canonical blocks; the repack kernel (shared with
// import) turns canonical blocks into the fragment layout described in
// q4mm_internal.h; export gathers them back.
#include <cuda_fp16.h>

#include "q4mm_internal.h"

namespace q4 {
namespace {

constexpr unsigned FLAG_NONFINITE = 1u;
constexpr unsigned FLAG_RANGE = 2u;

// One thread per (row, block): fp32 weights -> canonical 18-byte block.
__global__ void __launch_bounds__(TILE_N) quantize_kernel(const float* __restrict__ w, int64_t N,
                                                          int64_t K, int64_t KB,
                                                          uint8_t* __restrict__ canon,
                                                          unsigned int* flag) {
  const int64_t n = (int64_t)blockIdx.x * TILE_N + threadIdx.x;
  const int64_t b = blockIdx.y;
  if (n >= N) return;
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
  const uint16_t d16 = __half_as_ushort(__float2half_rn(d));
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
  uint8_t* blk = canon + (n * KB + b) * CANON_BLOCK_BYTES;
  blk[0] = (uint8_t)(d16 & 0xFFu);
  blk[1] = (uint8_t)(d16 >> 8);
#pragma unroll
  for (int j = 0; j < 16; ++j) blk[2 + j] = (uint8_t)(q[j] | (q[j + 16] << 4));
}

// Canonical bytes j = 2tq, 2tq+1, 2tq+8, 2tq+9 of a block hold, in their low
// nibbles, q at k0 = 2tq (+1, +8, +9) of k-step 0 and, in their high nibbles,
// the same offsets of k-step 1 (k + 16).  Missing rows and pad blocks read
// as q = 8 with d = 0.
struct LaneBlock {
  uint8_t byte[4];  // canonical bytes 2tq, 2tq+1, 2tq+8, 2tq+9
  uint16_t d16;
};

__device__ __forceinline__ LaneBlock load_lane_block(const uint8_t* canon, int64_t N, int64_t KB,
                                                     int64_t n, int64_t b, int tq) {
  LaneBlock r;
  if (n >= N || b >= KB) {
    r.byte[0] = r.byte[1] = r.byte[2] = r.byte[3] = 0x88u;
    r.d16 = 0;
    return r;
  }
  const uint8_t* blk = canon + (n * KB + b) * CANON_BLOCK_BYTES;
  r.d16 = (uint16_t)(blk[0] | (blk[1] << 8));
  r.byte[0] = blk[2 + 2 * tq];
  r.byte[1] = blk[2 + 2 * tq + 1];
  r.byte[2] = blk[2 + 2 * tq + 8];
  r.byte[3] = blk[2 + 2 * tq + 9];
  return r;
}

// Word for k-step s from the lane's blocks of rows R0 (lo) and R1 (hi):
// pair p holds row (p & 1 ? R1 : R0) at offsets (p >> 1) * 8 + {0, 1}.
__device__ __forceinline__ uint32_t make_word(const LaneBlock& r0, const LaneBlock& r1, int s) {
  uint32_t w = 0;
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const LaneBlock& r = (p & 1) ? r1 : r0;
    const int j = (p >> 1) * 2;  // byte index for offsets 0/1 (p < 2) or 8/9 (p >= 2)
    const uint32_t lo = s == 0 ? (r.byte[j] & 0xFu) : (r.byte[j] >> 4);
    const uint32_t hi = s == 0 ? (r.byte[j + 1] & 0xFu) : (r.byte[j + 1] >> 4);
    w |= lo << (4 * p);
    w |= hi << (16 + 4 * p);
  }
  return w;
}

// Canonical blocks [N][KB][18] (device) -> fragment layout.  One thread per
// (tile, block pair, row group, lane); blockDim = 256 (8 row groups x 32).
__global__ void __launch_bounds__(256) repack_kernel(const uint8_t* __restrict__ canon, int64_t N,
                                                     int64_t KB, int64_t KBP,
                                                     uint32_t* __restrict__ nib,
                                                     uint16_t* __restrict__ dsc,
                                                     unsigned int* flag) {
  const int64_t t = blockIdx.x, bp = blockIdx.y;
  const int rg = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, tq = lane & 3;
  const int64_t n0 = t * TILE_N + rg * 16 + g, n1 = n0 + 8;
  LaneBlock r[2][2];  // [upper][h]
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    r[0][h] = load_lane_block(canon, N, KB, n0, 2 * bp + h, tq);
    r[1][h] = load_lane_block(canon, N, KB, n1, 2 * bp + h, tq);
  }
  uint4 out;
  out.x = make_word(r[0][0], r[1][0], 0);
  out.y = make_word(r[0][0], r[1][0], 1);
  out.z = make_word(r[0][1], r[1][1], 0);
  out.w = make_word(r[0][1], r[1][1], 1);
  reinterpret_cast<uint4*>(nib)[nib_word_index(KBP, t, bp, rg, lane, 0, 0) / 4] = out;
  if (tq == 0) {  // flag == null: the caller validated the scales already
    bool bad = false;
#pragma unroll
    for (int u = 0; u < 2; ++u)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        dsc[scale_index(KBP, t, bp, rg, g, u, h)] = r[u][h].d16;
        bad = bad || ((r[u][h].d16 & 0x7C00u) == 0x7C00u);
      }
    if (bad && flag != nullptr) atomicOr(flag, FLAG_NONFINITE);
  }
}

// Fragment layout -> canonical blocks [N][KB][18]; one thread per (row, block).
__global__ void __launch_bounds__(TILE_N) export_kernel(const uint32_t* __restrict__ nib,
                                                        const uint16_t* __restrict__ dsc,
                                                        int64_t N, int64_t KB, int64_t KBP,
                                                        uint8_t* __restrict__ canon) {
  const int64_t n = (int64_t)blockIdx.x * TILE_N + threadIdx.x;
  const int64_t b = blockIdx.y;
  if (n >= N) return;
  const int64_t t = n / TILE_N;
  const int r = (int)(n % TILE_N);
  const int rg = r >> 4, upper = (r >> 3) & 1, g = r & 7;
  const int64_t bp = b >> 1;
  const int h = (int)(b & 1);
  uint8_t q[32];
#pragma unroll
  for (int tq = 0; tq < 4; ++tq)
#pragma unroll
    for (int s = 0; s < 2; ++s) {
      const uint32_t w = nib[nib_word_index(KBP, t, bp, rg, 4 * g + tq, h, s)];
#pragma unroll
      for (int half = 0; half < 2; ++half) {  // pair upper (k0) and upper + 2 (k0 + 8)
        const int p = upper + 2 * half;
        const int k = 16 * s + 2 * tq + 8 * half;
        q[k] = (w >> (4 * p)) & 0xFu;
        q[k + 1] = (w >> (16 + 4 * p)) & 0xFu;
      }
    }
  const uint16_t d16 = dsc[scale_index(KBP, t, bp, rg, g, upper, h)];
  uint8_t* blk = canon + (n * KB + b) * CANON_BLOCK_BYTES;
  blk[0] = (uint8_t)(d16 & 0xFFu);
  blk[1] = (uint8_t)(d16 >> 8);
#pragma unroll
  for (int j = 0; j < 16; ++j) blk[2 + j] = (uint8_t)(q[j] | (q[j + 16] << 4));
}

}  // namespace

int quantize_flag_status(unsigned f) {
  if (f & FLAG_NONFINITE) return Q4_ERR_NONFINITE;
  if (f & FLAG_RANGE) return Q4_ERR_RANGE;
  return Q4_OK;
}

int launch_quantize(const float* w, int64_t N, int64_t K, uint8_t* canon_dev, Weight* W,
                    unsigned int* flag, cudaStream_t s) {
  dim3 grid((unsigned)((N + TILE_N - 1) / TILE_N), (unsigned)W->KB);
  quantize_kernel<<<grid, TILE_N, 0, s>>>(w, N, K, W->KB, canon_dev, flag);
  if (cudaGetLastError() != cudaSuccess) return Q4_ERR_CUDA;
  return launch_import(canon_dev, W, nullptr, s);  // the quantizer reported range errors
}

int launch_import(const uint8_t* canon_dev, Weight* W, unsigned int* flag, cudaStream_t s) {
  dim3 grid((unsigned)W->tiles, (unsigned)W->KBP);
  repack_kernel<<<grid, 256, 0, s>>>(canon_dev, W->N, W->KB, W->KBP,
                                     reinterpret_cast<uint32_t*>(W->nib), W->d, flag);
  return cudaGetLastError() == cudaSuccess ? Q4_OK : Q4_ERR_CUDA;
}

int launch_export(const Weight* W, uint8_t* canon_dev, cudaStream_t s) {
  dim3 grid((unsigned)((W->N + TILE_N - 1) / TILE_N), (unsigned)W->KB);
  export_kernel<<<grid, TILE_N, 0, s>>>(reinterpret_cast<const uint32_t*>(W->nib), W->d, W->N,
                                        W->KB, W->KBP, canon_dev);
  return cudaGetLastError() == cudaSuccess ? Q4_OK : Q4_ERR_CUDA;
}

}  // namespace q4
