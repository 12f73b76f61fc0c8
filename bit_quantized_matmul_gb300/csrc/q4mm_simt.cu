// q4mm_simt.cu — CUDA-core streaming kernel for the Q4_0 matmul.
//
// The small-M path: each packed weight block is read from HBM exactly once
// per call, unpacked in registers and used for every activation row of the
// call, so a second or third token row costs FMAs but no extra weight bytes
// ("Why LLM Decoding Is Slow, and Why Batching Is (Almost) Free", §4 "Share
// the Weights Across Users").  It plays the role the one-row Metal GEMV plays
// in "Why Continuous Batching Slowed Down My LLM Inference Engine"
// (§"Two Rows of Input, Two Different Kernels": dequantize on the fly while
// streaming, linear and predictable access), but takes any number of rows in
// one launch instead of one launch per row.
//
// Shape of the work: one thread per weight row n of a 128-row tile, looping
// along its K range one 32-weight block at a time; a warp reads 512
// consecutive bytes per block (tiled layout).  Activations are staged in
// shared memory in chunks of KC blocks and read as broadcasts.  The K range
// may be split across CTAs (split count chosen from N and K only); partial
// sums are added in ascending split order by the last CTA to arrive, so the
// result does not depend on scheduling.
//
// Per-row arithmetic: s = sum over the block of (q-8) * x in ascending k
// (fp32 FMA, exact (q-8)), then acc = fma(d, s, acc) over the blocks of the
// split in ascending order.  No step depends on M or on other rows, so rows
// are bit-identical whatever they are batched with.
#include <cuda_fp16.h>

#include "q4mm_internal.h"

namespace q4 {
namespace {

constexpr int KC = 32;  // blocks of x staged per chunk (1024 values per row)

struct SimtArgs {
  const uint4* nib;
  const uint16_t* d;
  int64_t KB, K, N, N_pad;
  const float* x;  // rows [m_base, m_base + M) of the caller's x
  int64_t M;       // rows in this launch
  float* y;
  int32_t* idx;
  float* maxval;
  int splits;
  int64_t kb_per_split;
  int mchunks;
  int tiles;
  float* partial;
  unsigned int* counters;
  unsigned long long* keys;
  unsigned int* argmax_done;
};

// Exact (q - 8) as fp32 for the nibble at bit `shift`: 2^23 + q has q in the
// low mantissa bits; subtracting 2^23 + 8 is exact.
__device__ __forceinline__ float qm8(uint32_t w, int shift) {
  return __uint_as_float(0x4B000000u | ((w >> shift) & 0xFu)) - 8388616.0f;
}

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}

// Argmax key: order-preserving map of the value in the high word (NaN lowest,
// -0 folded into +0), complemented index in the low word so that equal values
// prefer the lower index under an unsigned max.
__device__ __forceinline__ unsigned long long argmax_key(float v, uint32_t n) {
  if (v != v) return 0ull;
  if (v == 0.0f) v = 0.0f;
  uint32_t u = __float_as_uint(v);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((unsigned long long)u << 32) | (unsigned long long)(0xFFFFFFFFu - n);
}

__device__ __forceinline__ float key_value(unsigned long long k) {
  const uint32_t u = (uint32_t)(k >> 32);
  if (u == 0u) return __uint_as_float(0x7FC00000u);
  return __uint_as_float((u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u);
}

__device__ __forceinline__ unsigned long long shfl_max_u64(unsigned long long k) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const unsigned long long o = __shfl_xor_sync(0xFFFFFFFFu, k, off);
    k = o > k ? o : k;
  }
  return k;
}

template <int MT>
__global__ void __launch_bounds__(TILE_N) simt_kernel(const SimtArgs a) {
  __shared__ __align__(16) float xs[MT][KC * BLOCK_K];
  __shared__ unsigned long long red[TILE_N / 32][MT];
  __shared__ int s_last;

  const int r = threadIdx.x;
  const int tile = blockIdx.x, split = blockIdx.y, mc = blockIdx.z;
  const int64_t n = (int64_t)tile * TILE_N + r;
  const int64_t m0 = (int64_t)mc * MT;
  const int mcount = (int)min((int64_t)MT, a.M - m0);
  const int64_t kb0 = (int64_t)split * a.kb_per_split;
  const int64_t kb1 = min(a.KB, kb0 + a.kb_per_split);
  const uint4* nibp = a.nib + (int64_t)tile * a.KB * TILE_N + r;
  const uint16_t* dp = a.d + (int64_t)tile * a.KB * TILE_N + r;

  float acc[MT];
#pragma unroll
  for (int m = 0; m < MT; ++m) acc[m] = 0.0f;

  for (int64_t c0 = kb0; c0 < kb1; c0 += KC) {
    const int nbk = (int)min((int64_t)KC, kb1 - c0);
    __syncthreads();
    const int f4_per_row = nbk * (BLOCK_K / 4);
    for (int i = r; i < MT * f4_per_row; i += TILE_N) {
      const int m = i / f4_per_row, j = i - m * f4_per_row;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (m < mcount)
        v = __ldg(reinterpret_cast<const float4*>(a.x + (m0 + m) * a.K + c0 * BLOCK_K) + j);
      reinterpret_cast<float4*>(xs[m])[j] = v;
    }
    __syncthreads();
#pragma unroll 4
    for (int bb = 0; bb < nbk; ++bb) {
      const uint4 v = ld_stream(nibp + (c0 + bb) * TILE_N);
      const float d = __half2float(__ushort_as_half(__ldg(dp + (c0 + bb) * TILE_N)));
      const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
      float s[MT];
#pragma unroll
      for (int m = 0; m < MT; ++m) s[m] = 0.0f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float q[8];
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          q[2 * p] = qm8(wv[i], 4 * p);            // k = 8i + 2p
          q[2 * p + 1] = qm8(wv[i], 16 + 4 * p);   // k = 8i + 2p + 1
        }
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          const float4 xa = *reinterpret_cast<const float4*>(&xs[m][bb * BLOCK_K + 8 * i]);
          const float4 xb = *reinterpret_cast<const float4*>(&xs[m][bb * BLOCK_K + 8 * i + 4]);
          float t = s[m];
          t = fmaf(q[0], xa.x, t);
          t = fmaf(q[1], xa.y, t);
          t = fmaf(q[2], xa.z, t);
          t = fmaf(q[3], xa.w, t);
          t = fmaf(q[4], xb.x, t);
          t = fmaf(q[5], xb.y, t);
          t = fmaf(q[6], xb.z, t);
          t = fmaf(q[7], xb.w, t);
          s[m] = t;
        }
      }
#pragma unroll
      for (int m = 0; m < MT; ++m) acc[m] = fmaf(d, s[m], acc[m]);
    }
  }

  // ---- split-K: the last CTA of this (tile, m-chunk) adds the partials ----
  if (a.splits > 1) {
#pragma unroll
    for (int m = 0; m < MT; ++m)
      if (m < mcount) a.partial[((int64_t)split * a.M + m0 + m) * a.N_pad + n] = acc[m];
    __threadfence();
    __syncthreads();
    if (r == 0) {
      const unsigned prev = atomicAdd(&a.counters[tile * a.mchunks + mc], 1u);
      s_last = (prev == (unsigned)(a.splits - 1));
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      if (m < mcount) {
        float v = 0.0f;
        for (int s = 0; s < a.splits; ++s)
          v += __ldcg(&a.partial[((int64_t)s * a.M + m0 + m) * a.N_pad + n]);
        acc[m] = v;
      }
    }
    if (r == 0) a.counters[tile * a.mchunks + mc] = 0u;  // ready for the next launch
  }

  if (a.idx == nullptr) {
    if (n < a.N) {
#pragma unroll
      for (int m = 0; m < MT; ++m)
        if (m < mcount) a.y[(m0 + m) * a.N + n] = acc[m];
    }
    return;
  }

  // ---- fused greedy pick: per-row max over this tile, then a global max ----
  const int warp = r >> 5, lane = r & 31;
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    unsigned long long k = (m < mcount && n < a.N) ? argmax_key(acc[m], (uint32_t)n) : 0ull;
    k = shfl_max_u64(k);
    if (lane == 0) red[warp][m] = k;
  }
  __syncthreads();
  if (r < mcount) {
    unsigned long long k = red[0][r];
#pragma unroll
    for (int w = 1; w < TILE_N / 32; ++w) k = red[w][r] > k ? red[w][r] : k;
    atomicMax(&a.keys[m0 + r], k);
  }
  __threadfence();
  __syncthreads();
  if (r == 0) {
    const unsigned prev = atomicAdd(a.argmax_done, 1u);
    s_last = (prev == (unsigned)(a.tiles * a.mchunks - 1));
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int64_t m = r; m < a.M; m += TILE_N) {
    const unsigned long long k = atomicExch(&a.keys[m], 0ull);
    a.idx[m] = k == 0ull ? 0 : (int32_t)(0xFFFFFFFFu - (uint32_t)(k & 0xFFFFFFFFull));
    if (a.maxval) a.maxval[m] = key_value(k);
  }
  if (r == 0) *a.argmax_done = 0u;
}

}  // namespace

SimtPlan simt_plan(const Weight* W, int num_sms) {
  SimtPlan p;
  const int64_t want = (8 * (int64_t)num_sms + W->tiles - 1) / W->tiles;
  int64_t cap = W->KB / 8;
  if (cap < 1) cap = 1;
  if (cap > 64) cap = 64;
  int64_t s = want < 1 ? 1 : (want > cap ? cap : want);
  p.kb_per_split = (W->KB + s - 1) / s;
  p.splits = (int)((W->KB + p.kb_per_split - 1) / p.kb_per_split);
  return p;
}

constexpr int64_t SIMT_M_LAUNCH = 64;  // rows per launch

size_t simt_partial_bytes(const Weight* W, const SimtPlan& p, int64_t M) {
  if (p.splits <= 1) return 0;
  const int64_t ml = M < SIMT_M_LAUNCH ? M : SIMT_M_LAUNCH;
  return (size_t)p.splits * (size_t)ml * (size_t)W->N_pad * sizeof(float);
}

int simt_launch_count(int64_t M) { return (int)((M + SIMT_M_LAUNCH - 1) / SIMT_M_LAUNCH); }

int launch_simt(const Weight* W, const float* x, int64_t M, float* y, int32_t* idx,
                float* maxval, const SimtPlan& plan, const Workspace& ws, cudaStream_t s) {
  for (int64_t mb = 0; mb < M; mb += SIMT_M_LAUNCH) {
    const int64_t ml = (M - mb) < SIMT_M_LAUNCH ? (M - mb) : SIMT_M_LAUNCH;
    const int mt = ml >= 8 ? 8 : (ml >= 4 ? 4 : (ml >= 2 ? 2 : 1));
    const int64_t mchunks = (ml + mt - 1) / mt;
    SimtArgs a;
    a.nib = reinterpret_cast<const uint4*>(W->nib);
    a.d = W->d;
    a.KB = W->KB;
    a.K = W->K;
    a.N = W->N;
    a.N_pad = W->N_pad;
    a.x = x + mb * W->K;
    a.M = ml;
    a.y = y ? y + mb * W->N : nullptr;
    a.idx = idx ? idx + mb : nullptr;
    a.maxval = (idx && maxval) ? maxval + mb : nullptr;
    a.splits = plan.splits;
    a.kb_per_split = plan.kb_per_split;
    a.mchunks = (int)mchunks;
    a.tiles = (int)W->tiles;
    a.partial = ws.partial;
    a.counters = ws.counters;
    a.keys = ws.keys + mb;
    a.argmax_done = ws.argmax_done;
    if (plan.splits > 1 && W->tiles * mchunks > MAX_COUNTERS) return Q4_ERR_SHAPE;
    dim3 grid((unsigned)W->tiles, (unsigned)plan.splits, (unsigned)mchunks);
    switch (mt) {
      case 1: simt_kernel<1><<<grid, TILE_N, 0, s>>>(a); break;
      case 2: simt_kernel<2><<<grid, TILE_N, 0, s>>>(a); break;
      case 4: simt_kernel<4><<<grid, TILE_N, 0, s>>>(a); break;
      default: simt_kernel<8><<<grid, TILE_N, 0, s>>>(a); break;
    }
    if (cudaGetLastError() != cudaSuccess) return Q4_ERR_CUDA;
  }
  return Q4_OK;
}

}  // namespace q4
