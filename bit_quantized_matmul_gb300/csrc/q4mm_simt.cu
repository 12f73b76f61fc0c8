// q4mm_simt.cu — CUDA-core streaming kernel for the Q4_0 matmul.
//
// The plain small-M path without tensor cores: each packed weight block is
// read from HBM exactly once per call, unpacked in registers and used for
// every token row of the call ("Why LLM Decoding Is Slow, and Why Batching Is
// (Almost) Free", §4 "Share the Weights Across Users").  It is the CUDA-core
// counterpart of the one-row Metal GEMV of "Why Continuous Batching Slowed
// Down My LLM Inference Engine" (§"Two Rows of Input, Two Different Kernels":
// dequantize on the fly during linear, predictable reads), taking any number
// of rows in one launch.
//
// Per warp: one 16-row group of a 128-row tile over the CTA's K range; lane
// (g, tq) owns rows 16rg + g and + 8 at the k offsets 16s + 2tq + {0,1,8,9}
// of each block (the fragment layout), so the four lanes of a row split K and
// their sums meet in a fixed-order warp-shuffle reduction (xor 1, then xor 2)
// shared by all token rows.  Per block and row: s = sum (q-8) x over the
// lane's 8 weights in a fixed order (exact (q-8), fp32 FMA), then
// acc = fma(d, s, acc) in ascending block order.  Nothing depends on M or on
// the other rows, so rows are bit-identical whatever they are batched with.
#include <cuda_fp16.h>

#include "q4mm_epilogue.cuh"
#include "q4mm_internal.h"

namespace q4 {
namespace {

constexpr int SIMT_THREADS = 256;  // 8 warps = the 8 row groups of a tile

struct SimtArgs {
  const uint4* nib;
  const uint2* scl;
  const float* x;  // rows [0, mrows) of this launch
  int64_t K, KBP;
  int mrows;
  int64_t kbp_per_split;
  EpiArgs e;
};

__device__ __forceinline__ uint4 ld_stream16(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint2 ld_stream8(const uint2* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];"
               : "=r"(v.x), "=r"(v.y)
               : "l"(p));
  return v;
}

// Exact (q - 8) as fp32 for the nibble at bit `shift`: 2^23 + q has q in the
// low mantissa bits; subtracting 2^23 + 8 is exact.
__device__ __forceinline__ float qm8(uint32_t w, int shift) {
  return __uint_as_float(0x4B000000u | ((w >> shift) & 0xFu)) - 8388616.0f;
}

template <int MT>
__global__ void __launch_bounds__(SIMT_THREADS) simt_kernel(const SimtArgs a) {
  __shared__ float red[MT][TILE_N];
  __shared__ unsigned long long kred[4][MT];
  __shared__ int s_flag;
  __shared__ unsigned s_arrival;  // split-K arrival word of this CTA

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, tq = lane & 3;
  const int64_t tile = blockIdx.x;
  const int split = blockIdx.y;
  const int rg = warp;
  const int64_t bp0 = (int64_t)split * a.kbp_per_split;
  const int64_t bp1 = min(a.KBP, bp0 + a.kbp_per_split);
  const uint4* nibp = a.nib + ((tile * a.KBP) * 8 + rg) * 32 + lane;
  const uint2* sclp = a.scl + ((tile * a.KBP) * 8 + rg) * 8 + g;
  const int64_t kmax = a.K;
  // arrival number for the split-K epilogue (stream order: the previous
  // launch has reset the word); the barrier before the epilogue publishes it
  if (threadIdx.x == 0 && a.e.splits > 1) s_arrival = split_arrive(&a.e.counters[tile]);

  float acc0[MT], acc1[MT];  // rows R0 = 16rg + g and R1 = R0 + 8
#pragma unroll
  for (int m = 0; m < MT; ++m) acc0[m] = acc1[m] = 0.0f;

  for (int64_t bp = bp0; bp < bp1; ++bp) {
    const uint4 wv = ld_stream16(nibp + bp * 256);
    const uint2 sv = ld_stream8(sclp + bp * 64);
    const __half2 s01 = *reinterpret_cast<const __half2*>(&sv.x);
    const __half2 s23 = *reinterpret_cast<const __half2*>(&sv.y);
    const float dr0[2] = {__low2float(s01), __high2float(s01)};
    const float dr1[2] = {__low2float(s23), __high2float(s23)};
    const uint32_t w4[4] = {wv.x, wv.y, wv.z, wv.w};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int64_t kb = (2 * bp + h) * BLOCK_K;
      if (kb >= kmax) break;  // pad block of an odd block count
      float s0[MT], s1[MT];
#pragma unroll
      for (int m = 0; m < MT; ++m) s0[m] = s1[m] = 0.0f;
#pragma unroll
      for (int s = 0; s < 2; ++s) {
        const uint32_t w = w4[2 * h + s];
        // pair p: row (p & 1 ? R1 : R0), k offset 8 * (p >> 1); lo nibble k, hi k + 1
        const float r0a = qm8(w, 0), r0b = qm8(w, 16);   // R0, k0, k0 + 1
        const float r1a = qm8(w, 4), r1b = qm8(w, 20);   // R1, k0, k0 + 1
        const float r0c = qm8(w, 8), r0d = qm8(w, 24);   // R0, k0 + 8, k0 + 9
        const float r1c = qm8(w, 12), r1d = qm8(w, 28);  // R1, k0 + 8, k0 + 9
        const int64_t k0 = kb + 16 * s + 2 * tq;
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          if (m < a.mrows) {
            const float2 xa = __ldg(reinterpret_cast<const float2*>(a.x + m * kmax + k0));
            const float2 xb = __ldg(reinterpret_cast<const float2*>(a.x + m * kmax + k0 + 8));
            float t0 = s0[m], t1 = s1[m];
            t0 = fmaf(r0a, xa.x, t0);
            t0 = fmaf(r0b, xa.y, t0);
            t0 = fmaf(r0c, xb.x, t0);
            t0 = fmaf(r0d, xb.y, t0);
            t1 = fmaf(r1a, xa.x, t1);
            t1 = fmaf(r1b, xa.y, t1);
            t1 = fmaf(r1c, xb.x, t1);
            t1 = fmaf(r1d, xb.y, t1);
            s0[m] = t0;
            s1[m] = t1;
          }
        }
      }
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        acc0[m] = fmaf(dr0[h], s0[m], acc0[m]);
        acc1[m] = fmaf(dr1[h], s1[m], acc1[m]);
      }
    }
  }

  // fixed-order reduction over the four lanes of each row (xor 1, then xor 2);
  // addition is commutative, so all four lanes end with the same bits
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    acc0[m] += __shfl_xor_sync(0xFFFFFFFFu, acc0[m], 1);
    acc0[m] += __shfl_xor_sync(0xFFFFFFFFu, acc0[m], 2);
    acc1[m] += __shfl_xor_sync(0xFFFFFFFFu, acc1[m], 1);
    acc1[m] += __shfl_xor_sync(0xFFFFFFFFu, acc1[m], 2);
  }
  if (tq == 0) {
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      red[m][rg * 16 + g] = acc0[m];
      red[m][rg * 16 + g + 8] = acc1[m];
    }
  }
  __syncthreads();
  const int row = threadIdx.x < TILE_N ? (int)threadIdx.x : -1;
  float val[MT];
#pragma unroll
  for (int m = 0; m < MT; ++m) val[m] = row >= 0 ? red[m][row] : 0.0f;
  finish_tile<MT, 1, MT>(a.e, val, row, 0, tile, 0, a.mrows, split, s_arrival, (int)tile, &s_flag,
                         kred, []() { __syncthreads(); });
}

constexpr int64_t SIMT_M_LAUNCH = 8;  // token rows per launch

}  // namespace

MmaPlan simt_plan(const Weight* W, int num_sms) { return mma_plan(W, num_sms); }

size_t simt_partial_bytes(const Weight* W, const MmaPlan& p, int64_t M) {
  if (p.splits <= 1) return 0;
  const int64_t ml = M < SIMT_M_LAUNCH ? M : SIMT_M_LAUNCH;
  return (size_t)p.splits * (size_t)ml * (size_t)W->N_pad * sizeof(unsigned long long);
}

int simt_launch_count(int64_t M) { return (int)((M + SIMT_M_LAUNCH - 1) / SIMT_M_LAUNCH); }

int launch_simt(const Weight* W, const float* x, int64_t M, float* y, int32_t* idx,
                float* maxval, const MmaPlan& plan, const Workspace& ws, cudaStream_t s) {
  if (plan.splits > 1 && W->tiles > MAX_COUNTERS) return Q4_ERR_SHAPE;
  for (int64_t mb = 0; mb < M; mb += SIMT_M_LAUNCH) {
    const int mrows = (int)((M - mb) < SIMT_M_LAUNCH ? (M - mb) : SIMT_M_LAUNCH);
    SimtArgs a;
    a.nib = reinterpret_cast<const uint4*>(W->nib);
    a.scl = reinterpret_cast<const uint2*>(W->d);
    a.x = x + mb * W->K;
    a.K = W->K;
    a.KBP = W->KBP;
    a.mrows = mrows;
    a.kbp_per_split = plan.kbp_per_split;
    a.e.N = W->N;
    a.e.N_pad = W->N_pad;
    a.e.M = mrows;
    a.e.y = y ? y + mb * W->N : nullptr;
    a.e.idx = idx ? idx + mb : nullptr;
    a.e.maxval = (idx && maxval) ? maxval + mb : nullptr;
    a.e.splits = plan.splits;
    a.e.partial = ws.partial;
    a.e.counters = ws.counters;
    a.e.status = ws.status;
    a.e.keys = ws.keys + mb;
    a.e.argmax_done = ws.argmax_done;
    a.e.tiles = (int)W->tiles;
    a.e.poll_limit = poll_rounds();
    a.e.stall = 0;
    dim3 grid((unsigned)W->tiles, (unsigned)plan.splits);
    if (mrows == 1) simt_kernel<1><<<grid, SIMT_THREADS, 0, s>>>(a);
    else if (mrows == 2) simt_kernel<2><<<grid, SIMT_THREADS, 0, s>>>(a);
    else if (mrows <= 4) simt_kernel<4><<<grid, SIMT_THREADS, 0, s>>>(a);
    else simt_kernel<8><<<grid, SIMT_THREADS, 0, s>>>(a);
    if (cudaGetLastError() != cudaSuccess) return Q4_ERR_CUDA;
  }
  return Q4_OK;
}

}  // namespace q4
