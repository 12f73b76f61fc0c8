// q4mm_mma.cu — streaming tensor-core kernel for small and medium M.
//
// This is the decode path of the linear layer: M token rows (1 to 16 per
// launch) times a Q4_0 weight matrix read from HBM exactly once per call
// ("Why LLM Decoding Is Slow, and Why Batching Is (Almost) Free", §2-§4: decode
// streams every weight once per step, and the extra token rows of a batch ride
// along almost for free while the step stays memory-bound).  It replaces the
// two kernels of "Why Continuous Batching Slowed Down My LLM Inference Engine"
// (§"Two Rows of Input, Two Different Kernels") — a one-row GEMV and a tiled
// GEMM — with one kernel whose cost per weight hardly changes between 1 and
// 16 rows, so no row count needs a different kernel or a per-row relaunch.
//
// Per warp: one 16-row group of a 128-row tile over the CTA's K range.  Each
// lane loads 16 bytes per block pair (coalesced: a warp reads 512 contiguous
// bytes) that are exactly its A fragments of two m16n8k16 MMAs per block.
// The nibbles are unpacked in registers to exact bf16 (q - 8); the
// activations enter as B fragments holding three exact bf16 terms
// x = x0 + x1 + x2 per token row (term t of row m is MMA column 3m + t, or
// column t of the row's own column group in batch-invariant mode), split
// inside the kernel one pipeline stage ahead of their use.  The two
// MMAs of a block accumulate D_b = sum_{k in b} (q-8) x_t in fresh fp32
// registers; the block's fp16 scale is applied on the CUDA cores,
// acc = fma(d, D_b, acc), in ascending block order.  At the end the three
// terms of each token row are added in a fixed order (t = 0, 1, 2) and the
// K splits, if any, are added in ascending split order.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "q4mm_epilogue.cuh"
#include "q4mm_internal.h"

namespace q4 {
namespace {

constexpr int MAX_CG = 6;         // column groups per launch (48 MMA columns)

struct MmaArgs {
  const uint4* nib;     // fragment layout, 16 bytes per (tile, pair, rg, lane)
  const uint2* scl;     // 8 bytes per (tile, pair, rg, g)
  const float* x;       // [mrows, K] activations of this launch
  int64_t K, KBP;       // K, block pairs
  int mrows;            // token rows in this launch
  int dense;            // 1: column 3m + t; 0: column 8m + t (one row per group)
  int64_t kbp_per_split;
  unsigned int* status; // device status word (bounded-wait expiry)
  EpiArgs e;
};

// bf16 pair (q - 8) for nibble pair p of word w: 0x4300 | q is bf16(128 + q),
// and one bf16x2 FMA x * 1 + (-136) is exact.
__device__ __forceinline__ uint32_t nib_pair(uint32_t w, int p) {
  const uint32_t t = ((w >> (4 * p)) & 0x000F000Fu) | 0x43004300u;
  uint32_t r;
  asm("fma.rn.bf16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(t), "r"(0x3F803F80u), "r"(0xC308C308u));
  return r;
}

// D = A B + C with C = 0 (first k-step of a block) and with C = D (second).
__device__ __forceinline__ void mma_bf16_first(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%10, %10, %10, %10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.0f));
}
__device__ __forceinline__ void mma_bf16_acc(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                             uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ----------------------------------------------------------------------------
// Main kernel.  Grid (tiles, splits), one CTA per SM: 16 compute warps (warp w
// takes row group w % 8 of the 128-row tile and block pair w / 8 of each
// stage) + 1 producer warp.
//
// A ring of STAGES shared-memory stages holds two block pairs (128 k) of the
// tile each: 8 KB of weight fragments and 1 KB of scales, brought in by the
// producer with two bulk copies completing on the stage's mbarrier (the
// tile's block pairs are contiguous in the fragment layout).  The activations
// of a stage are read from global memory (tiny and shared by every CTA, so
// they stay in L2) two stages ahead into registers, split into exact bf16 B
// fragments one stage ahead and stored in the stage's fragment area.  One
// __syncthreads per iteration publishes the fragments and retires the slot
// the producer refills next.  The two warps of a row group add their sums in
// a fixed order at the end.
// ----------------------------------------------------------------------------
constexpr int COMPUTE_WARPS = 16;
constexpr int COMPUTE_THREADS = COMPUTE_WARPS * 32;
constexpr int KERNEL_THREADS = COMPUTE_THREADS + 32;
constexpr int PAIRS_PER_STAGE = 2;
constexpr int SMEM_LIMIT = 220 * 1024;

template <int C>
struct MmaCfg {
  static constexpr int MAXM = (C * 8) / 3 > C ? (C * 8) / 3 : C;  // rows per launch
  static constexpr int NIB = PAIRS_PER_STAGE * PAIR_NIB_BYTES;     // [pair][rg][lane] 16 B
  static constexpr int SCL = PAIRS_PER_STAGE * PAIR_SCL_BYTES;     // [pair][rg][g] 8 B
  static constexpr int XF = PAIRS_PER_STAGE * C * 2 * 32 * 16;     // [pair][cg][h][lane] 16 B
  static constexpr int SCL_OFF = NIB;
  static constexpr int XF_OFF = NIB + SCL;
  static constexpr int STAGE = XF_OFF + XF;
  static constexpr int RED = C * 8 * (TILE_N + 1) * 4 * 2;  // two partial sums per row
  static constexpr int STAGES_RAW = (SMEM_LIMIT - 256) / STAGE;
  static constexpr int STAGES = STAGES_RAW >= 16 ? 16 : 8;  // a power of two
  static constexpr int RING = STAGE * STAGES;
  static constexpr int BAR_OFF = RING > RED ? RING : RED;
  static constexpr int BYTES = BAR_OFF + STAGES * 8;
  static_assert(STAGES >= 4, "pipeline too shallow");
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Bounded wait (1 s); returns false on expiry.  The timer is read only after
// many polls, off the common path.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity) {
  unsigned long long t0 = 0;
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 255u) == 0u) {
      const unsigned long long now = globaltimer();
      if (t0 == 0) t0 = now;
      else if (now - t0 > 1000000000ull) return false;
    }
  }
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

template <int C>
__global__ void __launch_bounds__(KERNEL_THREADS, 1) mma_kernel(const MmaArgs a) {
  using S = MmaCfg<C>;
  constexpr int MAXM = S::MAXM;
  constexpr int STAGES = S::STAGES;
  extern __shared__ __align__(16) uint8_t smem[];
  __shared__ unsigned long long kred[4][MAXM];
  __shared__ int s_flag;
  __shared__ int s_err;

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const bool producer = warp == COMPUTE_WARPS;
  const int g = lane >> 2, tq = lane & 3;
  const int rg = warp & 7, pis = (warp >> 3) & 1;  // row group, pair within a stage
  const int64_t tile = blockIdx.x;
  const int split = blockIdx.y;
  const int64_t bp0 = (int64_t)split * a.kbp_per_split;
  const int64_t bp1 = min(a.KBP, bp0 + a.kbp_per_split);
  const int npairs = (int)(bp1 - bp0);
  const int nst = (npairs + PAIRS_PER_STAGE - 1) / PAIRS_PER_STAGE;  // stages of this CTA
  const int mrows = a.mrows;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::BAR_OFF);

  // conversion work items: pair (k, k + 1) of row m in a stage (128 k = 64 pairs)
  const int items = 64 * mrows;
  const int conv_passes = producer ? 0 : (tid < items) + (tid + COMPUTE_THREADS < items);
  const float* conv_src[2];
  int64_t conv_k_end[2];
  uint32_t conv_dst[2][3];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int jj = tid + r * COMPUTE_THREADS;
    const int m = r < conv_passes ? (jj >> 6) : 0, pp = jj & 63;
    const int kk = 2 * pp;                      // 0..126 within the stage
    const int pr = kk >> 6;                     // pair of the stage
    const int h = (kk >> 5) & 1, kb = kk & 31;  // block of the pair, k within block
    const int sks = kb >> 4, ks = kb & 15, half = ks >> 3, tql = (ks & 7) >> 1;
    conv_src[r] = a.x + (int64_t)m * a.K + bp0 * 64 + kk;
    conv_k_end[r] = a.K - bp0 * 64 - kk;  // the pair of stage i is real iff 128 i < this
#pragma unroll
    for (int t = 0; t < 3; ++t) {
      const int c = a.dense ? 3 * m + t : 8 * m + t;
      const int cg = c >> 3, gl = c & 7;
      conv_dst[r][t] = (uint32_t)(S::XF_OFF + (((pr * C + cg) * 2 + h) * 32 + 4 * gl + tql) * 16 +
                                  (2 * sks + half) * 4);
    }
  }
  auto load_raw = [&](int i, float2 (&v)[2]) {
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      v[r] = make_float2(0.0f, 0.0f);
      if (r < conv_passes && i < nst && (int64_t)i * 128 < conv_k_end[r])
        v[r] = __ldg(reinterpret_cast<const float2*>(conv_src[r] + (int64_t)i * 128));
    }
  };
  auto convert = [&](int i, const float2 (&v)[2]) {
    if (i >= nst || conv_passes == 0) return;
    uint8_t* st = smem + (i & (STAGES - 1)) * S::STAGE;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      if (r < conv_passes) {
        float v0 = v[r].x, v1 = v[r].y;
#pragma unroll
        for (int t = 0; t < 3; ++t) {  // exact split x = x0 + x1 + x2, each bf16
          const __nv_bfloat162 p = __floats2bfloat162_rn(v0, v1);
          v0 -= __low2float(p);
          v1 -= __high2float(p);
          *reinterpret_cast<__nv_bfloat162*>(st + conv_dst[r][t]) = p;
        }
      }
    }
  };

  // producer: block pairs [bp0 + 2i, bp0 + 2i + 2) of the tile into stage i
  const uint8_t* nib_g = reinterpret_cast<const uint8_t*>(a.nib) + (tile * a.KBP + bp0) * PAIR_NIB_BYTES;
  const uint8_t* scl_g = reinterpret_cast<const uint8_t*>(a.scl) + (tile * a.KBP + bp0) * PAIR_SCL_BYTES;
  int produced = 0;
  auto produce = [&](int i) {
    if (i < nst) {
      produced = i + 1;
      const int np = min(PAIRS_PER_STAGE, npairs - i * PAIRS_PER_STAGE);
      const uint32_t st = smem_u32(smem + (i & (STAGES - 1)) * S::STAGE);
      const uint32_t bar = smem_u32(&full[i & (STAGES - 1)]);
      mbar_expect_tx(bar, (uint32_t)(np * (PAIR_NIB_BYTES + PAIR_SCL_BYTES)));
      bulk_g2s(st, nib_g + (int64_t)i * S::NIB, np * PAIR_NIB_BYTES, bar);
      bulk_g2s(st + S::SCL_OFF, scl_g + (int64_t)i * S::SCL, np * PAIR_SCL_BYTES, bar);
    }
  };

  // zero every fragment slot once: padding columns are never written again
  for (int j = tid; j < STAGES * (S::XF / 16); j += KERNEL_THREADS) {
    const int stg = j / (S::XF / 16), w = j % (S::XF / 16);
    *reinterpret_cast<uint4*>(smem + stg * S::STAGE + S::XF_OFF + w * 16) = make_uint4(0u, 0u, 0u, 0u);
  }
  if (tid == 0) {
    for (int b = 0; b < STAGES; ++b) mbar_init(smem_u32(&full[b]), 1);
    s_err = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (producer && lane == 0) {
    for (int i = 0; i < STAGES - 1; ++i) produce(i);  // weights do not depend on earlier kernels
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");  // activations may come from the previous kernel

  float acc[C][4];
#pragma unroll
  for (int cg = 0; cg < C; ++cg)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[cg][e] = 0.0f;

  float2 raw_a[2], raw_b[2];  // activations of stages i + 1 and i + 2
  load_raw(0, raw_a);
  convert(0, raw_a);
  load_raw(1, raw_a);
  load_raw(2, raw_b);

  for (int i = 0; i < nst; ++i) {
    __syncthreads();  // stage i's fragments visible; slot of stage i - 1 retired
    if (s_err) break;  // uniform: read after the barrier by every thread
    if (producer) {
      if (lane == 0) produce(i + STAGES - 1);
      continue;
    }
    convert(i + 1, raw_a);
#pragma unroll
    for (int r = 0; r < 2; ++r) raw_a[r] = raw_b[r];
    load_raw(i + 3, raw_b);
    const int slot = i & (STAGES - 1);
    if (!mbar_wait_bounded(smem_u32(&full[slot]), (uint32_t)((i / STAGES) & 1))) {
      s_err = 1;  // skip this stage; every thread leaves at the next barrier
      continue;
    }
    if (i * PAIRS_PER_STAGE + pis >= npairs) continue;  // odd pair count: no second pair
    const uint8_t* st = smem + slot * S::STAGE;
    const uint4 wv = *reinterpret_cast<const uint4*>(st + ((pis * 8 + rg) * 32 + lane) * 16);
    const uint2 sv = *reinterpret_cast<const uint2*>(st + S::SCL_OFF + ((pis * 8 + rg) * 8 + g) * 8);
    const float2 dr0 = __half22float2(*reinterpret_cast<const __half2*>(&sv.x));  // d(R0, b0/b1)
    const float2 dr1 = __half22float2(*reinterpret_cast<const __half2*>(&sv.y));  // d(R1, b0/b1)
    const uint32_t w4[4] = {wv.x, wv.y, wv.z, wv.w};
    const uint4* xf = reinterpret_cast<const uint4*>(st + S::XF_OFF) + pis * (C * 64) + lane;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t a0[4], a1[4];
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        a0[p] = nib_pair(w4[2 * h], p);      // k-step 0 of block h of the pair
        a1[p] = nib_pair(w4[2 * h + 1], p);  // k-step 1
      }
      const float d0 = h ? dr0.y : dr0.x, d1 = h ? dr1.y : dr1.x;
#pragma unroll
      for (int cg = 0; cg < C; ++cg) {
        const uint4 bf = xf[(cg * 2 + h) * 32];
        float d[4];
        mma_bf16_first(d, a0, bf.x, bf.y);
        mma_bf16_acc(d, a1, bf.z, bf.w);
        acc[cg][0] = fmaf(d0, d[0], acc[cg][0]);
        acc[cg][1] = fmaf(d0, d[1], acc[cg][1]);
        acc[cg][2] = fmaf(d1, d[2], acc[cg][2]);
        acc[cg][3] = fmaf(d1, d[3], acc[cg][3]);
      }
    }
  }
  // On the normal path every issued stage was waited for.  After a timeout
  // the producer waits (bounded) for the copies it issued before the CTA exits.
  __syncthreads();
  if (s_err) {
    if (producer && lane == 0) {
      for (int i = (produced > STAGES ? produced - STAGES : 0); i < produced; ++i)
        mbar_wait_bounded(smem_u32(&full[i & (STAGES - 1)]), (uint32_t)((i / STAGES) & 1));
      atomicOr(a.status, (unsigned)Q4_ERR_TIMEOUT);
    }
    return;
  }

  // ---- gather: per tile row and MMA column, the two pair-in-stage halves ----
  float* red = reinterpret_cast<float*>(smem);  // [2][C*8][TILE_N + 1]
  constexpr int RS = C * 8 * (TILE_N + 1);
  if (!producer) {
#pragma unroll
    for (int cg = 0; cg < C; ++cg)
#pragma unroll
      for (int e = 0; e < 4; ++e)
        red[pis * RS + (cg * 8 + 2 * tq + (e & 1)) * (TILE_N + 1) + rg * 16 + g + 8 * (e >> 1)] =
            acc[cg][e];
  }
  __syncthreads();

  const int row = tid < TILE_N ? tid : -1;
  float val[MAXM];
#pragma unroll
  for (int m = 0; m < MAXM; ++m) val[m] = 0.0f;
  if (row >= 0) {
#pragma unroll
    for (int m = 0; m < MAXM; ++m) {
      if (m < mrows) {
        const int c0 = a.dense ? 3 * m : 8 * m;
        float v = 0.0f;
#pragma unroll
        for (int t = 0; t < 3; ++t)  // fixed order: term 0..2, each the even + odd pair sums
          v += red[(c0 + t) * (TILE_N + 1) + row] + red[RS + (c0 + t) * (TILE_N + 1) + row];
        val[m] = v;
      }
    }
  }
  finish_tile<MAXM>(a.e, val, row, tile, 0, mrows, split, (int)tile, &s_flag, kred,
                    []() { __syncthreads(); });
}

template <int C>
int launch_c(const Weight* W, const float* x, int mrows, int dense, float* y, int32_t* idx,
             float* maxval, const MmaPlan& plan, const Workspace& ws, int64_t mb, cudaStream_t s) {
  using S = MmaCfg<C>;
  MmaArgs a;
  a.nib = reinterpret_cast<const uint4*>(W->nib);
  a.scl = reinterpret_cast<const uint2*>(W->d);
  a.x = x;
  a.K = W->K;
  a.KBP = W->KBP;
  a.mrows = mrows;
  a.dense = dense;
  a.kbp_per_split = plan.kbp_per_split;
  a.status = ws.status;
  a.e.N = W->N;
  a.e.N_pad = W->N_pad;
  a.e.M = mrows;
  a.e.y = y ? y + mb * W->N : nullptr;
  a.e.idx = idx ? idx + mb : nullptr;
  a.e.maxval = (idx && maxval) ? maxval + mb : nullptr;
  a.e.splits = plan.splits;
  a.e.partial = ws.partial;
  a.e.counters = ws.counters;
  a.e.keys = ws.keys + mb;
  a.e.argmax_done = ws.argmax_done;
  a.e.tiles = (int)W->tiles;
  static bool attr_set[64] = {};
  if (!attr_set[W->device & 63]) {
    if (cudaFuncSetAttribute(mma_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             S::BYTES) != cudaSuccess)
      return Q4_ERR_CUDA;
    attr_set[W->device & 63] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)W->tiles, (unsigned)plan.splits, 1);
  cfg.blockDim = dim3(KERNEL_THREADS);
  cfg.dynamicSmemBytes = S::BYTES;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mma_kernel<C>, a) == cudaSuccess ? Q4_OK : Q4_ERR_CUDA;
}

// Rows per launch: 16 with dense packing (6 column groups), 6 with one row
// per column group (batch-invariant mode).
int rows_per_launch(bool batch_invariant) { return batch_invariant ? MAX_CG : (MAX_CG * 8) / 3; }

}  // namespace

MmaPlan mma_plan(const Weight* W, int num_sms) {
  // K partition from N and K only (never from M).  One CTA per SM: splits =
  // floor(SMs / tiles) for a single wave, at least one, and small enough that
  // each CTA keeps at least four stages (eight block pairs).
  MmaPlan p;
  int64_t sp = (int64_t)num_sms / W->tiles;
  int64_t cap = W->KBP / (4 * PAIRS_PER_STAGE);
  if (cap < 1) cap = 1;
  if (cap > 64) cap = 64;
  if (sp < 1) sp = 1;
  if (sp > cap) sp = cap;
  p.kbp_per_split = (W->KBP + sp - 1) / sp;
  p.splits = (int)((W->KBP + p.kbp_per_split - 1) / p.kbp_per_split);
  return p;
}

size_t mma_partial_bytes(const Weight* W, const MmaPlan& p, int64_t M, bool batch_invariant) {
  if (p.splits <= 1) return 0;
  const int64_t rpl = rows_per_launch(batch_invariant);
  const int64_t ml = M < rpl ? M : rpl;
  return (size_t)p.splits * (size_t)ml * (size_t)W->N_pad * sizeof(float);
}

int mma_launch_count(int64_t M, bool batch_invariant) {
  const int64_t rpl = rows_per_launch(batch_invariant);
  return (int)((M + rpl - 1) / rpl);
}

int launch_mma(const Weight* W, const float* x, int64_t M, float* y, int32_t* idx, float* maxval,
               const MmaPlan& plan, bool batch_invariant, const Workspace& ws, cudaStream_t s) {
  const int64_t rpl = rows_per_launch(batch_invariant);
  const int dense = batch_invariant ? 0 : 1;
  for (int64_t mb = 0; mb < M; mb += rpl) {
    const int mrows = (int)((M - mb) < rpl ? (M - mb) : rpl);
    if (plan.splits > 1 && W->tiles > MAX_COUNTERS) return Q4_ERR_SHAPE;
    // column groups needed for this launch
    const int ncg = dense ? (3 * mrows + 7) / 8 : mrows;
    const float* xs = x + mb * W->K;
    int st;
    switch (ncg) {
      case 1: st = launch_c<1>(W, xs, mrows, dense, y, idx, maxval, plan, ws, mb, s); break;
      case 2: st = launch_c<2>(W, xs, mrows, dense, y, idx, maxval, plan, ws, mb, s); break;
      case 3: st = launch_c<3>(W, xs, mrows, dense, y, idx, maxval, plan, ws, mb, s); break;
      case 4: st = launch_c<4>(W, xs, mrows, dense, y, idx, maxval, plan, ws, mb, s); break;
      case 5: st = launch_c<5>(W, xs, mrows, dense, y, idx, maxval, plan, ws, mb, s); break;
      default: st = launch_c<6>(W, xs, mrows, dense, y, idx, maxval, plan, ws, mb, s); break;
    }
    if (st) return st;
  }
  return Q4_OK;
}

}  // namespace q4
