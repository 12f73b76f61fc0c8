// q4mm_tc.cu — tensor-core (tcgen05 / TMEM) path of the Q4_0 matmul.
//
// For M token rows this is the "GEMM" side of the kernel split described in
// "Why Continuous Batching Slowed Down My LLM Inference Engine"
// (§"Two Rows of Input, Two Different Kernels"): many rows processed together
// so each weight read serves all of them ("Why LLM Decoding Is Slow, and Why
// Batching Is (Almost) Free", §4).  Dequantization happens on the fly in the
// kernel; the weights are streamed from HBM exactly once per CTA pass.
//
// Exactness.  The contraction must match the fp64 reference to about fp32
// accuracy, so operands are exact:
//   A (weights)   = (q - 8), small integers, exact in bf16, written by the
//                   CUDA cores straight into tensor memory (no smem round
//                   trip): bf16(128 + q) is 0x4300 | q, minus 136 is exact;
//   B (activations) = x split into three bf16 terms x0 + x1 + x2 == x
//                   exactly (a pre-pass kernel), accumulated by three MMAs
//                   into the same fp32 accumulator;
//   the per-block scale d is applied on the CUDA cores: for each 32-weight
//   block the 128 x M_TILE accumulator D_b = sum_{k in b} (q-8) x is read
//   from TMEM and folded as acc = fma(d, D_b, acc).
//
// Per CTA: one 128-row weight tile (one TMEM lane per row), one K range (a
// fixed split that depends on N and K only), one tile of M_TILE token rows.
// Warp roles (320 threads):
//   warps 0-7  convert + epilogue.  Warp w serves TMEM lane quarter w % 4;
//              warps 0-3 take even blocks, warps 4-7 odd blocks.
//   warp 8     TMA producer: 1-D bulk copies of nibbles, scales and the
//              activation operand of one block per smem stage.
//   warp 9     TMEM allocator and the single MMA-issuing thread.
// Every mbarrier wait is bounded (globaltimer); on expiry the CTA records
// Q4_ERR_TIMEOUT in the device status word, drains what it issued and exits.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "q4mm_internal.h"

namespace q4 {
namespace {

constexpr int TC_THREADS = 320;
constexpr int MATH_WARPS = 8;
constexpr int PRODUCER_WARP = 8;
constexpr int MMA_WARP = 9;
constexpr int TMEM_COLS = 512;
constexpr int MAX_STAGES = 32;
constexpr int SMEM_BUDGET = 200 * 1024;
constexpr int LAG = 2;  // iterations between converting a block and reading its accumulator
constexpr unsigned long long WAIT_NS = 1000000000ull;  // 1 s bound on any wait

template <int MT>
struct Cfg {
  static constexpr int NIB_BYTES = TILE_N * 16;            // 2048
  static constexpr int SCL_BYTES = TILE_N * 2;             // 256
  static constexpr int BOP_BYTES = 192 * MT;               // 3 terms x 2 k-steps x MT rows x 16 k x 2 B
  static constexpr int STAGE_BYTES = NIB_BYTES + SCL_BYTES + BOP_BYTES;
  static constexpr int SLOT_COLS = 16 + MT;                // A: 16 columns, D: MT columns
  static constexpr int NSLOT = ((TMEM_COLS / SLOT_COLS) / 2) * 2;
  static constexpr int DSL_BYTES = NSLOT * TILE_N * 4;
  static constexpr int BAR_BYTES = (2 * MAX_STAGES + 2 * 16 + 4) * 8;
  static constexpr int NST_RAW = (SMEM_BUDGET - DSL_BYTES - BAR_BYTES - 64) / STAGE_BYTES;
  static constexpr int NST = NST_RAW > MAX_STAGES ? MAX_STAGES : NST_RAW;
  static constexpr int SMEM_BYTES = NST * STAGE_BYTES + DSL_BYTES + BAR_BYTES + 64;
  static_assert(NSLOT >= 2 * (LAG + 1), "TMEM slots must cover the conversion lag");
  static_assert(NSLOT <= 16, "barrier area sized for 16 slots");
  static_assert(NST >= 4, "pipeline too shallow");
  static_assert(MT % 16 == 0 && MT <= 64, "M tile");
  static_assert(MT * TILE_N * 4 <= NST * STAGE_BYTES, "group-combine buffer");
};

struct TcArgs {
  const uint8_t* nib;
  const uint16_t* d;
  const uint8_t* xop;  // activation operand, [mtiles][KB][192*MT] bytes
  int64_t KB, K, N, N_pad;
  int64_t M;           // rows in this launch
  float* y;
  int32_t* idx;
  float* maxval;
  int splits;
  int64_t kb_per_split;
  int mtiles;
  int tiles;
  float* partial;
  unsigned int* counters;
  unsigned long long* keys;
  unsigned int* argmax_done;
  unsigned int* status;
};

// ----------------------------------------------------------------------------
// PTX helpers
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
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

// Bounded wait: returns false (and raises the CTA error flag) if the phase
// does not complete within WAIT_NS, or if another role already gave up.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  for (uint32_t i = 0;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 63u) {
      if (*err) return false;
      if (globaltimer() - t0 > WAIT_NS) {
        *err = 1;
        return false;
      }
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

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]^T, kind::f16 (bf16 inputs, fp32 accumulate).
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15])
      : "memory");
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor: K-major, no swizzle.  Core matrices are
// 8 rows x 16 bytes stored contiguously; lbo = byte distance between core
// matrices adjacent along K, sbo = between core matrices adjacent along N.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((addr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version for tcgen05
  return d;                // base offset 0, relative LBO, layout type 0 (no swizzle)
}

// Instruction descriptor, kind::f16: fp32 accumulator, bf16 A and B, both
// K-major, M = 128, N = n.
__host__ __device__ constexpr uint32_t idesc_bf16(int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}

// (q - 8) for the nibble pair at bits (4p, 16 + 4p) of w, as exact bf16x2.
__device__ __forceinline__ uint32_t nib_pair_bf16(uint32_t w, int p) {
  const uint32_t t = ((w >> (4 * p)) & 0x000F000Fu) | 0x43004300u;  // bf16 (128 + q) pair
  __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162*>(&t);
  h = __hsub2(h, __floats2bfloat162_rn(136.0f, 136.0f));
  return *reinterpret_cast<const uint32_t*>(&h);
}

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

// ----------------------------------------------------------------------------
// Pre-pass: x[M, K] fp32 -> activation operand, three exact bf16 terms, laid
// out per (m tile, block) as the MMA reads it:
//   [k-step s (2)][term t (3)][k group g (2)][row group rg (MT/8)][row (8)][8 k]
// One thread per (m tile, block, row, s, g): 8 consecutive k of one row.
// ----------------------------------------------------------------------------
template <int MT>
__global__ void __launch_bounds__(256) xop_kernel(const float* __restrict__ x, int64_t M, int64_t K,
                                                  int64_t KB, int mtiles, uint8_t* __restrict__ xop) {
  asm volatile("griddepcontrol.launch_dependents;");
  const int64_t total = (int64_t)mtiles * KB * MT * 4;
  for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < total;
       t += (int64_t)gridDim.x * blockDim.x) {
    const int sg = (int)(t & 3);
    const int rr = (int)((t >> 2) % MT);
    const int64_t b = (t >> 2) / MT % KB;
    const int64_t mt = (t >> 2) / MT / KB;
    const int s = sg >> 1, g = sg & 1;
    const int64_t m = mt * MT + rr;
    float v[8];
    if (m < M) {
      const float4* src = reinterpret_cast<const float4*>(x + m * K + b * BLOCK_K + s * 16 + g * 8);
      const float4 a = src[0], c = src[1];
      v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
      v[4] = c.x; v[5] = c.y; v[6] = c.z; v[7] = c.w;
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) v[e] = 0.0f;
    }
    uint32_t out[3][4];
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
      float r0 = v[e], r1 = v[e + 1];
      __nv_bfloat162 p0 = __floats2bfloat162_rn(r0, r1);
      r0 -= __low2float(p0);
      r1 -= __high2float(p0);
      __nv_bfloat162 p1 = __floats2bfloat162_rn(r0, r1);
      r0 -= __low2float(p1);
      r1 -= __high2float(p1);
      __nv_bfloat162 p2 = __floats2bfloat162_rn(r0, r1);
      out[0][e / 2] = *reinterpret_cast<uint32_t*>(&p0);
      out[1][e / 2] = *reinterpret_cast<uint32_t*>(&p1);
      out[2][e / 2] = *reinterpret_cast<uint32_t*>(&p2);
    }
    uint8_t* base = xop + (mt * KB + b) * (int64_t)(192 * MT);
    const int rg = rr >> 3, r8 = rr & 7;
#pragma unroll
    for (int term = 0; term < 3; ++term) {
      const int64_t off = ((((int64_t)(s * 3 + term) * 2 + g) * (MT / 8) + rg) * 8 + r8) * 16;
      *reinterpret_cast<uint4*>(base + off) =
          make_uint4(out[term][0], out[term][1], out[term][2], out[term][3]);
    }
  }
}

// ----------------------------------------------------------------------------
// Main kernel
// ----------------------------------------------------------------------------
template <int MT>
__global__ void __launch_bounds__(TC_THREADS, 1) tc_kernel(const TcArgs a) {
  using C = Cfg<MT>;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* stages = smem;
  float* dsl = reinterpret_cast<float*>(smem + C::NST * C::STAGE_BYTES);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::NST * C::STAGE_BYTES + C::DSL_BYTES);
  uint64_t* full = bars;
  uint64_t* empty = bars + MAX_STAGES;
  uint64_t* afull = bars + 2 * MAX_STAGES;
  uint64_t* dfull = bars + 2 * MAX_STAGES + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * MAX_STAGES + 32);
  volatile int* err = reinterpret_cast<volatile int*>(tmem_slot + 2);
  __shared__ int s_last;

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int tile = blockIdx.x, split = blockIdx.y, mt = blockIdx.z;
  const int64_t kb0 = (int64_t)split * a.kb_per_split;
  const int64_t kb1 = min(a.KB, kb0 + a.kb_per_split);
  const int nblk = (int)(kb1 - kb0);

  if (tid == 0) {
    for (int i = 0; i < C::NST; ++i) {
      mbar_init(smem_u32(&full[i]), 1);
      mbar_init(smem_u32(&empty[i]), 4 + 1);
    }
    for (int i = 0; i < C::NSLOT; ++i) {
      mbar_init(smem_u32(&afull[i]), 4);
      mbar_init(smem_u32(&dfull[i]), 1);
    }
    *err = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == MMA_WARP) tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  float acc[MT];
#pragma unroll
  for (int m = 0; m < MT; ++m) acc[m] = 0.0f;

  if (warp == PRODUCER_WARP) {
    if (lane == 0) {
      asm volatile("griddepcontrol.wait;" ::: "memory");
      const uint8_t* nib_base = a.nib + ((int64_t)tile * a.KB + kb0) * TILE_N * 16;
      const uint8_t* scl_base =
          reinterpret_cast<const uint8_t*>(a.d + ((int64_t)tile * a.KB + kb0) * TILE_N);
      const uint8_t* bop_base = a.xop + ((int64_t)mt * a.KB + kb0) * (int64_t)C::BOP_BYTES;
      int issued = 0;
      for (int j = 0; j < nblk; ++j) {
        const int st = j % C::NST;
        if (!mbar_wait(smem_u32(&empty[st]), ((j / C::NST) & 1) ^ 1, err)) break;
        const uint32_t sb = smem_u32(stages + st * C::STAGE_BYTES);
        const uint32_t fb = smem_u32(&full[st]);
        mbar_expect_tx(fb, C::STAGE_BYTES);
        bulk_g2s(sb, nib_base + (int64_t)j * C::NIB_BYTES, C::NIB_BYTES, fb);
        bulk_g2s(sb + C::NIB_BYTES, scl_base + (int64_t)j * C::SCL_BYTES, C::SCL_BYTES, fb);
        bulk_g2s(sb + C::NIB_BYTES + C::SCL_BYTES, bop_base + (int64_t)j * C::BOP_BYTES,
                 C::BOP_BYTES, fb);
        issued = j + 1;
      }
      // drain: every issued copy has landed before the CTA may exit
      for (int j = max(0, issued - C::NST); j < issued; ++j) {
        const uint32_t fb = smem_u32(&full[j % C::NST]);
        const unsigned long long t0 = globaltimer();
        while (!mbar_try_wait(fb, (j / C::NST) & 1) && globaltimer() - t0 < WAIT_NS) {
        }
      }
    }
  } else if (warp == MMA_WARP) {
    if (lane == 0) {
      constexpr uint32_t IDESC = idesc_bf16(MT);
      int issued = 0;
      for (int j = 0; j < nblk; ++j) {
        const int st = j % C::NST, sl = j % C::NSLOT;
        if (!mbar_wait(smem_u32(&full[st]), (j / C::NST) & 1, err)) break;
        if (!mbar_wait(smem_u32(&afull[sl]), (j / C::NSLOT) & 1, err)) break;
        tc_fence_after();
        const uint32_t bop = smem_u32(stages + st * C::STAGE_BYTES + C::NIB_BYTES + C::SCL_BYTES);
        const uint32_t a_col = tmem + (uint32_t)(sl * C::SLOT_COLS);
        const uint32_t d_col = a_col + 16u;
#pragma unroll
        for (int s = 0; s < 2; ++s) {
#pragma unroll
          for (int t = 0; t < 3; ++t) {
            const uint64_t bd = smem_desc(bop + (uint32_t)((s * 3 + t) * 32 * MT), 16u * MT, 128u);
            mma_ts(d_col, a_col + 8u * s, bd, IDESC, (s | t) != 0);
          }
        }
        mma_commit(smem_u32(&dfull[sl]));
        mma_commit(smem_u32(&empty[st]));
        issued = j + 1;
      }
      if (issued > 0) {  // drain: the last commit covers every MMA issued
        const int j = issued - 1;
        const uint32_t db = smem_u32(&dfull[j % C::NSLOT]);
        const unsigned long long t0 = globaltimer();
        while (!mbar_try_wait(db, (j / C::NSLOT) & 1) && globaltimer() - t0 < WAIT_NS) {
        }
      }
    }
    __syncwarp();
  } else {
    // ---- convert + epilogue warps ----
    const int q = warp & 3, g = warp >> 2;
    const int row = q * 32 + lane;
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    const int n_g = nblk > g ? (nblk - g + 1) / 2 : 0;
    for (int i = 0; i < n_g + LAG; ++i) {
      if (i < n_g) {
        const int j = g + 2 * i;
        const int st = j % C::NST, sl = j % C::NSLOT;
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&full[st]), (j / C::NST) & 1, err))) break;
        const uint8_t* sp = stages + st * C::STAGE_BYTES;
        const uint4 v = *reinterpret_cast<const uint4*>(sp + row * 16);
        const uint16_t dh = *reinterpret_cast<const uint16_t*>(sp + C::NIB_BYTES + row * 2);
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty[st]));
        dsl[sl * TILE_N + row] = __half2float(__ushort_as_half(dh));
        const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
        uint32_t av[16];
#pragma unroll
        for (int w = 0; w < 4; ++w)
#pragma unroll
          for (int p = 0; p < 4; ++p) av[4 * w + p] = nib_pair_bf16(wv[w], p);
        tmem_st16(tmem + lane_off + (uint32_t)(sl * C::SLOT_COLS), av);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&afull[sl]));
      }
      if (i >= LAG) {
        const int j = g + 2 * (i - LAG);
        const int sl = j % C::NSLOT;
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&dfull[sl]), (j / C::NSLOT) & 1, err)))
          break;
        tc_fence_after();
        const float dsc = dsl[sl * TILE_N + row];
        const uint32_t dcol = tmem + lane_off + (uint32_t)(sl * C::SLOT_COLS + 16);
#pragma unroll
        for (int c = 0; c < MT; c += 16) {
          float dv[16];
          tmem_ld16(dcol + (uint32_t)c, dv);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; ++e) acc[c + e] = fmaf(dsc, dv[e], acc[c + e]);
        }
      }
    }
  }

  // ---- combine the two block groups (fixed order: even + odd) ----
  tc_fence_before();
  __syncthreads();
  float* comb = reinterpret_cast<float*>(stages);
  if (warp >= 4 && warp < MATH_WARPS) {
    const int row = (warp & 3) * 32 + lane;
#pragma unroll
    for (int m = 0; m < MT; ++m) comb[m * TILE_N + row] = acc[m];
  }
  __syncthreads();
  if (warp == MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
  const bool timed_out = *err != 0;
  if (timed_out) {
    if (tid == 0) atomicOr(a.status, (unsigned)Q4_ERR_TIMEOUT);
    return;
  }
  if (warp >= 4) return;  // warps 0-3 own the 128 rows from here on

  const int row = warp * 32 + lane;
  const int64_t n = (int64_t)tile * TILE_N + row;
  const int64_t m0 = (int64_t)mt * MT;
  const int mcount = (int)min((int64_t)MT, a.M - m0);
#pragma unroll
  for (int m = 0; m < MT; ++m) acc[m] += comb[m * TILE_N + row];

  // named barrier over warps 0-3 only (128 threads)
  auto sync128 = []() { asm volatile("bar.sync 1, 128;" ::: "memory"); };

  if (a.splits > 1) {
#pragma unroll
    for (int m = 0; m < MT; ++m)
      if (m < mcount) a.partial[((int64_t)split * a.M + m0 + m) * a.N_pad + n] = acc[m];
    __threadfence();
    sync128();
    if (row == 0) {
      const unsigned prev = atomicAdd(&a.counters[tile * a.mtiles + mt], 1u);
      s_last = (prev == (unsigned)(a.splits - 1));
    }
    sync128();
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
    if (row == 0) a.counters[tile * a.mtiles + mt] = 0u;
  }

  if (a.idx == nullptr) {
    if (n < a.N) {
#pragma unroll
      for (int m = 0; m < MT; ++m)
        if (m < mcount) a.y[(m0 + m) * a.N + n] = acc[m];
    }
    return;
  }

  // ---- fused greedy pick ----
  __shared__ unsigned long long red[4][MT];
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    unsigned long long k = (m < mcount && n < a.N) ? argmax_key(acc[m], (uint32_t)n) : 0ull;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const unsigned long long o = __shfl_xor_sync(0xFFFFFFFFu, k, off);
      k = o > k ? o : k;
    }
    if (lane == 0) red[warp][m] = k;
  }
  sync128();
  if (row < mcount) {
    unsigned long long k = red[0][row];
#pragma unroll
    for (int w = 1; w < 4; ++w) k = red[w][row] > k ? red[w][row] : k;
    atomicMax(&a.keys[m0 + row], k);
  }
  __threadfence();
  sync128();
  if (row == 0) {
    const unsigned prev = atomicAdd(a.argmax_done, 1u);
    s_last = (prev == (unsigned)(a.tiles * a.mtiles - 1));
  }
  sync128();
  if (!s_last) return;
  __threadfence();
  for (int64_t m = row; m < a.M; m += TILE_N) {
    const unsigned long long k = atomicExch(&a.keys[m], 0ull);
    a.idx[m] = k == 0ull ? 0 : (int32_t)(0xFFFFFFFFu - (uint32_t)(k & 0xFFFFFFFFull));
    if (a.maxval) a.maxval[m] = key_value(k);
  }
  if (row == 0) *a.argmax_done = 0u;
}

constexpr int64_t TC_M_LAUNCH = 256;  // rows per launch pair (pre-pass + main)

int mt_for(int64_t M, bool batch_invariant) {
  if (batch_invariant) return 16;
  return M <= 16 ? 16 : (M <= 32 ? 32 : 64);
}

template <int MT>
int launch_mt(const Weight* W, const float* x, int64_t ml, float* y, int32_t* idx, float* maxval,
              const TcPlan& plan, const Workspace& ws, int64_t mb, cudaStream_t s) {
  using C = Cfg<MT>;
  const int mtiles = (int)((ml + MT - 1) / MT);
  if (plan.splits > 1 && W->tiles * mtiles > MAX_COUNTERS) return Q4_ERR_SHAPE;
  // pre-pass
  {
    const int64_t total = (int64_t)mtiles * W->KB * MT * 4;
    const int64_t want = (total + 255) / 256;
    const int blocks = (int)(want < 4096 ? want : 4096);
    xop_kernel<MT><<<blocks, 256, 0, s>>>(x, ml, W->K, W->KB, mtiles, static_cast<uint8_t*>(ws.xop));
    if (cudaGetLastError() != cudaSuccess) return Q4_ERR_CUDA;
  }
  static bool attr_set[64] = {};
  if (!attr_set[W->device & 63]) {
    if (cudaFuncSetAttribute(tc_kernel<MT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::SMEM_BYTES) != cudaSuccess)
      return Q4_ERR_CUDA;
    attr_set[W->device & 63] = true;
  }
  TcArgs a;
  a.nib = W->nib;
  a.d = W->d;
  a.xop = static_cast<const uint8_t*>(ws.xop);
  a.KB = W->KB;
  a.K = W->K;
  a.N = W->N;
  a.N_pad = W->N_pad;
  a.M = ml;
  a.y = y ? y + mb * W->N : nullptr;
  a.idx = idx ? idx + mb : nullptr;
  a.maxval = (idx && maxval) ? maxval + mb : nullptr;
  a.splits = plan.splits;
  a.kb_per_split = plan.kb_per_split;
  a.mtiles = mtiles;
  a.tiles = (int)W->tiles;
  a.partial = ws.partial;
  a.counters = ws.counters;
  a.keys = ws.keys + mb;
  a.argmax_done = ws.argmax_done;
  a.status = ws.status;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)W->tiles, (unsigned)plan.splits, (unsigned)mtiles);
  cfg.blockDim = dim3(TC_THREADS);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, tc_kernel<MT>, a) != cudaSuccess) return Q4_ERR_CUDA;
  return Q4_OK;
}

}  // namespace

bool tc_kernel_built() { return true; }

TcPlan tc_plan(const Weight* W, int64_t M, int num_sms, bool batch_invariant) {
  TcPlan p;
  p.m_tile = mt_for(M < TC_M_LAUNCH ? M : TC_M_LAUNCH, batch_invariant);
  // K partition from N and K only: fill the SMs with one CTA each, balancing
  // waves against blocks per CTA.
  const int64_t tiles = W->tiles;
  int64_t best_s = 1, best_cost = -1;
  const int64_t smax = W->KB < 32 ? W->KB : 32;
  for (int64_t s = 1; s <= smax; ++s) {
    const int64_t kbps = (W->KB + s - 1) / s;
    const int64_t waves = (tiles * s + num_sms - 1) / num_sms;
    const int64_t cost = waves * (kbps + 8);  // + per-CTA fixed cost in block units
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best_s = s;
    }
  }
  p.kb_per_split = (W->KB + best_s - 1) / best_s;
  p.splits = (int)((W->KB + p.kb_per_split - 1) / p.kb_per_split);
  return p;
}

size_t tc_partial_bytes(const Weight* W, const TcPlan& p, int64_t M) {
  if (p.splits <= 1) return 0;
  const int64_t ml = M < TC_M_LAUNCH ? M : TC_M_LAUNCH;
  return (size_t)p.splits * (size_t)ml * (size_t)W->N_pad * sizeof(float);
}

size_t tc_xop_bytes(const Weight* W, const TcPlan& p, int64_t M) {
  const int64_t ml = M < TC_M_LAUNCH ? M : TC_M_LAUNCH;
  const int64_t mtiles = (ml + p.m_tile - 1) / p.m_tile;
  return (size_t)mtiles * (size_t)W->KB * 192u * (size_t)p.m_tile;
}

int tc_launch_count(const TcPlan&, int64_t M) {
  return 2 * (int)((M + TC_M_LAUNCH - 1) / TC_M_LAUNCH);
}

int launch_tc(const Weight* W, const float* x, int64_t M, float* y, int32_t* idx, float* maxval,
              const TcPlan& plan, const Workspace& ws, cudaStream_t s) {
  for (int64_t mb = 0; mb < M; mb += TC_M_LAUNCH) {
    const int64_t ml = (M - mb) < TC_M_LAUNCH ? (M - mb) : TC_M_LAUNCH;
    int st;
    switch (plan.m_tile) {
      case 16: st = launch_mt<16>(W, x + mb * W->K, ml, y, idx, maxval, plan, ws, mb, s); break;
      case 32: st = launch_mt<32>(W, x + mb * W->K, ml, y, idx, maxval, plan, ws, mb, s); break;
      default: st = launch_mt<64>(W, x + mb * W->K, ml, y, idx, maxval, plan, ws, mb, s); break;
    }
    if (st) return st;
  }
  return Q4_OK;
}

}  // namespace q4
