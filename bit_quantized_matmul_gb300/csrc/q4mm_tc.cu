// q4mm_tc.cu — tensor-core (tcgen05 / TMEM) path of the Q4_0 matmul, for
// many token rows.
//
// For several token rows this is the "GEMM" side of the kernel split in
// "Why Continuous Batching Slowed Down My LLM Inference Engine"
// (§"Two Rows of Input, Two Different Kernels"): all rows of the call share
// one pass over the weights ("Why LLM Decoding Is Slow, and Why Batching Is
// (Almost) Free", §4 "Share the Weights Across Users"), and the 4-bit
// weights are dequantized on the fly inside the kernel.
//
// Exactness.  The result must match the fp64 reference to about fp32
// accuracy, so every tensor-core product is exact:
//   A (weights)     w = (q - 8) * d has at most 14 significant bits (a 4-bit
//                   integer times the 11-bit significand of the fp16 scale),
//                   so it is the exact sum of two bf16 terms: hi = bf16(w)
//                   (round to nearest) and lo = w - hi.  The CUDA cores form
//                   both and write them into tensor memory.
//   B (activations) x split into three bf16 terms x0 + x1 + x2 == x exactly
//                   (pre-pass kernel), stacked along the MMA's N dimension
//                   (term t of token row m is B row t*MTR + m).
// With the scale inside A, one fp32 accumulator in tensor memory takes the
// whole K range: per k-step two MMAs (hi, lo) of 128 x NB x 16, NB up to 240
// (80 token rows per CTA), and the CUDA cores read the accumulator once at
// the end: y[m, n] = (D[n, m] + D[n, MTR+m]) + D[n, 2 MTR+m].
//
// Work decomposition.  CTA = one 128-row weight tile (a TMEM lane per row) x
// one K range (split from the shapes) x one tile of MTR token rows.  The K
// range is processed in units of U = 4 blocks; every barrier, bulk copy and
// commit is per unit.  Roles (320 threads):
//   warps 0-7  converters: nibbles and scales -> hi/lo bf16 weights in the
//              TMEM A ring; two groups of four (one per TMEM lane quarter)
//              take alternate units; warps 0-3 also run the epilogue
//   warp  8    bulk-copy producer: nibbles, scales and the activation
//              operand of a unit into one smem stage
//   warp  9    MMA issuer (one thread, so the accumulator's MMAs are ordered);
//              owns the TMEM allocation
// Every mbarrier wait is bounded; on expiry the CTA records STATUS_TIMEOUT in
// the device status word, drains what it issued, frees TMEM and exits.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>

#include "q4mm_epilogue.cuh"
#include "q4mm_internal.h"

namespace q4 {
namespace {

constexpr int U = 4;                    // blocks per unit (two block pairs)
constexpr int PROD_WARP = 8;
constexpr int MMA_WARP = 9;
constexpr int TC_THREADS = 10 * 32;
constexpr int TMEM_COLS = 512;
constexpr int EPI_ROWS = 16;            // token rows per epilogue chunk
// Barriers are per unit, in a ring of NBR units: unit u uses index u % NBR at
// phase parity (u / NBR) & 1.  Every role handles its units in order and NBR is
// a multiple of the role strides (1 and 2), so a waiter has always observed
// the previous phase of the same barrier before it waits for the next one.
constexpr int NBR = 64;
constexpr int SMEM_BUDGET = 200 * 1024;
constexpr unsigned long long WAIT_NS = 1000000000ull;  // 1 s bound on any wait

template <int NB>
struct Cfg {
  static constexpr int MTR = NB / 3;                   // token rows per CTA
  static constexpr int NIB_BYTES = U * TILE_N * 16;    // 8 KB
  static constexpr int SCL_OFF = NIB_BYTES;
  static constexpr int SCL_BYTES = U * TILE_N * 2;     // 1 KB
  static constexpr int BOP_OFF = SCL_OFF + SCL_BYTES;
  static constexpr int BOP_BLOCK = 64 * NB;            // 2 k-steps x NB rows x 16 k x 2 B
  static constexpr int STAGE_BYTES = BOP_OFF + U * BOP_BLOCK;
  static constexpr int A_BLOCK_COLS = 32;              // [term hi/lo][k-step][8 columns]
  static constexpr int A_UNIT_COLS = U * A_BLOCK_COLS;  // 128
  static constexpr int NA_RAW = (TMEM_COLS - NB) / A_UNIT_COLS;
  static constexpr int NA = NA_RAW > 3 ? 3 : NA_RAW;   // A ring (units)
  static constexpr int BAR_BYTES = (4 * NBR + 1) * 8 + 16;
  static constexpr int NST_RAW = (SMEM_BUDGET - BAR_BYTES) / STAGE_BYTES;
  static constexpr int NST = NST_RAW > 8 ? 8 : NST_RAW;
  static constexpr int SMEM_BYTES = NST * STAGE_BYTES + BAR_BYTES;
  static_assert(MTR % EPI_ROWS == 0 && 3 * MTR == NB, "token tile");
  static_assert(NA * A_UNIT_COLS + NB <= TMEM_COLS, "TMEM budget");
  static_assert(NA >= 2 && NST >= 2, "pipeline too shallow");
  static_assert(NBR % 2 == 0 && NBR > 2 * (NST + NA), "barrier ring depth");
  static_assert(NST * STAGE_BYTES >= MTR * TILE_N * 4, "epilogue sums fit over the stages");
};

// One weight of a launch.  A launch covers the tiles of up to MMA_GROUP_MAX
// weights that share K and the activations (the q, k and v projections, or
// gate and up): global tile t belongs to the last weight whose tile_start <= t.
struct TcWeight {
  const uint8_t* nib;  // fragment layout
  const uint8_t* scl;
  float* y;            // [rows of this launch, N], or null (greedy pick)
  int64_t N;
  int tile_start;      // first global tile
};

struct TcArgs {
  TcWeight w[MMA_GROUP_MAX];
  int nweights;
  const uint8_t* xop;  // activation operand, [mtiles][KB2][64*NB] bytes
  int64_t KBP, KB2;    // block pairs, padded blocks (2 * KBP)
  int64_t kbp_per_split;
  int mtiles;
  int rs;              // 1: split-K by reduce-scatter (every CTA of the launch resident at once)
  unsigned int* status;
  unsigned long long wait_ns;  // bound of the waits between roles and CTAs
  int stall;           // test setting: the producer issues no copy, so every wait runs out
  EpiArgs e;
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
// try_wait with a suspend-time hint: a thread whose phase is not complete is
// parked (it stops competing for issue slots) until the phase completes or
// the hint elapses.
constexpr uint32_t SUSPEND_NS = 1000000u;  // 1 ms per try

__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(SUSPEND_NS)
      : "memory");
  return ok != 0;
}

// Bounded wait: false (and the CTA error flag raised) if the phase does not
// complete within limit_ns (WAIT_NS by default), or if another role already
// gave up.  The timer is read only after a try has expired, off the common
// path.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* err,
                                          unsigned long long limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  unsigned long long t0 = 0;
  for (;;) {
    if (mbar_try_wait_sleep(bar, parity)) return true;
    if (*err) return false;
    const unsigned long long now = globaltimer();
    if (t0 == 0) {
      t0 = now;
    } else if (now - t0 > limit_ns) {
      *err = 1;
      return false;
    }
  }
}

// Bounded wait used only while draining (no error flag to consult).
__device__ __forceinline__ void mbar_drain(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return;
  unsigned long long t0 = 0;
  for (;;) {
    if (mbar_try_wait_sleep(bar, parity)) return;
    const unsigned long long now = globaltimer();
    if (t0 == 0) {
      t0 = now;
    } else if (now - t0 > WAIT_NS) {
      return;
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

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, "
      "%29, %30, %31, %32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]),
      "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]),
      "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
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

// (q - 8) for the nibble pair at bits (4p, 16 + 4p) of w, as exact bf16x2:
// (w >> 4p) & 0x000F000F | 0x43004300 is bf16(128 + q), minus 136 is exact.
__device__ __forceinline__ uint32_t nib_pair_bf16(uint32_t w, int p) {
  uint32_t t, r;
  asm("lop3.b32 %0, %1, 0x000F000F, 0x43004300, 0xEA;" : "=r"(t) : "r"(w >> (4 * p)));
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(t), "r"(0x43084308u));
  return r;
}

// The two weights (q0 - 8) * d, (q1 - 8) * d of a bf16x2 (q - 8) pair as the
// exact sums hi + lo of two bf16x2 values (see the file comment).
__device__ __forceinline__ void scale_split(uint32_t qa, float d, uint32_t& hi, uint32_t& lo) {
  const float p0 = __uint_as_float(qa << 16) * d;            // exact in fp32
  const float p1 = __uint_as_float(qa & 0xFFFF0000u) * d;
  const __nv_bfloat162 h = __floats2bfloat162_rn(p0, p1);   // low half: p0
  hi = *reinterpret_cast<const uint32_t*>(&h);
  const __nv_bfloat162 l = __floats2bfloat162_rn(p0 - __low2float(h), p1 - __high2float(h));
  lo = *reinterpret_cast<const uint32_t*>(&l);               // remainders are exact in bf16
}

// ----------------------------------------------------------------------------
// Pre-pass: x[M, K] fp32 -> activation operand: three exact bf16 terms per
// value, laid out per (m tile, block) exactly as the MMA reads it from smem,
//   [k-step s (2)][k group g (2)][B row (NB)][8 k]   (16-byte rows)
// with B row t*MTR + m holding term t of token row m, and rows >= 3*MTR zero.
// One thread per (m tile, block, s, g, token row in tile).
// ----------------------------------------------------------------------------
template <int NB>
__global__ void __launch_bounds__(256) xop_kernel(const float* __restrict__ x, int64_t M, int64_t K,
                                                  int64_t KB, int mtiles, uint8_t* __restrict__ xop) {
  // KB here is the padded block count; blocks past the real K read as zero
  constexpr int MTR = NB / 3;
  asm volatile("griddepcontrol.launch_dependents;");
  const int64_t total = (int64_t)mtiles * KB * 4 * MTR;
  for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < total;
       t += (int64_t)gridDim.x * blockDim.x) {
    const int mm = (int)(t % MTR);
    const int sg = (int)((t / MTR) & 3);
    const int64_t b = (t / MTR / 4) % KB;
    const int64_t mt = t / MTR / 4 / KB;
    const int s = sg >> 1, g = sg & 1;
    const int64_t m = mt * MTR + mm;
    float v[8];
    if (m < M && b * BLOCK_K < K) {
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
    uint8_t* chunk = xop + (mt * KB + b) * (int64_t)(64 * NB) + (int64_t)(s * 2 + g) * NB * 16;
#pragma unroll
    for (int term = 0; term < 3; ++term)
      *reinterpret_cast<uint4*>(chunk + (term * MTR + mm) * 16) =
          make_uint4(out[term][0], out[term][1], out[term][2], out[term][3]);
    if (mm == 0) {
      for (int r = 3 * MTR; r < NB; ++r)
        *reinterpret_cast<uint4*>(chunk + r * 16) = make_uint4(0u, 0u, 0u, 0u);
    }
  }
}

// ----------------------------------------------------------------------------
// Main kernel
// ----------------------------------------------------------------------------
template <int NB>
__global__ void __launch_bounds__(TC_THREADS, 1) tc_kernel(const TcArgs a) {
  using C = Cfg<NB>;
  constexpr int MTR = C::MTR;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* stages = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::NST * C::STAGE_BYTES);
  uint64_t* full = bars;           // unit data landed in its smem stage (tx count)
  uint64_t* empty = full + NBR;    // stage consumed: 4 converter warps + MMA commit
  uint64_t* afull = empty + NBR;   // A terms written to TMEM: 4 converter warps
  uint64_t* afree = afull + NBR;   // MMAs of the unit done (A slot reusable): commit
  uint64_t* dfull = afree + NBR;   // every MMA of the CTA done: commit
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(dfull + 1);
  volatile int* err = reinterpret_cast<volatile int*>(tmem_slot + 2);
  __shared__ int s_last[2];
  __shared__ unsigned s_arrival;  // split-K arrival word of this CTA
  __shared__ unsigned long long red[2][4][EPI_ROWS];  // greedy-pick scratch of the epilogue

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int mt = blockIdx.x, gtile = blockIdx.y, split = blockIdx.z;
  int wi = 0;
#pragma unroll
  for (int i = 1; i < MMA_GROUP_MAX; ++i)
    if (i < a.nweights && gtile >= a.w[i].tile_start) wi = i;
  const int tile = gtile - a.w[wi].tile_start;  // tile within its weight
  const int64_t bp0 = (int64_t)split * a.kbp_per_split;
  const int64_t bp1 = min(a.KBP, bp0 + a.kbp_per_split);
  const int nblk = (int)(2 * (bp1 - bp0));  // includes the zero pad block of an odd count
  const int nunits = (nblk + U - 1) / U;
  const int64_t m0 = (int64_t)mt * MTR;
  const int mcount = (int)min((int64_t)MTR, a.e.M - m0);

  if (tid == 0) {
    for (int i = 0; i < NBR; ++i) {
      mbar_init(smem_u32(&full[i]), 1);
      mbar_init(smem_u32(&empty[i]), 4 + 1);
      mbar_init(smem_u32(&afull[i]), 4);
      mbar_init(smem_u32(&afree[i]), 1);
    }
    mbar_init(smem_u32(dfull), 1);
    *err = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == MMA_WARP) tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t a_base = tmem;                                      // A ring columns
  const uint32_t d_base = tmem + (uint32_t)(C::NA * C::A_UNIT_COLS);  // accumulator columns

  if (warp == PROD_WARP) {
    // ---------------- producer ----------------
    if (lane == 0) {
      int nunits_issue = nunits;
      asm volatile("griddepcontrol.wait;" ::: "memory");  // the activation operand of the pre-pass
      if (a.stall) nunits_issue = 0;  // (test setting) nothing arrives: every consumer's wait runs out
      const uint8_t* nib_base = a.w[wi].nib + ((int64_t)tile * a.KBP + bp0) * PAIR_NIB_BYTES;
      const uint8_t* scl_base = a.w[wi].scl + ((int64_t)tile * a.KBP + bp0) * PAIR_SCL_BYTES;
      const uint8_t* bop_base = a.xop + ((int64_t)mt * a.KB2 + 2 * bp0) * (int64_t)C::BOP_BLOCK;
      int last = -1;
      for (int u = 0; u < nunits_issue; ++u) {
        const int st = u % C::NST;
        const int ub = min(U, nblk - u * U);
        if (u >= C::NST) {  // stage reuse: unit u - NST must be consumed
          const int v = u - C::NST;
          if (!mbar_wait(smem_u32(&empty[v % NBR]), (v / NBR) & 1, err, a.wait_ns)) break;
        }
        const uint32_t sb = smem_u32(stages + st * C::STAGE_BYTES);
        const uint32_t fb = smem_u32(&full[u % NBR]);
        mbar_expect_tx(fb, (uint32_t)(ub * (TILE_N * 16 + TILE_N * 2 + C::BOP_BLOCK)));
        bulk_g2s(sb, nib_base + (int64_t)u * U * TILE_N * 16, ub * TILE_N * 16, fb);
        bulk_g2s(sb + C::SCL_OFF, scl_base + (int64_t)u * U * TILE_N * 2, ub * TILE_N * 2, fb);
        bulk_g2s(sb + C::BOP_OFF, bop_base + (int64_t)u * U * C::BOP_BLOCK, ub * C::BOP_BLOCK, fb);
        last = u;
      }
      // drain: every copy this producer issued has landed before the CTA exits
      for (int u = last; u >= 0 && u > last - C::NST; --u)
        mbar_drain(smem_u32(&full[u % NBR]), (u / NBR) & 1);
    }
  } else if (warp == MMA_WARP) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t IDESC = idesc_bf16(NB);
      uint32_t accumulate = 0;
      bool ok = true;
      for (int u = 0; u < nunits; ++u) {
        const int st = u % C::NST, sa = u % C::NA;
        const int ub = min(U, nblk - u * U);
        const int bi = u % NBR;
        const uint32_t par = (u / NBR) & 1;
        if (!mbar_wait(smem_u32(&full[bi]), par, err, a.wait_ns) ||
            !mbar_wait(smem_u32(&afull[bi]), par, err, a.wait_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t bop = smem_u32(stages + st * C::STAGE_BYTES + C::BOP_OFF);
        const uint32_t acol = a_base + (uint32_t)(sa * C::A_UNIT_COLS);
        for (int b = 0; b < ub; ++b) {
#pragma unroll
          for (int s = 0; s < 2; ++s) {
            const uint64_t bd = smem_desc(bop + (uint32_t)(b * C::BOP_BLOCK + s * 32 * NB), 16u * NB, 128u);
#pragma unroll
            for (int term = 0; term < 2; ++term) {
              mma_ts(d_base, acol + (uint32_t)(b * C::A_BLOCK_COLS + term * 16 + s * 8), bd, IDESC,
                     accumulate);
              accumulate = 1;
            }
          }
        }
        mma_commit(smem_u32(&afree[bi]));
        mma_commit(smem_u32(&empty[bi]));
      }
      mma_commit(smem_u32(dfull));  // arrives once every MMA issued above has completed
      mbar_drain(smem_u32(dfull), 0);
      (void)ok;
    }
    __syncwarp();
  } else {
    // ---------------- converters ----------------
    const int q = warp & 3, g = warp >> 2;
    const int row = q * 32 + lane;
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    // this row's place in the fragment layout
    const int frg = row >> 4, fup = (row >> 3) & 1, fg = row & 7;
    for (int u = g; u < nunits; u += 2) {
      const int st = u % C::NST, sa = u % C::NA;
      const int ub = min(U, nblk - u * U);
      const int bi = u % NBR;
      if (!__all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&full[bi]), (u / NBR) & 1, err, a.wait_ns))) break;
      const uint8_t* sp = stages + st * C::STAGE_BYTES;
      // Block b of the unit (pair b / 2, half b % 2): the row's 32 weights sit
      // in the words of lanes 4fg + tq (tq = 0..3), two k-steps each.
      uint2 v[U][4];
      float dsc[U];
#pragma unroll
      for (int b = 0; b < U; ++b) {
        const int bpl = b >> 1, h = b & 1;
        if (b < ub) {
#pragma unroll
          for (int tq = 0; tq < 4; ++tq)
            v[b][tq] = *reinterpret_cast<const uint2*>(
                sp + (((bpl * 8 + frg) * 32 + 4 * fg + tq) * 16) + h * 8);
          const uint16_t dh = *reinterpret_cast<const uint16_t*>(
              sp + C::SCL_OFF + ((bpl * 8 + frg) * 8 + fg) * 8 + (fup * 2 + h) * 2);
          dsc[b] = __half2float(__ushort_as_half(dh));
        } else {
#pragma unroll
          for (int tq = 0; tq < 4; ++tq) v[b][tq] = make_uint2(0x88888888u, 0x88888888u);
          dsc[b] = 0.0f;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&empty[bi]));
      if (u >= C::NA) {  // A slot reuse: the MMAs of unit u - NA must be done
        const int w = u - C::NA;
        if (!__all_sync(0xFFFFFFFFu, mbar_wait(smem_u32(&afree[w % NBR]), (w / NBR) & 1, err, a.wait_ns))) break;
      }
      const uint32_t acol = a_base + lane_off + (uint32_t)(sa * C::A_UNIT_COLS);
#pragma unroll
      for (int b = 0; b < U; ++b) {
        // TMEM column c of a term and k-step holds k = 2c, 2c + 1: the pair at
        // k0 = 16s + 2tq is column 8s + tq, the pair at k0 + 8 is 8s + 4 + tq
        uint32_t av[32];  // [term][k-step][8 columns]
#pragma unroll
        for (int tq = 0; tq < 4; ++tq) {
          const uint32_t ws[2] = {v[b][tq].x, v[b][tq].y};
#pragma unroll
          for (int s = 0; s < 2; ++s) {
            uint32_t hi, lo;
            scale_split(nib_pair_bf16(ws[s], fup), dsc[b], hi, lo);
            av[8 * s + tq] = hi;
            av[16 + 8 * s + tq] = lo;
            scale_split(nib_pair_bf16(ws[s], fup + 2), dsc[b], hi, lo);
            av[8 * s + 4 + tq] = hi;
            av[16 + 8 * s + 4 + tq] = lo;
          }
        }
        tmem_st32(acol + (uint32_t)(b * C::A_BLOCK_COLS), av);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&afull[bi]));
    }
  }

  // ---- epilogue: warps 0-7 read the accumulator once.  Warps w and w + 4
  // reach the same TMEM lanes (32 (w % 4) ...); quad q = w / 4 takes the
  // chunks of 16 token rows c = q, q + 2, ... ----
  tc_fence_before();
  __syncthreads();
  const bool skip = *err != 0;
  __syncthreads();  // every thread has read the flag before the epilogue can raise it
  if (warp < 8 && !skip) {
    const bool ok = mbar_wait(smem_u32(dfull), 0, err, a.wait_ns);
    // every epilogue thread takes the same decision
    uint32_t any_bad;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.eq.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, 1, 256, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(any_bad)
        : "r"((uint32_t)ok)
        : "memory");
    if (!any_bad) {
      tc_fence_after();
      const int quad = warp >> 2;
      const int row = (warp & 3) * 32 + lane;
      const uint32_t drow = d_base + ((uint32_t)((warp & 3) * 32) << 16);
      asm volatile("griddepcontrol.wait;" ::: "memory");  // outputs and scratch: after earlier kernels
      if (a.e.splits > 1 && !a.rs) {
        // last-CTA exchange: the arrival is drawn once the accumulator is
        // complete, so the CTA that draws last is the last to finish and its
        // peers' partial sums are already on their way
        if (warp == 0 && lane == 0) s_arrival = split_arrive(&a.e.counters[gtile * a.mtiles + mt]);
        asm volatile("bar.sync 2, 256;" ::: "memory");
      }
      const unsigned arrival = s_arrival;
      const int nchunk = (mcount + EPI_ROWS - 1) / EPI_ROWS;  // the same for every split
      if (a.rs) {
        // Reduce-scatter: CTA `split` owns tile rows [r0, r1) of every token
        // row.  Each CTA keeps all its sums in shared memory and stores the
        // other CTAs' rows to global memory (64-bit words with a zero high
        // half, which no flagged reader accepts); then the tile's CTAs meet at
        // a barrier on the tile's arrival word, and each adds up its own rows
        // over the splits in ascending order (the order of every other path).
        // All CTAs of the launch are resident together, so the barrier
        // completes; one thread per CTA polls the word, with back-off.
        float* xch = reinterpret_cast<float*>(stages);  // [MTR][TILE_N]; the stages are dead
        const int S = a.e.splits;
        const int r0 = split * TILE_N / S, r1 = (split + 1) * TILE_N / S;
        const int64_t sstride = a.e.M * a.e.N_pad;
        unsigned long long* part = a.e.partial + m0 * a.e.N_pad + (int64_t)gtile * TILE_N;
        const bool mine = row >= r0 && row < r1;
#pragma unroll 1
        for (int c = quad; c < nchunk; c += 2) {
          const int c0 = c * EPI_ROWS;
          float t0[16], t1[16], t2[16];
          tmem_ld16(drow + (uint32_t)c0, t0);
          tmem_ld16(drow + (uint32_t)(MTR + c0), t1);
          tmem_ld16(drow + (uint32_t)(2 * MTR + c0), t2);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < EPI_ROWS; ++j) {
            const int m = c0 + j;
            if (m < mcount) {
              const float v = (t0[j] + t1[j]) + t2[j];
              xch[m * TILE_N + row] = v;
              if (!mine)
                __stcg(part + (int64_t)split * sstride + (int64_t)m * a.e.N_pad + row,
                       (unsigned long long)__float_as_uint(v));
            }
          }
        }
        __threadfence();  // this CTA's stores before its arrival
        asm volatile("bar.sync 2, 256;" ::: "memory");
        const int et = warp * 32 + lane;  // 0..255
        if (et == 0) {
          unsigned* ctr = &a.e.counters[gtile * a.mtiles + mt];
          const unsigned w = split_arrive(ctr);
          if (arrival_last(w, S)) {
            __threadfence();  // every peer's stores are visible before the epoch moves on
            atomicExch(ctr, arrival_next(w));  // the others see the epoch move on
          } else {
            const unsigned ep = w >> ARRIVAL_BITS;
            unsigned long long t_start = 0;
            for (uint32_t n = 1;; ++n) {
              unsigned cur;
              asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(cur) : "l"(ctr) : "memory");
              if ((cur >> ARRIVAL_BITS) != ep) break;
              __nanosleep(100);
              if ((n & 63u) == 0u) {
                const unsigned long long now = globaltimer();
                if (t_start == 0) t_start = now;
                else if (now - t_start > a.wait_ns) {
                  atomicOr(a.e.status, STATUS_TIMEOUT);
                  break;
                }
              }
            }
          }
          __threadfence();
        }
        asm volatile("bar.sync 2, 256;" ::: "memory");  // every peer's rows are visible
        // own rows: OB outputs per thread at a time, every split of them read
        // before anything is added or stored
        const int rows = r1 - r0, outs = rows * mcount;
        constexpr int OB = 4, SB = 8;
        for (int ob = et; ob < outs; ob += 256 * OB) {
          float acc[OB];
#pragma unroll
          for (int q = 0; q < OB; ++q) acc[q] = 0.0f;
          for (int s0 = 0; s0 < S; s0 += SB) {
            float t[OB][SB];
#pragma unroll
            for (int q = 0; q < OB; ++q) {
              const int o = ob + 256 * q;
              const int m = o / rows, r = r0 + o % rows;
#pragma unroll
              for (int j = 0; j < SB; ++j) {
                const int sj = s0 + j;
                t[q][j] = 0.0f;
                if (o < outs && sj < S)
                  t[q][j] = sj == split ? xch[m * TILE_N + r]
                                        : __uint_as_float((uint32_t)__ldcg(
                                              part + (int64_t)sj * sstride + (int64_t)m * a.e.N_pad + r));
              }
            }
#pragma unroll
            for (int q = 0; q < OB; ++q)
#pragma unroll
              for (int j = 0; j < SB; ++j)
                if (s0 + j < S) acc[q] += t[q][j];
          }
#pragma unroll
          for (int q = 0; q < OB; ++q) {
            const int o = ob + 256 * q;
            const int64_t n = (int64_t)tile * TILE_N + r0 + o % rows;
            if (o < outs && n < a.w[wi].N) a.w[wi].y[(m0 + o / rows) * a.w[wi].N + n] = acc[q];
          }
        }
      } else {
        // this weight's outputs; partial sums and counters by the global tile
        EpiArgs e = a.e;
        e.y = a.w[wi].y;
        e.N = a.w[wi].N;
        e.partial = a.e.partial + (int64_t)a.w[wi].tile_start * TILE_N;
#pragma unroll 1
        for (int c = quad; c < nchunk; c += 2) {
          const int c0 = c * EPI_ROWS;
          float t0[16], t1[16], t2[16], val[EPI_ROWS];
          tmem_ld16(drow + (uint32_t)c0, t0);
          tmem_ld16(drow + (uint32_t)(MTR + c0), t1);
          tmem_ld16(drow + (uint32_t)(2 * MTR + c0), t2);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < EPI_ROWS; ++j) val[j] = (t0[j] + t1[j]) + t2[j];
          finish_tile<EPI_ROWS, 1, EPI_ROWS>(
              e, val, row, 0, tile, m0 + c0, min(EPI_ROWS, mcount - c0), split, arrival,
              c == 0 ? gtile * a.mtiles + mt : -1, &s_last[quad], red[quad],
              [quad]() { asm volatile("bar.sync %0, 128;" ::"r"(3 + quad) : "memory"); });
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
  if (*err != 0 && tid == 0) atomicOr(a.status, STATUS_TIMEOUT);
}

constexpr int64_t TC_M_LAUNCH = 256;  // rows per launch pair (pre-pass + main)

// MMA N (3 x token rows per CTA) for a launch of ml rows: as few token tiles
// as the largest N (80 rows) needs, each as small as that count allows.
// Forced with the batch-invariant flag: always NB = 96, independent of M.
// Batch-invariant mode: one token tile of 64 rows (B rows = 3 terms x 64) for
// every M.  Measured on GB300 (gate/up group + down of a 7B layer, 8 layers
// per graph, us per layer at M = 1 / 32 / 124; the default mode 27.5 / 109.5 /
// 250.3): 32-row tiles 105.3 / 109.5 / 402.5, 48 rows 106.1 / 110.1 / 318.9,
// 64 rows 123.3 / 128.1 / 250.1, 80 rows 166.8 / 170.8 / 347.1.
#ifndef Q4MM_TC_BI_NB
#define Q4MM_TC_BI_NB 192
#endif
int nb_for(int64_t ml, bool batch_invariant) {
  if (batch_invariant) return Q4MM_TC_BI_NB;
  const int64_t passes = (ml + 79) / 80;
  const int64_t r = (ml + passes - 1) / passes;
  if (r <= 16) return 48;
  if (r <= 32) return 96;
  if (r <= 48) return 144;
  if (r <= 64) return 192;
  return 240;
}

template <int NB>
int launch_nb(const MmaLaunch& L, const float* x, int64_t ml, int32_t* idx, float* maxval,
              const TcPlan& plan, const Workspace& ws, int64_t mb, cudaStream_t s) {
  using C = Cfg<NB>;
  const Weight* W = L.W[0];  // K, KBP and the device are the group's
  int64_t tiles = 0;
  for (int i = 0; i < L.count; ++i) tiles += L.W[i]->tiles;
  const int mtiles = (int)((ml + C::MTR - 1) / C::MTR);
  const int64_t KB2 = 2 * W->KBP;
  if (plan.splits > 1 && tiles * mtiles > MAX_COUNTERS) return Q4_ERR_SHAPE;
  {
    const int64_t total = (int64_t)mtiles * KB2 * 4 * C::MTR;
    const int64_t want = (total + 255) / 256;
    const int blocks = (int)(want < 4096 ? want : 4096);
    xop_kernel<NB><<<blocks, 256, 0, s>>>(x, ml, W->K, KB2, mtiles, static_cast<uint8_t*>(ws.xop));
    if (cudaGetLastError() != cudaSuccess) return Q4_ERR_CUDA;
  }
  static std::atomic<bool> attr_set[64];  // per device, once (setting it twice is harmless)
  if (!attr_set[W->device & 63].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(tc_kernel<NB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::SMEM_BYTES) != cudaSuccess)
      return Q4_ERR_CUDA;
    attr_set[W->device & 63].store(true, std::memory_order_release);
  }
  // greedy-pick completion count: one epilogue chunk per (tile, token chunk)
  int64_t chunks = 0;
  for (int mt = 0; mt < mtiles; ++mt) {
    const int64_t rows = ml - (int64_t)mt * C::MTR < C::MTR ? ml - (int64_t)mt * C::MTR : C::MTR;
    chunks += (rows + EPI_ROWS - 1) / EPI_ROWS;
  }
  TcArgs a;
  {
    int t0 = 0;
    for (int i = 0; i < MMA_GROUP_MAX; ++i) {
      if (i < L.count) {
        const Weight* Wi = L.W[i];
        a.w[i].nib = Wi->nib;
        a.w[i].scl = reinterpret_cast<const uint8_t*>(Wi->d);
        a.w[i].y = L.y[i] ? L.y[i] + mb * Wi->N : nullptr;
        a.w[i].N = Wi->N;
        a.w[i].tile_start = t0;
        t0 += (int)Wi->tiles;
      } else {
        a.w[i] = a.w[0];
        a.w[i].tile_start = 1 << 30;
      }
    }
  }
  a.nweights = L.count;
  a.xop = static_cast<const uint8_t*>(ws.xop);
  a.KBP = W->KBP;
  a.KB2 = KB2;
  a.kbp_per_split = plan.kbp_per_split;
  a.mtiles = mtiles;
  a.status = ws.status;
  a.wait_ns = wait_limit_ns();
  a.stall = stall_for_test();
  a.e.poll_limit = poll_rounds();
  a.e.stall = 0;
  a.e.N = W->N;
  a.e.N_pad = tiles * TILE_N;
  a.e.M = ml;
  a.e.y = a.w[0].y;
  a.e.idx = idx ? idx + mb : nullptr;
  a.e.maxval = (idx && maxval) ? maxval + mb : nullptr;
  a.e.splits = plan.splits;
  a.e.partial = ws.partial;
  a.e.counters = ws.counters;
  a.e.status = ws.status;
  a.e.keys = ws.keys + mb;
  a.e.argmax_done = ws.argmax_done;
  a.e.tiles = (int)(tiles * chunks);
  // reduce-scatter exchange when every CTA of the launch is resident at once
  // (one CTA per SM), otherwise (and for the greedy pick) the last CTA of a
  // tile adds up all its splits
  a.rs = plan.splits > 1 && idx == nullptr && mtiles * tiles * plan.splits <= plan.num_sms;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)mtiles, (unsigned)tiles, (unsigned)plan.splits);
  cfg.blockDim = dim3(TC_THREADS);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, tc_kernel<NB>, a) != cudaSuccess) return Q4_ERR_CUDA;
  return Q4_OK;
}

}  // namespace

bool tc_kernel_built() { return true; }

TcPlan tc_plan_tiles(int64_t wtiles, int64_t KBP, int64_t M, int num_sms, bool batch_invariant) {
  TcPlan p;
  p.num_sms = num_sms;
  const int64_t ml = M < TC_M_LAUNCH ? M : TC_M_LAUNCH;
  p.m_tile = nb_for(ml, batch_invariant);
  const int64_t mtiles = (ml + p.m_tile / 3 - 1) / (p.m_tile / 3);
  // K partition: fill the SMs, balancing waves against units per CTA (+ a
  // fixed per-CTA cost in unit terms).  It depends on M through the token
  // tiles, except in batch-invariant mode (one token tile assumed).
  const int64_t tiles = wtiles * (batch_invariant ? 1 : mtiles);
  // at least 16 blocks (four units) per split: the split-K epilogue runs once
  // per 16 token rows of every CTA, so very short K ranges cost more than
  // they save
  int64_t best_s = 1, best_cost = -1;
  int64_t smax = KBP / 8;
  if (smax < 1) smax = 1;
  if (smax > 64) smax = 64;
  for (int64_t s = 1; s <= smax; ++s) {
    const int64_t kbps = (KBP + s - 1) / s;  // block pairs per split
    const int64_t waves = (tiles * s + num_sms - 1) / num_sms;
    const int64_t cost = waves * ((2 * kbps + U - 1) / U + 6);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best_s = s;
    }
  }
  p.kbp_per_split = (KBP + best_s - 1) / best_s;
  p.splits = (int)((KBP + p.kbp_per_split - 1) / p.kbp_per_split);
  return p;
}

TcPlan tc_plan(const Weight* W, int64_t M, int num_sms, bool batch_invariant) {
  return tc_plan_tiles(W->tiles, W->KBP, M, num_sms, batch_invariant);
}

size_t tc_partial_bytes_tiles(int64_t tiles, const TcPlan& p, int64_t M) {
  if (p.splits <= 1) return 0;
  const int64_t ml = M < TC_M_LAUNCH ? M : TC_M_LAUNCH;
  return (size_t)p.splits * (size_t)ml * (size_t)(tiles * TILE_N) * sizeof(unsigned long long);
}

size_t tc_partial_bytes(const Weight* W, const TcPlan& p, int64_t M) {
  return tc_partial_bytes_tiles(W->tiles, p, M);
}

size_t tc_xop_bytes_kbp(int64_t KBP, const TcPlan& p, int64_t M) {
  const int64_t ml = M < TC_M_LAUNCH ? M : TC_M_LAUNCH;
  const int64_t mtr = p.m_tile / 3;
  const int64_t mtiles = (ml + mtr - 1) / mtr;
  return (size_t)mtiles * (size_t)(2 * KBP) * 64u * (size_t)p.m_tile;
}

size_t tc_xop_bytes(const Weight* W, const TcPlan& p, int64_t M) { return tc_xop_bytes_kbp(W->KBP, p, M); }

int64_t tc_rows_per_launch() { return TC_M_LAUNCH; }

int tc_launch_count(const TcPlan&, int64_t M) {
  return 2 * (int)((M + TC_M_LAUNCH - 1) / TC_M_LAUNCH);
}

int launch_tc_group(const MmaLaunch& L, const float* x, int64_t M, int32_t* idx, float* maxval,
                    const TcPlan& plan, const Workspace& ws, cudaStream_t s) {
  const int64_t K = L.W[0]->K;
  for (int64_t mb = 0; mb < M; mb += TC_M_LAUNCH) {
    const int64_t ml = (M - mb) < TC_M_LAUNCH ? (M - mb) : TC_M_LAUNCH;
    const float* xs = x + mb * K;
    int st;
    switch (plan.m_tile) {
      case 48: st = launch_nb<48>(L, xs, ml, idx, maxval, plan, ws, mb, s); break;
      case 96: st = launch_nb<96>(L, xs, ml, idx, maxval, plan, ws, mb, s); break;
      case 144: st = launch_nb<144>(L, xs, ml, idx, maxval, plan, ws, mb, s); break;
      case 192: st = launch_nb<192>(L, xs, ml, idx, maxval, plan, ws, mb, s); break;
      default: st = launch_nb<240>(L, xs, ml, idx, maxval, plan, ws, mb, s); break;
    }
    if (st) return st;
  }
  return Q4_OK;
}

int launch_tc(const Weight* W, const float* x, int64_t M, float* y, int32_t* idx, float* maxval,
              const TcPlan& plan, const Workspace& ws, cudaStream_t s) {
  MmaLaunch L;
  L.count = 1;
  L.W[0] = W;
  L.y[0] = y;
  return launch_tc_group(L, x, M, idx, maxval, plan, ws, s);
}

}  // namespace q4
