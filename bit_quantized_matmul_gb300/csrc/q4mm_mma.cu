// q4mm_mma.cu — streaming tensor-core kernel for small M (the decode path).
//
// This is the linear layer of a decode step: M token rows (1 to 16 per launch)
// times a Q4_0 weight matrix read from HBM exactly once per call ("Why LLM
// Decoding Is Slow, and Why Batching Is (Almost) Free", §3-§4: decode streams
// every weight once per step, and the extra token rows of a batch ride along
// almost for free while the step stays memory-bound).  It replaces the two
// kernels of "Why Continuous Batching Slowed Down My LLM Inference Engine"
// (§"Two Rows of Input, Two Different Kernels") — a one-row GEMV and a tiled
// GEMM — with one kernel whose cost per weight hardly changes between 1 and
// 16 rows, so no row count needs a different kernel or a per-row relaunch.
//
// CTA = one 128-row tile over a K range (block pairs [bp0, bp1)); 640 threads:
//
//   16 compute warps  warp w takes row groups 2(w&3), 2(w&3)+1 (32 rows) and
//                     K slice w>>2: block pairs bp0 + slice + 4i (with four
//                     to six column groups, 9 to 16 rows: row group w&7 and
//                     K slice (w>>3)&1, block pairs bp0 + slice + 2i).  Its lanes
//                     copy their 16-byte weight fragments (coalesced, 1 KB per
//                     warp and pair) and lanes 0..7 the pair's 128 bytes of
//                     fp16 scales (512 and 64 bytes with one row group per
//                     warp) from HBM into the warp's private cp.async
//                     ring, two pairs ahead; each lane reads back its own
//                     fragments, which in the fragment layout are exactly the
//                     A registers of m16n8k16 MMAs once unpacked to exact bf16
//                     (q - 8).  The first pairs are on their way before the
//                     kernel waits for the previous one on the stream (weights
//                     never depend on it).  No CTA barrier in the loop.
//   4 converter warps stage, per chunk of 8 block pairs, the activations as
//                     exact three-term bf16 B fragments (x = x0 + x1 + x2,
//                     term t of row m in MMA column 3m + t, or column t of the
//                     row's own column group in batch-invariant mode) into a
//                     4-slot (2-slot from four column groups) shared-memory
//                     ring with full/empty mbarriers
//                     (every wait bounded).  The fp32 rows arrive by cp.async
//                     four or five chunks ahead (two from four column groups).
//
// Launches of more tiles than SMs with one K split (the gate/up group of a 7B
// layer: 296 tiles) and one or two column groups run as two-tile CTAs: a CTA
// streams tiles 2b and 2b + 1 over the whole K, its warps covering the same
// row groups of both and its converted activations serving both, so the
// launch is one wave instead of two.
//
// Short-K launches whose tiles x 4 fit on the SMs (the q/k/v group and o_proj
// of a 7B layer) run as row-group CTAs instead: a CTA takes one row-group pair
// (32 rows) of a tile over the whole K, and its 16 compute warps are 16 K
// slices.  Its K reduction is then a shared-memory sum; no partial sums cross
// CTAs, whose exchange costs 1-2 us in the tail of every split launch.
//
// Per block the two MMAs accumulate D_b = sum_{k in b} (q-8) x_t in fresh
// fp32 registers; the block's fp16 scale is applied on the CUDA cores,
// acc = fma(d, D_b, acc), in ascending block order.  At the end the four (or
// two) K slices and the three terms of each row are added in a fixed order,
// then the K splits in ascending split order (q4mm_epilogue.cuh).  In
// batch-invariant mode nothing in that order depends on M; in the default
// mode the launch's row count picks the CTA layout (row-group or two-tile CTAs
// up to 8 rows, two K slices from 9), so a row's bits may differ with M
// within the tolerance.
#include <cuda_fp16.h>

#include <atomic>

#include "q4mm_epilogue.cuh"
#include "q4mm_internal.h"

namespace q4 {
namespace {

constexpr int MAX_CG = 3;          // column groups per launch with one row per group
constexpr int MAX_CG_DENSE = 6;    // column groups per launch with dense packing (48 MMA columns)
constexpr int SLICES = 4;          // K slices per CTA
constexpr int COMPUTE_WARPS = 16;  // 4 row-group pairs x 4 slices
constexpr int CONV_WARPS = 4;
constexpr int COMPUTE_THREADS = COMPUTE_WARPS * 32;
constexpr int CONV_THREADS = CONV_WARPS * 32;
constexpr int KERNEL_THREADS = COMPUTE_THREADS + CONV_THREADS;
constexpr int CHUNK_PAIRS = 8;              // block pairs per ring slot (512 k)
constexpr int CHUNK_K = CHUNK_PAIRS * 64;
// Block pairs in flight per compute warp (its private cp.async ring) and the
// unroll of its pair loop.  Measured on GB300 over the 7B decoder layers at
// M = 1..8: a ring of two pairs with the loop unrolled twice (slot indices and
// the once-per-chunk barrier steps become compile-time constants) beat rings
// of 3, 4 and 8 pairs, four-fold unrolling and loading the next pair early.
#ifndef Q4MM_WD
#define Q4MM_WD 2
#endif
#ifndef Q4MM_UNROLL
#define Q4MM_UNROLL 2
#endif
// largest K split whose CTAs exchange partial sums through a thread-block
// cluster (distributed shared memory) instead of global memory
#ifndef Q4MM_CLUSTER_MAX
#define Q4MM_CLUSTER_MAX 4
#endif
// row-group CTAs (one 32-row group pair over the whole K, no K split) for
// launches whose tiles x 4 fit on the SMs and whose K is at most this
#ifndef Q4MM_RG_MAX_K
#define Q4MM_RG_MAX_K 4096
#endif
#ifndef Q4MM_TWO_TILES
#define Q4MM_TWO_TILES 1
#endif
constexpr int RG_LD = 36;  // row stride of the row-group slice sums (32 rows + 4)
constexpr int T2_LD = 2 * TILE_N + 4;  // row stride of the two-tile slice sums (256 rows + 4)
// row stride of the slice sums in shared memory: 4 (mod 32 banks), so that
// the accumulator stores of a warp (lanes 4g + tq at column 2tq, row g) hit
// 32 different banks and the per-row reads stay consecutive
constexpr int RED_LD = TILE_N + 4;

// One weight of a launch.  A launch covers the tiles of up to MMA_GROUP_MAX
// weights that share K and the activations (e.g. the q, k and v projections):
// global tile t belongs to the last weight whose tile_start <= t.
struct MmaWeight {
  const uint4* nib;     // fragment layout, 16 bytes per (tile, pair, rg, lane)
  const uint8_t* scl;   // scale plane, 512 bytes per (tile, pair)
  float* y;             // [mrows, N] rows of this launch, or null (greedy pick)
  int64_t N;
  int tile_start;       // first global tile
};

struct MmaArgs {
  MmaWeight w[MMA_GROUP_MAX];
  int nweights;
  const float* x;       // [mrows, K] activations of this launch, or the whole x with xrows
  const int32_t* xrows; // null, or token row m of this launch is row xrows[m] of x
  int64_t x_rows;       // rows of x when xrows is given (indices are checked)
  int64_t K, KBP;       // K, block pairs
  int mrows;            // token rows in this launch
  int64_t kbp_per_split;
  unsigned int* status; // device status word (bounded-wait expiry)
  int cluster;          // 1: the K splits of a tile are one thread-block cluster
  EpiArgs e;
};

template <int C, int TPC = 1, bool DENSE = true, bool RG = false>
struct MmaCfg {
  static constexpr int MAXM = (C * 8) / 3 > C ? (C * 8) / 3 : C;  // rows per launch
  // four to six column groups (9 to 16 token rows, dense): one row group per
  // compute warp, 8 row groups x 2 K slices, so that the accumulators of six
  // groups fit; a two-slot B ring and three x stages, so that the larger
  // fragments fit in shared memory
  // (measured on GB300: three column groups are faster with two row groups
  // per warp, and batch-invariant launches keep one layout for every C)
  static constexpr bool R1 = DENSE && !RG && TPC == 1 && C >= 4;
  static constexpr int NSL = R1 ? 2 : SLICES;  // K slices of a tile's CTA
  static constexpr int NRG = R1 ? 1 : 2;       // row groups per compute warp
  static constexpr int NSLOT = R1 ? 2 : 4;     // B ring depth (a power of two)
  static constexpr int BF_PAIR = C * 1024;  // B fragments of a pair: [cg][h][32 slots] x 16 B
  static constexpr int SLOT = CHUNK_PAIRS * BF_PAIR;
  static constexpr int RING = NSLOT * SLOT;
  // converter staging: per slot the chunk's raw fp32 x rows
  static constexpr int XSTAGES = R1 ? 3 : (C == 3 ? 5 : 6);  // chunks of x in flight + the one converted
  static constexpr int XSLOT = MAXM * CHUNK_K * 4;
  static constexpr int XRAW_OFF = RING;
  static constexpr int RED = NSL * C * 8 * RED_LD * 4;  // per-slice sums for the gather
  static constexpr int XCH_OFF = (RED + 15) / 16 * 16;  // cluster split-K: this CTA's sums
  static constexpr int XCH = MAXM * TILE_N * 4;           // [token row][tile row] fp32
  // weight pairs in flight per compute warp: a private ring of WD slots, each
  // the warp's 16-byte fragments of its two row groups (1 KB) and their fp16
  // scales (128 B), filled by cp.async (half of that with one row group)
  static constexpr int WD = Q4MM_WD;
  static constexpr int WSLOT = NRG * (512 + 64);
  static constexpr int WSCL = NRG * 512;  // offset of the scales in a slot
  static constexpr int WR_OFF = RING + XSTAGES * XSLOT;
  static constexpr int WR = COMPUTE_WARPS * WD * WSLOT * TPC;
  static constexpr int BAR_OFF = WR_OFF + WR > XCH_OFF + XCH ? WR_OFF + WR : XCH_OFF + XCH;
  static constexpr int BYTES = BAR_OFF + 2 * NSLOT * 8;
  static_assert(!R1 || TPC == 1, "one row group per warp: one tile per CTA");
  static_assert(BYTES <= 227 * 1024, "shared memory of one CTA");
};

// bf16 pair (q - 8) for nibble pair p of word w: 0x4300 | q is bf16(128 + q),
// and one bf16x2 subtraction of 136 is exact.
__device__ __forceinline__ uint32_t nib_pair(uint32_t w, int p) {
  uint32_t t, r;
  // (w >> 4p) & 0x000F000F | 0x43004300 as one three-input logic op
  asm("lop3.b32 %0, %1, 0x000F000F, 0x43004300, 0xEA;" : "=r"(t) : "r"(w >> (4 * p)));
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(t), "r"(0x43084308u));
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

// Two fp32 accumulators in one 64-bit register pair: acc += s * (c0, c1), one
// packed instruction, each half an ordinary fp32 fma.  `ss` holds {s, s}.
__device__ __forceinline__ unsigned long long dup2(float s) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %1};" : "=l"(r) : "f"(s));
  return r;
}
__device__ __forceinline__ void ffma2(unsigned long long& acc, unsigned long long ss, float c0,
                                      float c1) {
  asm("{\n\t.reg .b64 rc;\n\t"
      "mov.b64 rc, {%2, %3};\n\t"
      "fma.rn.f32x2 %0, %1, rc, %0;\n\t}"
      : "+l"(acc)
      : "l"(ss), "f"(c0), "f"(c1));
}
__device__ __forceinline__ float2 split2(unsigned long long v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// Thread-block cluster: barrier over every thread of every CTA of the cluster
// (all of them are resident together), and reads of another CTA's shared
// memory through the cluster window.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_map(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
__device__ __forceinline__ float ld_cluster(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
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
// Bounded wait (1 s, or until another thread of the CTA reported an expiry);
// returns false on expiry.  The timer is read only after many polls.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  const volatile int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  unsigned long long t0 = 0;
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 255u) == 0u) {
      if (*err) return false;
      const unsigned long long now = globaltimer();
      if (t0 == 0) t0 = now;
      else if (now - t0 > 1000000000ull) return false;
    }
  }
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
// Exact three-term bf16 split of two consecutive activations: term 0 is the
// top 16 bits of x (truncation), term 1 the top 16 bits of the exact
// remainder, term 2 the rest (at most 8 significant bits, exact in bf16).
// Each term packs (k, k + 1) as a bf16x2 word, k in the low half.
__device__ __forceinline__ void split3(float x0, float x1, uint32_t& t0, uint32_t& t1,
                                       uint32_t& t2) {
  uint32_t u0 = __float_as_uint(x0), u1 = __float_as_uint(x1);
  t0 = __byte_perm(u0, u1, 0x7632);
  float r0 = x0 - __uint_as_float(u0 & 0xFFFF0000u);
  float r1 = x1 - __uint_as_float(u1 & 0xFFFF0000u);
  u0 = __float_as_uint(r0);
  u1 = __float_as_uint(r1);
  t1 = __byte_perm(u0, u1, 0x7632);
  r0 -= __uint_as_float(u0 & 0xFFFF0000u);
  r1 -= __uint_as_float(u1 & 0xFFFF0000u);
  t2 = __byte_perm(__float_as_uint(r0), __float_as_uint(r1), 0x7632);
}

// ----------------------------------------------------------------------------
// Shared-memory B fragments of one block pair: [cg][h][32 slots] x 16 bytes,
// slot of lane L = 4g + tq at L ^ sw with sw = 4 (pair & 1) + h, so that the
// converters' scattered 4-byte stores hit 32 distinct banks (a compute warp
// reads its 512 contiguous bytes conflict-free in any slot order).  The slot
// holds {b0, b1} of k-step 0 and {b0, b1} of k-step 1 for column g.
// ----------------------------------------------------------------------------
template <int C, bool DENSE, bool RG, int TPC>
__global__ void __launch_bounds__(KERNEL_THREADS, 1) mma_kernel(const MmaArgs a) {
  using S = MmaCfg<C, TPC, DENSE, RG>;
  constexpr int MAXM = S::MAXM;
  constexpr int WD = S::WD;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ unsigned long long kred[4][MAXM];
  __shared__ int s_flag;
  __shared__ unsigned s_arrival;  // split-K arrival word of this CTA
  __shared__ volatile int s_err;

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  // RG: the CTA is row-group pair blockIdx.x & 3 of global tile blockIdx.x >> 2
  // over the whole K, and its 16 compute warps are 16 K slices; otherwise the
  // CTA is global tile blockIdx.x over K split blockIdx.y, its compute warps
  // 4 row-group pairs x 4 K slices (8 row groups x 2 K slices with four to
  // six column groups)
  // TPC = 2: the CTA takes global tiles 2 blockIdx.x and 2 blockIdx.x + 1 (the
  // second when it exists) over the whole K; its warps cover the same row
  // groups of both, and the converted activations serve both
  const int gtile = RG ? (int)(blockIdx.x >> 2) : (int)blockIdx.x * TPC;
  int wi = 0;
#pragma unroll
  for (int i = 1; i < MMA_GROUP_MAX; ++i)
    if (i < a.nweights && gtile >= a.w[i].tile_start) wi = i;
  const int64_t tile = (int64_t)gtile - a.w[wi].tile_start;  // tile within its weight
  const bool has1 = TPC == 2 && (int64_t)gtile + 1 < a.e.N_pad / TILE_N;  // second tile
  int wi1 = wi;
#pragma unroll
  for (int i = 1; i < MMA_GROUP_MAX; ++i)
    if (i < a.nweights && gtile + 1 >= a.w[i].tile_start) wi1 = i;
  const int64_t tile1 = (int64_t)gtile + 1 - a.w[wi1].tile_start;
  const uint4* nib_w = a.w[wi].nib;
  const uint8_t* scl_w = a.w[wi].scl;
  const int split = blockIdx.y;
  const int64_t bp0 = (int64_t)split * a.kbp_per_split;
  const int64_t bp1 = min(a.KBP, bp0 + a.kbp_per_split);
  const int npairs = (int)(bp1 - bp0);
  const int nchunks = (npairs + CHUNK_PAIRS - 1) / CHUNK_PAIRS;
  const int mrows = a.mrows;
  uint64_t* bfull = reinterpret_cast<uint64_t*>(smem + S::BAR_OFF);
  constexpr int NSLOT = S::NSLOT;
  constexpr bool R1 = S::R1;
  constexpr int NRG = S::NRG;
  uint64_t* bempty = bfull + NSLOT;
  const bool compute = warp < COMPUTE_WARPS;

  // the next kernel on the stream may be scheduled now: its CTAs take the SMs
  // this launch leaves idle or gives back and start their own weight stream
  // (weights never depend on an earlier kernel) while this one finishes
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // compute warps: first weight loads before anything else (weights never
  // depend on an earlier kernel)
  constexpr int NSL = RG ? COMPUTE_WARPS : S::NSL;  // K slices
  const int rgp = RG ? (int)(blockIdx.x & 3) : (warp & 3);
  const int sl = RG ? (warp & (COMPUTE_WARPS - 1)) : (R1 ? ((warp >> 3) & 1) : ((warp >> 2) & 3));
  const int rg0 = R1 ? (warp & 7) : 2 * rgp;  // first row group of this warp
  const int n_i = (compute && npairs > sl) ? (npairs - sl + NSL - 1) / NSL : 0;
  const uint4* wp = nib_w + ((tile * a.KBP + bp0 + sl) * 8 + rg0) * 32 + lane;
  const uint4* wp1 = a.w[wi1].nib + ((tile1 * a.KBP + bp0 + sl) * 8 + rg0) * 32 + lane;
  constexpr int64_t WSTEP = NSL * 8 * 32;  // uint4 between a slice's consecutive pairs
  // ring slot j of this warp: [row groups rg0 .. rg0 + NRG - 1][lane][16 B] of
  // nibbles, then the 64 scale bytes of each row group ([rg][g][4 x fp16])
  // (with two tiles per CTA a slot holds the first tile's 1152 bytes, then the second's)
  const uint32_t wring = smem_u32(smem + S::WR_OFF + warp * (WD * S::WSLOT * TPC));
  const uint8_t* sp = scl_w + (tile * a.KBP + bp0 + sl) * PAIR_SCL_BYTES + rg0 * 64 + lane * 16;
  const uint8_t* sp1 = a.w[wi1].scl + (tile1 * a.KBP + bp0 + sl) * PAIR_SCL_BYTES + rg0 * 64 + lane * 16;
  constexpr int64_t SSTEP = NSL * PAIR_SCL_BYTES;  // scale bytes between a slice's pairs
  auto fetch = [&](int i) {  // pair i of this warp's K slice into slot i % WD
    if (i < n_i) {
      const uint32_t d = wring + (uint32_t)(i % WD) * (S::WSLOT * TPC);
      cp_async16(d + lane * 16, wp + (int64_t)i * WSTEP);
      if (NRG == 2) cp_async16(d + 512u + lane * 16, wp + (int64_t)i * WSTEP + 32);
      if (lane < 4 * NRG) cp_async16(d + S::WSCL + lane * 16, sp + (int64_t)i * SSTEP);
      if (TPC == 2 && has1) {
        cp_async16(d + S::WSLOT + lane * 16, wp1 + (int64_t)i * WSTEP);
        cp_async16(d + S::WSLOT + 512u + lane * 16, wp1 + (int64_t)i * WSTEP + 32);
        if (lane < 8) cp_async16(d + S::WSLOT + 1024u + lane * 16, sp1 + (int64_t)i * SSTEP);
      }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");  // one group per pair, empty or not
  };
  if (compute) {
#pragma unroll
    for (int u = 0; u < WD; ++u) fetch(u);
  }

  // zero the B-fragment columns no converter writes: the last column group
  // (dense packing with 3 * mrows < 8C) or every group (one row per group)
  {
    const bool part = DENSE ? (3 * mrows < 8 * C) : true;
    if (part) {
      constexpr int PER_SLOT = DENSE ? CHUNK_PAIRS * 2 * 32 : CHUNK_PAIRS * C * 2 * 32;  // uint4
      for (int j = tid; j < NSLOT * PER_SLOT; j += KERNEL_THREADS) {
        const int slot = j / PER_SLOT, r = j % PER_SLOT;
        int off;
        if (DENSE) {
          const int pc = r >> 6, h = (r >> 5) & 1, q = r & 31;
          off = ((pc * C + (C - 1)) * 2 + h) * 512 + q * 16;
        } else {
          off = r * 16;
        }
        *reinterpret_cast<uint4*>(smem + slot * S::SLOT + off) = make_uint4(0u, 0u, 0u, 0u);
      }
    }
  }
  if (tid == 0) {
    for (int b = 0; b < NSLOT; ++b) {
      mbar_init(smem_u32(&bfull[b]), CONV_THREADS);
      // a chunk's 8 pairs go to all 16 compute warps (two each, or four
      // with one row group per warp), or with row-group CTAs to the 8 warps
      // whose slices hold them (one each)
      mbar_init(smem_u32(&bempty[b]), RG ? COMPUTE_WARPS / 2 : COMPUTE_WARPS);
    }
    s_err = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  // accumulators: [rg][cg][row R0 / R1] as {column 2tq, column 2tq + 1} pairs
  // (packed fp32x2 updates) up to two column groups; as four floats [rg][cg][e]
  // for three, where the extra registers of the packed form would spill
  // (packed with one row group per warp for four and five groups; six spill,
  // measured slower)
  constexpr bool PACKED = C <= 2 || (R1 && C <= 5);
  static_assert(!(R1 && RG), "row-group CTAs have two row groups per warp");
  unsigned long long acc[TPC][NRG][C][2];
  float accf[TPC][NRG][C][4];
#pragma unroll
  for (int tt = 0; tt < TPC; ++tt)
#pragma unroll
    for (int r = 0; r < NRG; ++r)
#pragma unroll
      for (int cg = 0; cg < C; ++cg) {
        acc[tt][r][cg][0] = acc[tt][r][cg][1] = 0ull;
#pragma unroll
        for (int e = 0; e < 4; ++e) accf[tt][r][cg][e] = 0.0f;
      }

  if (compute) {
    const int g = lane >> 2;
    const int lsw0 = (lane ^ ((sl & 1) * 4)) * 16;        // slot of this lane, h = 0
    const int lsw1 = (lane ^ ((sl & 1) * 4 + 1)) * 16;    // h = 1
    // the 16-byte words and scales of pair i of this warp, once they are in
    // (this lane's groups complete in order, WD - 1 may still fly; the warp
    // barrier makes lanes 0..7's scale copies visible to all lanes)
    auto load_pair = [&](int i, int tt, uint4& a0, uint4& a1, uint2& s0, uint2& s1) {
      if (tt == 0) {
        asm volatile("cp.async.wait_group %0;" ::"n"(WD - 1) : "memory");
        __syncwarp();
      }
      const uint32_t src = wring + (uint32_t)(i % WD) * (S::WSLOT * TPC) + (uint32_t)(tt * S::WSLOT);
      asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(a0.x), "=r"(a0.y), "=r"(a0.z), "=r"(a0.w) : "r"(src + lane * 16) : "memory");
      asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(a1.x), "=r"(a1.y), "=r"(a1.z), "=r"(a1.w) : "r"(src + 512u + lane * 16) : "memory");
      asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(s0.x), "=r"(s0.y) : "r"(src + 1024u + g * 8) : "memory");
      asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(s1.x), "=r"(s1.y) : "r"(src + 1088u + g * 8) : "memory");
    };
    // the same with one row group per warp
    auto load_pair1 = [&](int i, uint4& a0, uint2& s0) {
      asm volatile("cp.async.wait_group %0;" ::"n"(WD - 1) : "memory");
      __syncwarp();
      const uint32_t src = wring + (uint32_t)(i % WD) * S::WSLOT;
      asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(a0.x), "=r"(a0.y), "=r"(a0.z), "=r"(a0.w) : "r"(src + lane * 16) : "memory");
      asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(s0.x), "=r"(s0.y) : "r"(src + S::WSCL + g * 8) : "memory");
    };
    {
#if Q4MM_UNROLL == 2
#pragma unroll 2
#elif Q4MM_UNROLL == 4
#pragma unroll 4
#endif
      for (int i = 0; i < n_i; ++i) {
        // chunk of this pair: slice sl's pairs are sl + NSL i
        const int c = RG ? 2 * i + (sl >> 3) : (R1 ? (i >> 2) : (i >> 1));
        const int slot = c & (NSLOT - 1);
        if ((RG || (R1 ? (i & 3) == 0 : (i & 1) == 0)) &&
            !mbar_wait_bounded(smem_u32(&bfull[slot]), (uint32_t)((c / NSLOT) & 1), &s_err)) {
          s_err = 1;
          goto compute_done;
        }
        const int pc = RG ? (sl & 7) : (R1 ? sl + 2 * (i & 3) : sl + 4 * (i & 1));  // pair within the chunk
        const uint8_t* sb = smem + slot * S::SLOT;
        if constexpr (R1) {
          // one row group: A fragments of its two k-steps per block, C column
          // groups of MMAs, the block scale on the CUDA cores as below
          uint4 w0;
          uint2 sv0;  // .x = d(R0, b0), d(R0, b1); .y = d(R1, b0), d(R1, b1)
          load_pair1(i, w0, sv0);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t a0[4], a1[4];  // [k-step]
            const uint32_t x0 = h ? w0.z : w0.x, x1 = h ? w0.w : w0.y;
#pragma unroll
            for (int p = 0; p < 4; ++p) {
              a0[p] = nib_pair(x0, p);
              a1[p] = nib_pair(x1, p);
            }
            if (h == 1) {  // every lane has unpacked both its words: refill the slot
              __syncwarp();
              fetch(i + WD);
            }
            const __half2* q0 = reinterpret_cast<const __half2*>(&sv0);
            const float f0 = h ? __high2float(q0[0]) : __low2float(q0[0]);
            const float f1 = h ? __high2float(q0[1]) : __low2float(q0[1]);
            unsigned long long s0 = 0, s1 = 0;
            if constexpr (PACKED) {
              s0 = dup2(f0);
              s1 = dup2(f1);
            }
            const uint8_t* bb = sb + (pc * C * 2 + h) * 512 + (h ? lsw1 : lsw0);
#pragma unroll
            for (int cg = 0; cg < C; ++cg) {
              const uint4 bf = *reinterpret_cast<const uint4*>(bb + cg * 1024);
              float d[4];
              mma_bf16_first(d, a0, bf.x, bf.y);
              mma_bf16_acc(d, a1, bf.z, bf.w);
              if constexpr (PACKED) {
                ffma2(acc[0][0][cg][0], s0, d[0], d[1]);
                ffma2(acc[0][0][cg][1], s1, d[2], d[3]);
              } else {
                accf[0][0][cg][0] = fmaf(f0, d[0], accf[0][0][cg][0]);
                accf[0][0][cg][1] = fmaf(f0, d[1], accf[0][0][cg][1]);
                accf[0][0][cg][2] = fmaf(f1, d[2], accf[0][0][cg][2]);
                accf[0][0][cg][3] = fmaf(f1, d[3], accf[0][0][cg][3]);
              }
            }
          }
        } else {
#pragma unroll
        for (int tt = 0; tt < TPC; ++tt) {
        if (tt == 1 && !has1) break;  // the same for every thread of the CTA
        uint4 w0, w1;
        uint2 sv0, sv1;  // .x = d(R0, b0), d(R0, b1); .y = d(R1, b0), d(R1, b1)
        load_pair(i, tt, w0, w1, sv0, sv1);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t a00[4], a01[4], a10[4], a11[4];  // [rg][k-step]
          const uint32_t x0 = h ? w0.z : w0.x, x1 = h ? w0.w : w0.y;
          const uint32_t y0 = h ? w1.z : w1.x, y1 = h ? w1.w : w1.y;
#pragma unroll
          for (int p = 0; p < 4; ++p) {
            a00[p] = nib_pair(x0, p);
            a01[p] = nib_pair(x1, p);
            a10[p] = nib_pair(y0, p);
            a11[p] = nib_pair(y1, p);
          }
          // refill the slot once every lane has unpacked both its words (the
          // shared loads have completed, so the copy cannot overtake them);
          // with two tiles, after the second tile's words (or the first's
          // when there is no second)
          if (h == 1 && (TPC == 1 || tt == 1 || !has1)) {
            __syncwarp();
            fetch(i + WD);
          }
          const __half2* q0 = reinterpret_cast<const __half2*>(&sv0);
          const __half2* q1 = reinterpret_cast<const __half2*>(&sv1);
          const float f00 = h ? __high2float(q0[0]) : __low2float(q0[0]);
          const float f01 = h ? __high2float(q0[1]) : __low2float(q0[1]);
          const float f10 = h ? __high2float(q1[0]) : __low2float(q1[0]);
          const float f11 = h ? __high2float(q1[1]) : __low2float(q1[1]);
          unsigned long long s00 = 0, s01 = 0, s10 = 0, s11 = 0;
          if constexpr (PACKED) {
            s00 = dup2(f00);
            s01 = dup2(f01);
            s10 = dup2(f10);
            s11 = dup2(f11);
          }
          const uint8_t* bb = sb + (pc * C * 2 + h) * 512 + (h ? lsw1 : lsw0);
#pragma unroll
          for (int cg = 0; cg < C; ++cg) {
            const uint4 bf = *reinterpret_cast<const uint4*>(bb + cg * 1024);
            float d[4];
            mma_bf16_first(d, a00, bf.x, bf.y);
            mma_bf16_acc(d, a01, bf.z, bf.w);
            if constexpr (PACKED) {
              ffma2(acc[tt][0][cg][0], s00, d[0], d[1]);
              ffma2(acc[tt][0][cg][1], s01, d[2], d[3]);
            } else {
              accf[tt][0][cg][0] = fmaf(f00, d[0], accf[tt][0][cg][0]);
              accf[tt][0][cg][1] = fmaf(f00, d[1], accf[tt][0][cg][1]);
              accf[tt][0][cg][2] = fmaf(f01, d[2], accf[tt][0][cg][2]);
              accf[tt][0][cg][3] = fmaf(f01, d[3], accf[tt][0][cg][3]);
            }
            float e[4];
            mma_bf16_first(e, a10, bf.x, bf.y);
            mma_bf16_acc(e, a11, bf.z, bf.w);
            if constexpr (PACKED) {
              ffma2(acc[tt][1][cg][0], s10, e[0], e[1]);
              ffma2(acc[tt][1][cg][1], s11, e[2], e[3]);
            } else {
              accf[tt][1][cg][0] = fmaf(f10, e[0], accf[tt][1][cg][0]);
              accf[tt][1][cg][1] = fmaf(f10, e[1], accf[tt][1][cg][1]);
              accf[tt][1][cg][2] = fmaf(f11, e[2], accf[tt][1][cg][2]);
              accf[tt][1][cg][3] = fmaf(f11, e[3], accf[tt][1][cg][3]);
            }
          }
        }
        }
        }
        if ((RG || (R1 ? (i & 3) == 3 : (i & 1))) && c + NSLOT < nchunks) {  // this warp is done with the slot
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&bempty[slot]));
        }
      }
    }
  compute_done:;
    asm volatile("cp.async.wait_all;" ::: "memory");  // no copy into the ring outlives the loop
  } else {
    // ---- converter warps ----
    const int ct = tid - COMPUTE_THREADS;  // k = 4ct .. 4ct + 3 of each chunk
    const int pc = ct >> 4, h = (ct >> 3) & 1, j = (ct >> 1) & 3, tql = 2 * (ct & 1);
    // byte offset of column (cg, gl) for the k pairs 4ct (.x/.y) and 4ct + 2 (.z/.w)
    const int kbase = (pc * C * 2 + h) * 512 + j * 4;
    const int s2 = pc & 1;
    const int oa = ((tql) ^ h) * 16, ob = ((tql + 1) ^ h) * 16;
    asm volatile("griddepcontrol.wait;" ::: "memory");  // x may come from the previous kernel
    // row m of this launch: x row xrows[m] when a row list is given (checked:
    // an index outside [0, x_rows) reads zeros and sets STATUS_BAD_ROW)
    int64_t xoff[MAXM];
#pragma unroll
    for (int m = 0; m < MAXM; ++m) {
      xoff[m] = -1;
      if (m < mrows) {
        if (a.xrows == nullptr) {
          xoff[m] = (int64_t)m * a.K;
        } else {
          const int32_t r = __ldg(a.xrows + m);
          if (r >= 0 && (int64_t)r < a.x_rows) xoff[m] = (int64_t)r * a.K;
          else if (ct == 0 && split == 0) atomicOr(a.status, STATUS_BAD_ROW);
        }
      }
    }
    const float* xr = a.x + bp0 * 64 + 4 * ct;
    // Stage chunk c: this thread's 16 bytes of every token row (k = 4ct..4ct+3).
    // Each thread reads back only what it copied, so completion needs no barrier.
    auto stage = [&](int c) {
      if (c < nchunks) {
        uint8_t* xs = smem + S::XRAW_OFF + (c % S::XSTAGES) * S::XSLOT;
        const bool pair_ok = c * CHUNK_PAIRS + pc < npairs;
        const bool k_ok = pair_ok && (bp0 + (int64_t)c * CHUNK_PAIRS) * 64 + 4 * ct < a.K;
        if (k_ok) {
#pragma unroll
          for (int m = 0; m < MAXM; ++m)
            if (xoff[m] >= 0)
              cp_async16(smem_u32(xs + m * (CHUNK_K * 4) + ct * 16),
                         xr + xoff[m] + (int64_t)c * CHUNK_K);
        }
      }
      asm volatile("cp.async.commit_group;" ::: "memory");
    };
    constexpr int XLEAD = S::XSTAGES - 1;  // chunks of x staged ahead of the one converted
#pragma unroll
    for (int c = 0; c < XLEAD; ++c) stage(c);
    for (int c = 0; c < nchunks; ++c) {
      const int slot = c & (NSLOT - 1);
      uint8_t* sb = smem + slot * S::SLOT;
      const uint8_t* xs = smem + S::XRAW_OFF + (c % S::XSTAGES) * S::XSLOT;
      const bool pair_ok = c * CHUNK_PAIRS + pc < npairs;
      const bool k_ok = pair_ok && (bp0 + (int64_t)c * CHUNK_PAIRS) * 64 + 4 * ct < a.K;
      // chunk c staged (the next XLEAD - 1 may be in flight)
      asm volatile("cp.async.wait_group %0;" ::"n"(XLEAD - 1) : "memory");
      stage(c + XLEAD);  // refills the slot read in the previous iteration
      if (c >= NSLOT &&
          !mbar_wait_bounded(smem_u32(&bempty[slot]), (uint32_t)(((c / NSLOT) + 1) & 1), &s_err)) {
        s_err = 1;
        break;
      }
      if (pair_ok) {
        constexpr int MG = MAXM < 4 ? MAXM : 4;  // rows read back together
#pragma unroll
        for (int m0 = 0; m0 < MAXM; m0 += MG) {
          float4 v[MG];
#pragma unroll
          for (int mm = 0; mm < MG; ++mm) {
            v[mm] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            if (m0 + mm < mrows && k_ok && xoff[m0 + mm] >= 0)
              v[mm] = *reinterpret_cast<const float4*>(xs + (m0 + mm) * (CHUNK_K * 4) + ct * 16);
          }
#pragma unroll
          for (int mm = 0; mm < MG; ++mm) {
            const int m = m0 + mm;
            if (m < mrows) {
              uint32_t ta[3], tb[3];
              split3(v[mm].x, v[mm].y, ta[0], ta[1], ta[2]);
              split3(v[mm].z, v[mm].w, tb[0], tb[1], tb[2]);
#pragma unroll
              for (int t = 0; t < 3; ++t) {
                const int col = DENSE ? 3 * m + t : 8 * m + t;
                const int cg = col >> 3, gl = col & 7;
                uint8_t* base = sb + kbase + cg * 1024 + (gl ^ s2) * 64;
                *reinterpret_cast<uint32_t*>(base + oa) = ta[t];
                *reinterpret_cast<uint32_t*>(base + ob) = tb[t];
              }
            }
          }
        }
      }
      mbar_arrive(smem_u32(&bfull[slot]));
    }
    // arrival number for the split-K epilogue, drawn once the last chunk is
    // handed over: the compute warps still have up to a ring of chunks to go,
    // which hides the atomic's latency, and CTAs draw in about the order they
    // finish (the previous launch has reset the word)
    if (ct == 0 && a.e.splits > 1 && !a.cluster) s_arrival = split_arrive(&a.e.counters[blockIdx.x]);
    asm volatile("cp.async.wait_all;" ::: "memory");
  }

  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");  // outputs and scratch: after the previous kernel
  __syncthreads();
  const bool failed = s_err != 0;
  // a CTA of a cluster stays for the cluster barriers below whatever happened
  if (failed && !a.cluster) {
    if (tid == 0) atomicOr(a.status, STATUS_TIMEOUT);
    return;
  }

  if constexpr (TPC == 2) {
    // ---- two tiles, whole K: add the four K slices in shared memory, write y ----
    float* red = reinterpret_cast<float*>(smem);  // [SLICES][C*8 columns][T2_LD]
    constexpr int RS = C * 8 * T2_LD;
    if (compute) {
      const int g = lane >> 2, tq = lane & 3;
#pragma unroll
      for (int tt = 0; tt < 2; ++tt)
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
          for (int cg = 0; cg < C; ++cg)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              float v;
              if constexpr (PACKED) {
                const float2 pr = split2(acc[tt][r][cg][e >> 1]);
                v = (e & 1) ? pr.y : pr.x;
              } else {
                v = accf[tt][r][cg][e];
              }
              red[sl * RS + (cg * 8 + 2 * tq + (e & 1)) * T2_LD + tt * TILE_N + (2 * rgp + r) * 16 + g +
                  8 * (e >> 1)] = v;
            }
    }
    __syncthreads();
    if (a.e.idx != nullptr) {
      // greedy pick: per tile, thread tid owns row tid % 128 for token rows
      // tid / 128 + 5k (as on the one-tile path), then the tile's maximum
      constexpr int MG = KERNEL_THREADS / TILE_N;
      constexpr int MT = (MAXM + MG - 1) / MG;
      const int row = tid % TILE_N, mfirst = tid / TILE_N;
#pragma unroll 1
      for (int tt = 0; tt < 2; ++tt) {
        if (tt == 1 && !has1) break;  // the same for every thread of the CTA
        float val[MT];
#pragma unroll
        for (int k = 0; k < MT; ++k) {
          const int m = mfirst + k * MG;
          val[k] = 0.0f;
          if (m < mrows) {
            const int c0 = DENSE ? 3 * m : 8 * m;
            float v = 0.0f;
#pragma unroll
            for (int t = 0; t < 3; ++t)
#pragma unroll
              for (int s = 0; s < SLICES; ++s) v += red[s * RS + (c0 + t) * T2_LD + tt * TILE_N + row];
            val[k] = v;
          }
        }
        EpiArgs e = a.e;
        e.N = a.w[tt ? wi1 : wi].N;
        finish_tile<MT, MG, MAXM>(e, val, row, mfirst, tt ? tile1 : tile, 0, mrows, 0, 0u, -1, &s_flag,
                                  kred, []() { __syncthreads(); });
      }
      return;
    }
    // thread t < 512: row t % 256 of the two tiles, token rows t / 256 + 2k;
    // fixed order of terms and slices, as on the other paths
    if (tid < 2 * 2 * TILE_N) {
      const int row = tid & (2 * TILE_N - 1);
      const int tt = row >> 7;
      if (tt == 0 || has1) {
        const int ww = tt ? wi1 : wi;
        const int64_t n = (tt ? tile1 : tile) * TILE_N + (row & (TILE_N - 1));
        float* y = a.w[ww].y;
        const int64_t N = a.w[ww].N;
        if (n < N) {
          for (int m = tid >> 8; m < mrows; m += 2) {
            const int c0 = DENSE ? 3 * m : 8 * m;
            float v = 0.0f;
#pragma unroll
            for (int t = 0; t < 3; ++t)
#pragma unroll
              for (int s = 0; s < SLICES; ++s) v += red[s * RS + (c0 + t) * T2_LD + row];
            y[(int64_t)m * N + n] = v;
          }
        }
      }
    }
    return;
  }

  if constexpr (RG) {
    // ---- row-group CTA: add the 16 K slices in shared memory and write y ----
    float* red = reinterpret_cast<float*>(smem);  // [16 slices][C*8 columns][RG_LD]
    constexpr int RS = C * 8 * RG_LD;
    if (compute) {
      const int g = lane >> 2, tq = lane & 3;
#pragma unroll
      for (int r = 0; r < 2; ++r)
#pragma unroll
        for (int cg = 0; cg < C; ++cg)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float v;
            if constexpr (PACKED) {
              const float2 pr = split2(acc[0][r][cg][e >> 1]);
              v = (e & 1) ? pr.y : pr.x;
            } else {
              v = accf[0][r][cg][e];
            }
            red[sl * RS + (cg * 8 + 2 * tq + (e & 1)) * RG_LD + r * 16 + g + 8 * (e >> 1)] = v;
          }
    }
    __syncthreads();
    // thread: row tid % 32 of the pair, token rows tid / 32 + 20k; fixed order
    // of terms and slices, as on the split path
    const int row = tid & 31;
    const int64_t n = tile * TILE_N + rgp * 32 + row;
    float* y = a.w[wi].y;
    if (n < a.w[wi].N) {
      for (int m = tid >> 5; m < mrows; m += KERNEL_THREADS / 32) {
        const int c0 = DENSE ? 3 * m : 8 * m;
        float v = 0.0f;
#pragma unroll
        for (int t = 0; t < 3; ++t)
#pragma unroll
          for (int s = 0; s < NSL; ++s) v += red[s * RS + (c0 + t) * RG_LD + row];
        y[(int64_t)m * a.w[wi].N + n] = v;
      }
    }
    return;
  }

  // ---- gather: per tile row and MMA column, the four (two) K slices ----
  float* red = reinterpret_cast<float*>(smem);  // [NSL][C*8][RED_LD]
  constexpr int RS = C * 8 * RED_LD;
  if (compute) {
    const int g = lane >> 2, tq = lane & 3;
#pragma unroll
    for (int r = 0; r < NRG; ++r)
#pragma unroll
      for (int cg = 0; cg < C; ++cg)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float v;
          if constexpr (PACKED) {
            const float2 pr = split2(acc[0][r][cg][e >> 1]);
            v = (e & 1) ? pr.y : pr.x;
          } else {
            v = accf[0][r][cg][e];
          }
          red[sl * RS + (cg * 8 + 2 * tq + (e & 1)) * RED_LD + ((R1 ? (warp & 7) : 2 * rgp) + r) * 16 + g +
              8 * (e >> 1)] = v;
        }
  }
  __syncthreads();

  // all threads take part from here: thread tid owns tile row tid % 128 for
  // the token rows tid / 128 + 5k, so the split-K reads of the last CTA are
  // spread over the whole CTA and issued in a single round
  constexpr int MGROUPS = KERNEL_THREADS / TILE_N;
  constexpr int MT = (MAXM + MGROUPS - 1) / MGROUPS;
  static_assert(KERNEL_THREADS % TILE_N == 0, "whole groups of tile rows");
  const int row = tid % TILE_N, mfirst = tid / TILE_N;
  float val[MT];
#pragma unroll
  for (int k = 0; k < MT; ++k) {
    const int m = mfirst + k * MGROUPS;
    val[k] = 0.0f;
    if (m < mrows) {
      const int c0 = DENSE ? 3 * m : 8 * m;
      float v = 0.0f;
#pragma unroll
      for (int t = 0; t < 3; ++t)  // fixed order: term 0..2, each slice 0..3
#pragma unroll
        for (int s = 0; s < S::NSL; ++s) v += red[s * RS + (c0 + t) * RED_LD + row];
      val[k] = v;
    }
  }
  if (a.cluster) {
    // K splits of this tile = the CTAs of this cluster, rank = split.  Each
    // CTA publishes its sums in its own shared memory; after the cluster
    // barrier CTA r adds up the r-th share of the tile's outputs, reading the
    // splits' sums in ascending split order (the same order and operations as
    // the global-memory path), then a second barrier keeps every CTA's shared
    // memory alive until its peers have read it.
    float* xch = reinterpret_cast<float*>(smem + S::XCH_OFF);
#pragma unroll
    for (int k = 0; k < MT; ++k) {
      const int m = mfirst + k * MGROUPS;
      if (m < mrows) xch[m * TILE_N + row] = val[k];
    }
    const uint32_t nsplit = (uint32_t)a.e.splits;
    const bool layout_ok = cluster_rank() == (uint32_t)split && cluster_size() == nsplit;
    cluster_sync_all();
    if (!failed && layout_ok) {
      float* y = a.w[wi].y;
      const int64_t N = a.w[wi].N;
      const int outs = mrows * TILE_N;
      const int per = (outs + (int)nsplit - 1) / (int)nsplit;
      const int o_end = min(outs, (split + 1) * per);
      const uint32_t xa = smem_u32(xch);
      for (int o = split * per + tid; o < o_end; o += KERNEL_THREADS) {
        float t[8];
#pragma unroll
        for (int s = 0; s < 8; ++s)
          t[s] = s < (int)nsplit ? ld_cluster(cluster_map(xa + 4u * (uint32_t)o, (uint32_t)s)) : 0.0f;
        float v = 0.0f;
#pragma unroll
        for (int s = 0; s < 8; ++s)
          if (s < (int)nsplit) v += t[s];
        const int64_t n = tile * TILE_N + (o % TILE_N);
        if (n < N) y[(int64_t)(o / TILE_N) * N + n] = v;
      }
    }
    cluster_sync_all();
    if ((failed || !layout_ok) && tid == 0) atomicOr(a.status, STATUS_TIMEOUT);
    return;
  }

  // this weight's outputs; partial sums and counters indexed by the global tile
  EpiArgs e = a.e;
  e.y = a.w[wi].y;
  e.N = a.w[wi].N;
  e.partial = a.e.partial + (int64_t)a.w[wi].tile_start * TILE_N;
  finish_tile<MT, MGROUPS, MAXM>(e, val, row, mfirst, tile, 0, mrows, split, s_arrival,
                                 (int)blockIdx.x, &s_flag, kred, []() { __syncthreads(); });
}

// Clusters of `size` CTAs of this kernel that the device holds at once (0 if
// none or unknown), per device, cached.
template <int C, bool DENSE>
int cluster_capacity(int device, int size) {
  static std::atomic<int> cache[64][9];  // value + 1; 0 = not yet asked
  if (size < 2 || size > 8) return 0;
  std::atomic<int>& slot = cache[device & 63][size];
  const int c = slot.load();
  if (c > 0) return c - 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1, (unsigned)size, 1);
  cfg.blockDim = dim3(KERNEL_THREADS);
  cfg.dynamicSmemBytes = MmaCfg<C, 1, DENSE>::BYTES;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = (unsigned)size;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, mma_kernel<C, DENSE, false, 1>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  slot.store(n + 1);
  return n;
}

template <int C, bool DENSE, bool RG, int TPC = 1>
int launch_c(const MmaLaunch& L, const float* x, int mrows, int32_t* idx, float* maxval,
             const MmaPlan& plan, const Workspace& ws, int64_t mb, cudaStream_t s,
             const int32_t* xrows, int64_t x_rows) {
  using S = MmaCfg<C, TPC, DENSE, RG>;
  const Weight* W0 = L.W[0];
  MmaArgs a;
  int tiles = 0;
  for (int i = 0; i < MMA_GROUP_MAX; ++i) {
    if (i < L.count) {
      const Weight* W = L.W[i];
      a.w[i].nib = reinterpret_cast<const uint4*>(W->nib);
      a.w[i].scl = reinterpret_cast<const uint8_t*>(W->d);
      a.w[i].y = L.y[i] ? L.y[i] + mb * W->N : nullptr;
      a.w[i].N = W->N;
      a.w[i].tile_start = tiles;
      tiles += (int)W->tiles;
    } else {
      a.w[i] = a.w[0];
      a.w[i].tile_start = 1 << 30;
    }
  }
  a.nweights = L.count;
  a.x = x;
  a.xrows = xrows;
  a.x_rows = x_rows;
  a.K = W0->K;
  a.KBP = W0->KBP;
  a.mrows = mrows;
  a.kbp_per_split = RG ? W0->KBP : plan.kbp_per_split;
  a.status = ws.status;
  a.e.N = W0->N;
  a.e.N_pad = (int64_t)tiles * TILE_N;
  a.e.M = mrows;
  a.e.y = nullptr;
  a.e.idx = idx ? idx + mb : nullptr;
  a.e.maxval = (idx && maxval) ? maxval + mb : nullptr;
  a.e.splits = RG ? 1 : plan.splits;
  a.e.partial = ws.partial;
  a.e.counters = ws.counters;
  a.e.status = ws.status;
  a.e.keys = ws.keys + mb;
  a.e.argmax_done = ws.argmax_done;
  a.e.tiles = tiles;
  // per device, once (atomic: q4mm_forward and q4mm_forward_noalloc hold
  // different locks; setting the attribute twice is harmless)
  static std::atomic<bool> attr_set[64];
  if (!attr_set[W0->device & 63].load(std::memory_order_acquire)) {
    if (cudaFuncSetAttribute(mma_kernel<C, DENSE, RG, TPC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             S::BYTES) != cudaSuccess)
      return Q4_ERR_CUDA;
    attr_set[W0->device & 63].store(true, std::memory_order_release);
  }
  // Split-K through distributed shared memory when the K splits of every tile
  // fit in one cluster of at most 4 CTAs and all the launch's clusters are
  // resident at once; otherwise (and for the greedy pick) through global
  // memory.  Both add the splits in the same order.  (Measured on GB300 for
  // the 7B decoder layers: clusters of 4 beat the global-memory exchange,
  // clusters of 5 lost to it.)
  a.cluster = !RG && TPC == 1 && plan.splits > 1 && plan.splits <= Q4MM_CLUSTER_MAX && idx == nullptr &&
              tiles <= cluster_capacity<C, DENSE>(W0->device, plan.splits);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = RG ? dim3((unsigned)tiles * 4u, 1, 1)
                   : dim3((unsigned)((tiles + TPC - 1) / TPC), (unsigned)plan.splits, 1);
  cfg.blockDim = dim3(KERNEL_THREADS);
  cfg.dynamicSmemBytes = S::BYTES;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 1;
  attr[1].val.clusterDim.y = (unsigned)plan.splits;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = a.cluster ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, mma_kernel<C, DENSE, RG, TPC>, a) == cudaSuccess ? Q4_OK : Q4_ERR_CUDA;
}

// Rows per launch: 16 with dense packing (6 column groups), 3 with one row
// per column group (batch-invariant mode).
int rows_per_launch(bool batch_invariant) { return batch_invariant ? MAX_CG : (MAX_CG_DENSE * 8) / 3; }

}  // namespace

MmaPlan mma_plan_tiles(int64_t tiles, int64_t KBP, int num_sms) {
  // K partition from the shapes only (never from M).  One CTA per SM: splits =
  // floor(SMs / tiles) for a single wave, at least one, and small enough that
  // each CTA keeps at least two block pairs.
  MmaPlan p;
  p.num_sms = num_sms;
  int64_t sp = (int64_t)num_sms / tiles;
  int64_t cap = KBP / 2;
  if (cap < 1) cap = 1;
  if (sp < 1) sp = 1;
  if (sp > cap) sp = cap;
  if (sp > MAX_SPLITS) sp = MAX_SPLITS;  // the arrival count field of the epilogue
  p.kbp_per_split = (KBP + sp - 1) / sp;
  p.splits = (int)((KBP + p.kbp_per_split - 1) / p.kbp_per_split);
  return p;
}

MmaPlan mma_plan(const Weight* W, int num_sms) { return mma_plan_tiles(W->tiles, W->KBP, num_sms); }

size_t mma_partial_bytes_tiles(int64_t tiles, const MmaPlan& p, int64_t M, bool batch_invariant) {
  if (p.splits <= 1) return 0;
  const int64_t rpl = rows_per_launch(batch_invariant);
  const int64_t ml = M < rpl ? M : rpl;
  return (size_t)p.splits * (size_t)ml * (size_t)(tiles * TILE_N) * sizeof(unsigned long long);
}

size_t mma_partial_bytes(const Weight* W, const MmaPlan& p, int64_t M, bool batch_invariant) {
  return mma_partial_bytes_tiles(W->tiles, p, M, batch_invariant);
}

int mma_rows_per_launch(bool batch_invariant) { return rows_per_launch(batch_invariant); }

int mma_launch_count(int64_t M, bool batch_invariant) {
  const int64_t rpl = rows_per_launch(batch_invariant);
  return (int)((M + rpl - 1) / rpl);
}

bool mma_row_groups(const MmaPlan& plan, int64_t K, bool batch_invariant, bool greedy_pick,
                    int64_t launch_rows) {
  return !batch_invariant && !greedy_pick && launch_rows <= 8 && plan.splits >= 4 &&
         K <= Q4MM_RG_MAX_K;
}

int launch_mma_group(const MmaLaunch& L, const float* x, int64_t M, int32_t* idx, float* maxval,
                     const MmaPlan& plan, bool batch_invariant, const Workspace& ws, cudaStream_t s,
                     const int32_t* xrows, int64_t x_rows) {
  int64_t tiles = 0;
  for (int i = 0; i < L.count; ++i) tiles += L.W[i]->tiles;
  if (plan.splits > 1 && tiles > MAX_COUNTERS) return Q4_ERR_SHAPE;
  const int64_t K = L.W[0]->K;
  const int64_t rpl = rows_per_launch(batch_invariant);
  // row-group CTAs (per launch, below): no K split and so no cross-CTA
  // exchange, when four CTAs per tile fit on the SMs (the split plan has at
  // least 4 splits), K is short and the launch has at most 8 rows; the plan
  // depends on the shapes and that row count only (y output, default mode)
  // two tiles per CTA (whole K, no split): launches of more tiles than SMs
  // run as CTAs that stream two tiles each, for one or two column groups in
  // default mode (y output or the greedy pick)
  const bool two = Q4MM_TWO_TILES && !batch_invariant && plan.splits == 1 && plan.num_sms > 0 &&
                   tiles > plan.num_sms;
  for (int64_t mb = 0; mb < M; mb += rpl) {
    const int mrows = (int)((M - mb) < rpl ? (M - mb) : rpl);
    const bool rg = mma_row_groups(plan, K, batch_invariant, idx != nullptr || xrows != nullptr, mrows);
    const float* xs = xrows ? x : x + mb * K;
    const int32_t* xr = xrows ? xrows + mb : nullptr;
    int st;
    if (batch_invariant) {
      switch (mrows) {
        case 1: st = launch_c<1, false, false>(L, xs, mrows, idx, maxval, plan, ws, mb, s, xr, x_rows); break;
        case 2: st = launch_c<2, false, false>(L, xs, mrows, idx, maxval, plan, ws, mb, s, xr, x_rows); break;
        default: st = launch_c<3, false, false>(L, xs, mrows, idx, maxval, plan, ws, mb, s, xr, x_rows); break;
      }
    } else {
      const int cgs = (3 * mrows + 7) / 8;  // column groups of this launch
      if (cgs >= 4) {  // 9 to 16 rows: one row group per warp, K splits
        switch (cgs) {
          case 4: st = launch_c<4, true, false>(L, xs, mrows, idx, maxval, plan, ws, mb, s, xr, x_rows); break;
          case 5: st = launch_c<5, true, false>(L, xs, mrows, idx, maxval, plan, ws, mb, s, xr, x_rows); break;
          default: st = launch_c<6, true, false>(L, xs, mrows, idx, maxval, plan, ws, mb, s, xr, x_rows); break;
        }
      } else if (rg) {
        switch (cgs) {
          case 1: st = launch_c<1, true, true>(L, xs, mrows, idx, maxval, plan, ws, mb, s, xr, x_rows); break;
          case 2: st = launch_c<2, true, true>(L, xs, mrows, idx, maxval, plan, ws, mb, s, xr, x_rows); break;
          default: st = launch_c<3, true, true>(L, xs, mrows, idx, maxval, plan, ws, mb, s, xr, x_rows); break;
        }
      } else {
        switch (cgs) {
          case 1:
            st = two ? launch_c<1, true, false, 2>(L, xs, mrows, idx, maxval, plan, ws, mb, s, xr, x_rows)
                     : launch_c<1, true, false>(L, xs, mrows, idx, maxval, plan, ws, mb, s, xr, x_rows);
            break;
          case 2:
            st = two ? launch_c<2, true, false, 2>(L, xs, mrows, idx, maxval, plan, ws, mb, s, xr, x_rows)
                     : launch_c<2, true, false>(L, xs, mrows, idx, maxval, plan, ws, mb, s, xr, x_rows);
            break;
          default: st = launch_c<3, true, false>(L, xs, mrows, idx, maxval, plan, ws, mb, s, xr, x_rows); break;
        }
      }
    }
    if (st) return st;
  }
  return Q4_OK;
}

int launch_mma(const Weight* W, const float* x, int64_t M, float* y, int32_t* idx, float* maxval,
               const MmaPlan& plan, bool batch_invariant, const Workspace& ws, cudaStream_t s) {
  MmaLaunch L;
  L.count = 1;
  L.W[0] = W;
  L.y[0] = y;
  return launch_mma_group(L, x, M, idx, maxval, plan, batch_invariant, ws, s);
}

}  // namespace q4
