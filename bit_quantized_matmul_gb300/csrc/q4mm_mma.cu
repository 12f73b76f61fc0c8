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
// Operands (every product exact, only fp32 accumulation rounds):
//   weights  (q - 8) as binary16: one three-input LOP3 puts a nibble pair
//            into the mantissas of 1024 + q (or 1024 + 16 q for the nibbles
//            in bits 4..7 of a byte), one f16x2 subtraction leaves q - 8 (or
//            16 (q - 8)), exact.  Rows R1 = R0 + 8 of a row group come from
//            the high nibble positions and carry the factor 16, removed with
//            the activation scale below.
//   x        two binary16 terms per value, x * s = t0 + t1 to 2^-21, with s a
//            power of two per (token row, 128 consecutive activations: two
//            block pairs) chosen from their largest |x| so that x * s stays
//            inside binary16's range; t0 keeps the top 11 significant bits of
//            x * s, t1 the rest.
// Per block the two MMAs accumulate D_b = sum_{k in b} (q-8) t in fresh fp32
// registers; the block's fp16 scale d is applied on the CUDA cores, per block
// pair P = d_0 D_0 + d_1 D_1, then acc += P / s (1/s exact), in ascending
// block-pair order.  At the end the K slices and the two terms of each row
// are added in a fixed order, then the K splits in ascending split order
// (q4mm_epilogue.cuh).
//
// CTA = one 128-row tile over a K range (block pairs [bp0, bp1)); 640 threads:
//
//   16 compute warps  warp w takes row groups 2(w&3), 2(w&3)+1 (32 rows) and
//                     K slice w>>2: block pairs bp0 + slice + 4i (with three or
//                     four column groups, 9 to 16 rows: row group w&7 and K
//                     slice (w>>3)&1, block pairs bp0 + slice + 2i).  Its lanes
//                     copy their 16-byte weight fragments (coalesced, 1 KB per
//                     warp and pair) and lanes 0..7 the pair's 128 bytes of
//                     fp16 scales (512 and 64 bytes with one row group per
//                     warp) from HBM into the warp's private cp.async ring,
//                     two pairs ahead; each lane reads back its own fragments,
//                     which in the fragment layout are exactly the A registers
//                     of m16n8k16 MMAs once unpacked.  The first pairs are on
//                     their way before the kernel waits for the previous one
//                     on the stream (weights never depend on it).  No CTA
//                     barrier in the loop.
//   4 converter warps stage, per chunk of 8 block pairs, the activations as
//                     the two binary16 terms above in B-fragment order (term t
//                     of token row m in MMA column 2m + t) together with each
//                     row's 1/s, into a 4-slot (2-slot from three column
//                     groups) shared-memory ring with full/empty mbarriers
//                     (every wait bounded).  The fp32 rows arrive by cp.async
//                     several chunks ahead.
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
// Batch-invariant mode runs every launch, whatever its row count, with the
// same four-column-group kernel and the K partition of the shapes: a row goes
// through the same operations in the same order wherever it sits in the
// launch (an MMA output element depends only on its own row of A, column of
// B and accumulator input) and whatever its neighbours hold (its scales come
// from its own values).  In the default mode the launch's row count picks the
// CTA layout, so a row's bits may differ with M within the tolerance.
#include <cuda_fp16.h>

#include <atomic>

#include "q4mm_epilogue.cuh"
#include "q4mm_internal.h"

namespace q4 {
namespace {

constexpr int MAX_CG = 4;          // column groups per launch: two terms per token row, 16 rows
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
#ifndef Q4MM_WD1
#define Q4MM_WD1 2  // CTAs of one tile
#endif
#ifndef Q4MM_WD2
#define Q4MM_WD2 2  // two-tile CTAs (twice the bytes per pair)
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
// row-group CTAs for launches of at most this many token rows
#ifndef Q4MM_RG_MAX_ROWS
#define Q4MM_RG_MAX_ROWS 8
#endif
#ifndef Q4MM_RG_MAX_K
#define Q4MM_RG_MAX_K 4096
#endif
// B ring depth of row-group CTAs: every chunk of a K up to 4096
#ifndef Q4MM_RG_NSLOT
#define Q4MM_RG_NSLOT 4
#endif
// convert every chunk of a CTA's activations before its main loop (launches
// of one or two column groups whose CTAs cover at most UP_CHUNKS chunks);
// for two-tile CTAs too, which then run without converter warps.  Measured
// on GB300 (gate/up group of a 7B layer, us per call, up front / converter
// warps): 14.79 / 15.64 at M = 1, 15.83 / 16.82 at M = 4, 22.73 / 23.76 at
// M = 8
#ifndef Q4MM_UPFRONT
#define Q4MM_UPFRONT 1
#endif
#ifndef Q4MM_UP_TWO
#define Q4MM_UP_TWO 1
#endif
#ifndef Q4MM_TWO_TILES
#define Q4MM_TWO_TILES 1
#endif
// Up-front launches take their activations from a pre-conversion pass (one
// small kernel converts x once into the chunk-slot image that every CTA
// copies in) instead of converting the whole x in every CTA, from these row
// counts on (0: never).  Measured on GB300 over the 7B layer (8 layer copies
// per graph, us per call, without / with the pass): row-group CTAs q/k/v
// 7.95 / 6.58 and o 7.84 / 6.34 at M = 8, 5.30 / 5.06 and 5.28 / 5.05 at
// M = 4, even at M = 3 and slower at M = 2; two-tile CTAs (gate/up) slower at
// every M (22.04 / 22.30 at M = 8, 15.35 / 16.39 at M = 2); K-split CTAs
// (down) 17.39 / 17.00 at M = 8, 16.32 / 16.22 at M = 5 and slower at M <= 4,
// but slower in a batch-invariant M = 124 step (16 launches of 8 rows on one
// L2-resident weight: 600 / 621 us per layer for gate/up and down), so off.
#ifndef Q4MM_XPRE_RG_ROWS
#define Q4MM_XPRE_RG_ROWS 4
#endif
#ifndef Q4MM_XPRE_SPLIT_ROWS
#define Q4MM_XPRE_SPLIT_ROWS 0
#endif
#ifndef Q4MM_XPRE_TWO_ROWS
#define Q4MM_XPRE_TWO_ROWS 0
#endif
// and only for activations of at least this many chunks (512 k each): a
// short K converts quickly in the kernel, and an extra launch costs more
// (Q4_0 896 x 896, 400 copies per graph: 2.69 / 3.21 us per call at M = 4)
#ifndef Q4MM_XPRE_MIN_CHUNKS
#define Q4MM_XPRE_MIN_CHUNKS 4
#endif
constexpr int RG_LD = 36;  // row stride of the row-group slice sums (32 rows + 4)
constexpr int T2_LD = 2 * TILE_N + 4;  // row stride of the two-tile slice sums (256 rows + 4)
// row stride of the slice sums in shared memory: 4 (mod 32 banks), so that
// the accumulator stores of a warp (lanes 4g + tq at column 2tq, row g) hit
// 32 different banks and the per-row reads stay consecutive
constexpr int RED_LD = TILE_N + 4;
constexpr int TERMS = 2;  // binary16 terms per activation

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
  // 0, or the tile count of the first weight when two-tile CTAs pair tile b
  // of weight 0 with tile b of weight 1 and write h = SiLU(y0) * y1 into
  // weight 0's output (gate and up projections of a gated MLP)
  int gated;
  unsigned int* status; // device status word (bounded-wait expiry)
  unsigned long long wait_ns;  // bound of the waits between roles
  int stall;            // test setting: the converters hand over no chunk
  int cluster;          // 1: the K splits of a tile are one thread-block cluster
  // up-front launches: null, or the chunk-slot image written by the
  // pre-conversion pass ([split][chunk] slots, xpre_stride bytes per split)
  const uint8_t* xpre;
  int64_t xpre_stride;
  EpiArgs e;
};

// Launches of one or two column groups whose CTAs cover at most this many
// chunks convert all their activations before the main loop, with every
// thread of the CTA, into one ring slot per chunk.
constexpr int UP_CHUNKS = 8;

template <int C, int TPC = 1, bool RG = false, bool UP = false>
struct MmaCfg {
  static constexpr int MAXM = C * 8 / TERMS;  // token rows per launch
  // three or four column groups (9 to 16 token rows): one row group per
  // compute warp, 8 row groups x 2 K slices, so that the accumulators fit;
  // a two-slot B ring and three x stages, so that the larger fragments fit in
  // shared memory
  static constexpr bool R1 = !RG && TPC == 1 && C >= 3;
  static constexpr int NSL = R1 ? 2 : SLICES;  // K slices of a tile's CTA
  static constexpr int NRG = R1 ? 1 : 2;       // row groups per compute warp
  // B ring depth (a power of two); row-group CTAs hold every chunk of their
  // K (at most 8) so that their converters never wait for a slot
  static constexpr int NSLOT = UP ? UP_CHUNKS : (RG ? Q4MM_RG_NSLOT : (R1 ? 2 : 4));
  static constexpr int BF_PAIR = C * 1024;  // B fragments of a pair: [cg][h][32 slots] x 16 B
  // per (pair, token row) {1/s, 1/s, 1/(16 s), 1/(16 s)}, after the fragments
  static constexpr int SIG_OFF = CHUNK_PAIRS * BF_PAIR;
  static constexpr int SLOT = SIG_OFF + CHUNK_PAIRS * MAXM * 16;
  static constexpr int RING = NSLOT * SLOT;
  // converter staging: per slot the chunk's raw fp32 x rows
  // chunks of x in flight + the one converted
  static constexpr int XSTAGES = UP ? 0 : ((R1 || (RG && C == 2)) ? 3 : (C == 2 ? 4 : 6));
  static constexpr int XSLOT = MAXM * CHUNK_K * 4;
  static constexpr int XRAW_OFF = RING;
  static constexpr int RED = NSL * C * 8 * RED_LD * 4;  // per-slice sums for the gather
  static constexpr int XCH_OFF = (RED + 15) / 16 * 16;  // cluster split-K: this CTA's sums
  static constexpr int XCH = MAXM * TILE_N * 4;           // [token row][tile row] fp32
  // weight pairs in flight per compute warp: a private ring of WD slots, each
  // the warp's 16-byte fragments of its two row groups (1 KB) and their fp16
  // scales (128 B), filled by cp.async (half of that with one row group)
  static constexpr int WD = TPC == 2 ? Q4MM_WD2 : Q4MM_WD1;
  static constexpr int WSLOT = NRG * (512 + 64);
  static constexpr int WSCL = NRG * 512;  // offset of the scales in a slot
  static constexpr int WR_OFF = RING + XSTAGES * XSLOT;
  static constexpr int WR = COMPUTE_WARPS * WD * WSLOT * TPC;
  static constexpr int BAR_OFF = WR_OFF + WR > XCH_OFF + XCH ? WR_OFF + WR : XCH_OFF + XCH;
  static constexpr int BYTES = BAR_OFF + 2 * NSLOT * 8;
  static_assert(!R1 || TPC == 1, "one row group per warp: one tile per CTA");
  static_assert(!UP || C <= 2, "up-front conversion: one or two column groups");
  // threads: CTAs that convert up front need no converter warps and get the
  // register file of 512 threads (128 registers each, where 640 threads get
  // 96), except row-group CTAs of two column groups.  Measured on GB300 over
  // the 7B layer (us per call, 640 / 512 threads): down 12.11 / 11.73 at M = 1,
  // 17.41 / 16.81 at M = 8; o 4.20 / 4.05 at M = 1; q/k/v and o at M = 8
  // 6.45 / 6.65 and 6.39 / 6.55 (row-group, two column groups).
  static constexpr int THREADS = (UP && !(RG && C == 2)) ? COMPUTE_THREADS : KERNEL_THREADS;
  static_assert(BYTES <= 227 * 1024 - 1024, "shared memory of one CTA");
  static_assert(SLOT % 16 == 0 && XSLOT % 16 == 0, "16-byte aligned ring slots");
  static_assert(SIG_OFF == CHUNK_PAIRS * C * 1024 && SLOT == CHUNK_PAIRS * C * 1024 + CHUNK_PAIRS * MAXM * 16,
                "chunk slot layout of the up-front conversion");
};

// The four A-fragment registers of one 32-bit fragment word (nibble pairs
// p = 0..3 at bits 4p and 16 + 4p) as exact binary16 pairs: 0x6400 | q is
// 1024 + q and 0x6400 | (q << 4) is 1024 + 16 q; one f16x2 subtraction of
// 1032 (or 1152) leaves q - 8 (or 16 (q - 8)).  Pairs 0 and 2 are rows R0,
// pairs 1 and 3 rows R1 (factor 16).
__device__ __forceinline__ void unpack_word(uint32_t w, uint32_t (&a)[4]) {
  const uint32_t w8 = w >> 8;
  uint32_t t0, t1, t2, t3;
  asm("lop3.b32 %0, %1, 0x000F000F, 0x64006400, 0xEA;" : "=r"(t0) : "r"(w));
  asm("lop3.b32 %0, %1, 0x00F000F0, 0x64006400, 0xEA;" : "=r"(t1) : "r"(w));
  asm("lop3.b32 %0, %1, 0x000F000F, 0x64006400, 0xEA;" : "=r"(t2) : "r"(w8));
  asm("lop3.b32 %0, %1, 0x00F000F0, 0x64006400, 0xEA;" : "=r"(t3) : "r"(w8));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(a[0]) : "r"(t0), "r"(0x64086408u));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(a[1]) : "r"(t1), "r"(0x64806480u));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(a[2]) : "r"(t2), "r"(0x64086408u));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(a[3]) : "r"(t3), "r"(0x64806480u));
}

// D = A B + C with C = 0 (first k-step of a block) and with C = D (second).
__device__ __forceinline__ void mma_f16_first(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                              uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%10, %10, %10, %10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.0f));
}
__device__ __forceinline__ void mma_f16_acc(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                            uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Two fp32 values in one 64-bit register pair; packed fp32x2 arithmetic, each
// half an ordinary fp32 operation.  `ss` holds {s, s} (or two factors).
__device__ __forceinline__ unsigned long long dup2(float s) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %1};" : "=l"(r) : "f"(s));
  return r;
}
// r = ss * (c0, c1)
__device__ __forceinline__ unsigned long long fmul2(unsigned long long ss, float c0, float c1) {
  unsigned long long r;
  asm("{\n\t.reg .b64 rc;\n\t"
      "mov.b64 rc, {%2, %3};\n\t"
      "mul.rn.f32x2 %0, %1, rc;\n\t}"
      : "=l"(r)
      : "l"(ss), "f"(c0), "f"(c1));
  return r;
}
// acc += ss * (c0, c1)
__device__ __forceinline__ void ffma2(unsigned long long& acc, unsigned long long ss, float c0,
                                      float c1) {
  asm("{\n\t.reg .b64 rc;\n\t"
      "mov.b64 rc, {%2, %3};\n\t"
      "fma.rn.f32x2 %0, %1, rc, %0;\n\t}"
      : "+l"(acc)
      : "l"(ss), "f"(c0), "f"(c1));
}
// acc += ss * v (both packed)
__device__ __forceinline__ void ffma2p(unsigned long long& acc, unsigned long long ss,
                                       unsigned long long v) {
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(ss), "l"(v));
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
// Bounded wait (limit_ns, 1 s by default, or until another thread of the CTA
// reported an expiry); returns false on expiry.  The timer is read only after
// many polls.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  const volatile int* err, unsigned long long limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  unsigned long long t0 = 0;
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 255u) == 0u) {
      if (*err) return false;
      const unsigned long long now = globaltimer();
      if (t0 == 0) t0 = now;
      else if (now - t0 > limit_ns) return false;
    }
  }
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
// the same copy, issued only where `on` is nonzero (a predicate, no branch)
__device__ __forceinline__ void cp_async16_if(uint32_t dst, const void* src, uint32_t on) {
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %2, 0;\n\t@p cp.async.cg.shared.global [%0], [%1], 16;\n\t}"
               ::"r"(dst), "l"(src), "r"(on) : "memory");
}

// binary16 pair (lo, hi) rounded to nearest
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// Two-term binary16 split of four activations (k .. k + 3) scaled by s:
// y = x s (exact, s a power of two), t0 keeps the top 11 significant bits of
// y (exact in binary16 whenever |y| >= 2^-14), t1 = y - t0 rounded to
// binary16, so y - t0 - t1 is at most 2^-21 |y| (plus 2^-24 where the terms
// fall below binary16's normal range).  Each term packs (k, k + 1) or
// (k + 2, k + 3) as an f16x2 word, the lower k in the low half.
__device__ __forceinline__ void split4(const float4& v, float s, uint32_t (&ta)[2], uint32_t (&tb)[2]) {
  float y0, y1, y2, y3, r0, r1, r2, r3;
  asm("{\n\t.reg .b64 xa, xb, ss, ya, yb;\n\t"
      "mov.b64 xa, {%8, %9};\n\t"
      "mov.b64 xb, {%10, %11};\n\t"
      "mov.b64 ss, {%12, %12};\n\t"
      "mul.rn.f32x2 ya, xa, ss;\n\t"
      "mul.rn.f32x2 yb, xb, ss;\n\t"
      "mov.b64 {%0, %1}, ya;\n\t"
      "mov.b64 {%2, %3}, yb;\n\t}"
      : "=f"(y0), "=f"(y1), "=f"(y2), "=f"(y3), "=f"(r0), "=f"(r1), "=f"(r2), "=f"(r3)
      : "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "f"(s));
  const float h0 = __uint_as_float(__float_as_uint(y0) & 0xFFFFE000u);
  const float h1 = __uint_as_float(__float_as_uint(y1) & 0xFFFFE000u);
  const float h2 = __uint_as_float(__float_as_uint(y2) & 0xFFFFE000u);
  const float h3 = __uint_as_float(__float_as_uint(y3) & 0xFFFFE000u);
  asm("{\n\t.reg .b64 ya, yb, ha, hb, ra, rb;\n\t"
      "mov.b64 ya, {%4, %5};\n\t"
      "mov.b64 yb, {%6, %7};\n\t"
      "mov.b64 ha, {%8, %9};\n\t"
      "mov.b64 hb, {%10, %11};\n\t"
      "sub.rn.f32x2 ra, ya, ha;\n\t"
      "sub.rn.f32x2 rb, yb, hb;\n\t"
      "mov.b64 {%0, %1}, ra;\n\t"
      "mov.b64 {%2, %3}, rb;\n\t}"
      : "=f"(r0), "=f"(r1), "=f"(r2), "=f"(r3)
      : "f"(y0), "f"(y1), "f"(y2), "f"(y3), "f"(h0), "f"(h1), "f"(h2), "f"(h3));
  ta[0] = pack_f16x2(h0, h1);
  ta[1] = pack_f16x2(r0, r1);
  tb[0] = pack_f16x2(h2, h3);
  tb[1] = pack_f16x2(r2, r3);
}

// Bytes of one chunk slot of C column groups: the B fragments of 8 block
// pairs, then per (pair, token row) {1/s, 1/s, 1/(16 s), 1/(16 s)}.
template <int C>
__host__ __device__ constexpr int chunk_slot_bytes() { return CHUNK_PAIRS * C * 1024 + CHUNK_PAIRS * (C * 8 / TERMS) * 16; }

// Up-front conversion of four activations (k .. k + 3, this thread's) of
// token row m into chunk slot sb: the largest |x| of the row over the warp's
// 128 elements (two block pairs) sets the power-of-two scale s, the two
// binary16 terms go to the row's B columns, and the pair's first thread
// writes 1/s and 1/(16 s).  sb is shared memory or the global image of the
// pre-conversion pass: the same operations either way, so the slot bytes are
// the same.  Every lane of the warp calls it with the same m (the reduction).
template <int C>
__device__ __forceinline__ void convert_row4(const float4& v, int m, uint8_t* sb, int kbase, int s2, int oa,
                                             int ob, int pc, bool sig_lane, bool pair_ok) {
  constexpr int MAXM = C * 8 / TERMS;
  constexpr int SIG_OFF = CHUNK_PAIRS * C * 1024;
  uint32_t u = __float_as_uint(fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
  asm volatile("redux.sync.max.u32 %0, %0, 0xffffffff;" : "+r"(u));
  int e = 14 - ((int)(u >> 23) - 127);
  e = max(-120, min(120, e));
  const float sc = __int_as_float((e + 127) << 23);
  if (pair_ok) {
    uint32_t ta[TERMS], tb[TERMS];
    split4(v, sc, ta, tb);
#pragma unroll
    for (int t = 0; t < TERMS; ++t) {
      const int col = TERMS * m + t;
      const int cg = col >> 3, gl = col & 7;
      uint8_t* base = sb + kbase + cg * 1024 + (gl ^ s2) * 64;
      *reinterpret_cast<uint32_t*>(base + oa) = ta[t];
      *reinterpret_cast<uint32_t*>(base + ob) = tb[t];
    }
    if (sig_lane) {
      const float r1 = __int_as_float((127 - e) << 23);
      const float r16 = __int_as_float((123 - e) << 23);
      *reinterpret_cast<float4*>(sb + SIG_OFF + (pc * MAXM + m) * 16) = make_float4(r1, r1, r16, r16);
    }
  }
}

// ----------------------------------------------------------------------------
// Shared-memory B fragments of one block pair: [cg][h][32 slots] x 16 bytes,
// slot of lane L = 4g + tq at L ^ sw with sw = 4 (pair & 1) + h, so that the
// converters' scattered 4-byte stores hit 32 distinct banks (a compute warp
// reads its 512 contiguous bytes conflict-free in any slot order).  The slot
// holds {b0, b1} of k-step 0 and {b0, b1} of k-step 1 for column g.
// ----------------------------------------------------------------------------
template <int C, bool RG, int TPC, bool UP>
__global__ void __launch_bounds__(MmaCfg<C, TPC, RG, UP>::THREADS, 1) mma_kernel(const MmaArgs a) {
  using S = MmaCfg<C, TPC, RG, UP>;
  constexpr int NT = S::THREADS;
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
  // 4 row-group pairs x 4 K slices (8 row groups x 2 K slices with three or
  // four column groups)
  // TPC = 2: the CTA takes global tiles 2 blockIdx.x and 2 blockIdx.x + 1 (the
  // second when it exists) over the whole K; its warps cover the same row
  // groups of both, and the converted activations serve both.  Gated
  // launches pair tile blockIdx.x of the gate weight with the same tile of
  // the up weight instead.
  const int gtile = RG ? (int)(blockIdx.x >> 2) : (a.gated ? (int)blockIdx.x : (int)blockIdx.x * TPC);
  const int gtile_b = a.gated ? (int)blockIdx.x + a.gated : gtile + 1;  // the second tile
  int wi = 0;
#pragma unroll
  for (int i = 1; i < MMA_GROUP_MAX; ++i)
    if (i < a.nweights && gtile >= a.w[i].tile_start) wi = i;
  const int64_t tile = (int64_t)gtile - a.w[wi].tile_start;  // tile within its weight
  const bool has1 = TPC == 2 && (int64_t)gtile_b < a.e.N_pad / TILE_N;  // second tile
  int wi1 = wi;
#pragma unroll
  for (int i = 1; i < MMA_GROUP_MAX; ++i)
    if (i < a.nweights && gtile_b >= a.w[i].tile_start) wi1 = i;
  const int64_t tile1 = (int64_t)gtile_b - a.w[wi1].tile_start;
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
  // the next pair of this warp's K slice to fetch, and its sources (running
  // pointers; past the end nothing is dereferenced: every copy is predicated)
  int fnext = 0;
  const uint4* wsrc = wp;
  const uint4* wsrc1 = wp1;
  const uint8_t* ssrc = sp;
  const uint8_t* ssrc1 = sp1;
  auto fetch = [&]() {  // pair fnext into slot fnext % WD
    const uint32_t ok = fnext < n_i;
    const uint32_t d = wring + (uint32_t)(fnext % WD) * (S::WSLOT * TPC);
    cp_async16_if(d + lane * 16, wsrc, ok);
    if (NRG == 2) cp_async16_if(d + 512u + lane * 16, wsrc + 32, ok);
    cp_async16_if(d + S::WSCL + lane * 16, ssrc, ok & (uint32_t)(lane < 4 * NRG));
    if (TPC == 2) {
      const uint32_t ok1 = ok & (uint32_t)has1;
      cp_async16_if(d + S::WSLOT + lane * 16, wsrc1, ok1);
      cp_async16_if(d + S::WSLOT + 512u + lane * 16, wsrc1 + 32, ok1);
      cp_async16_if(d + S::WSLOT + 1024u + lane * 16, ssrc1, ok1 & (uint32_t)(lane < 8));
      wsrc1 += WSTEP;
      ssrc1 += SSTEP;
    }
    asm volatile("cp.async.commit_group;" ::: "memory");  // one group per pair, empty or not
    wsrc += WSTEP;
    ssrc += SSTEP;
    ++fnext;
  };
  // first weight pairs: at entry (weights never depend on an earlier kernel),
  // or with up-front conversion once the activation loads are issued (ahead
  // of them they delay the conversion)
  if (!UP && compute) {
#pragma unroll
    for (int u = 0; u < WD; ++u) fetch();
  }

  // B columns of token rows beyond the launch's are never written: an MMA
  // output column depends on its own B column only, and the outputs of those
  // columns are never read
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

  if constexpr (UP) {
   if (a.xpre != nullptr) {
    // ---- activations converted by the pre-conversion pass ----
    // weight pairs first (they never depend on an earlier kernel), then this
    // split's chunk slots of the image, copied as they are
    if (compute) {
#pragma unroll
      for (int u = 0; u < WD; ++u) fetch();
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the image comes from the previous kernel
    const uint8_t* src = a.xpre + (int64_t)split * a.xpre_stride;
    const int nbytes = nchunks * S::SLOT;
    for (int o = tid * 16; o < nbytes; o += NT * 16) cp_async16(smem_u32(smem + o), src + o);
    asm volatile("cp.async.commit_group;" ::: "memory");
    asm volatile("cp.async.wait_all;" ::: "memory");
    __syncthreads();
   } else {
    // ---- every thread: the activations of all chunks, straight from x ----
    // 128 threads per chunk (k = 4ct .. 4ct + 3), five chunk sets; every load
    // is issued before any is used
    asm volatile("griddepcontrol.wait;" ::: "memory");  // x may come from the previous kernel
    constexpr int CSETS = NT / 128;
    constexpr int PER = (UP_CHUNKS + CSETS - 1) / CSETS;
    const int ct = tid & 127, cset = tid >> 7;
    const int pc = ct >> 4, h = (ct >> 3) & 1, j = (ct >> 1) & 3, tql = 2 * (ct & 1);
    const int kbase = (pc * C * 2 + h) * 512 + j * 4;
    const int s2 = pc & 1;
    const int oa = ((tql) ^ h) * 16, ob = ((tql + 1) ^ h) * 16;
    // row m of this launch: x row xrows[m] when a row list is given (checked:
    // an index outside [0, x_rows) reads zeros and sets STATUS_BAD_ROW)
    auto row_off = [&](int m) -> int64_t {
      if (a.xrows == nullptr) return (int64_t)m * a.K;
      const int32_t r = __ldg(a.xrows + m);
      if (r >= 0 && (int64_t)r < a.x_rows) return (int64_t)r * a.K;
      if (tid == 0 && split == 0) atomicOr(a.status, STATUS_BAD_ROW);
      return -1;
    };
    const float* xr = a.x + bp0 * 64 + 4 * ct;
    // batches of (chunk, up to 4 rows); every batch's loads are issued, then
    // the first weight pairs, then the batches are converted
    constexpr int MG = MAXM < 4 ? MAXM : 4;
    constexpr int NB = PER * (MAXM / MG);
    auto load_batch = [&](int b, float4 (&v)[MG]) {
      const int q = b / (MAXM / MG), m0 = (b % (MAXM / MG)) * MG;
      const int c = cset + q * CSETS;
      const bool k_ok = c < nchunks && c * CHUNK_PAIRS + pc < npairs &&
                        (bp0 + (int64_t)c * CHUNK_PAIRS) * 64 + 4 * ct < a.K;
#pragma unroll
      for (int mm = 0; mm < MG; ++mm) {
        v[mm] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        if (k_ok && m0 + mm < mrows) {
          const int64_t off = row_off(m0 + mm);
          if (off >= 0) v[mm] = __ldg(reinterpret_cast<const float4*>(xr + off + (int64_t)c * CHUNK_K));
        }
      }
    };
    float4 vall[NB][MG];
#pragma unroll
    for (int b = 0; b < NB; ++b) load_batch(b, vall[b]);
    if (compute) {
#pragma unroll
      for (int u = 0; u < WD; ++u) fetch();
    }
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      const float4 (&vc)[MG] = vall[b];
      const int q = b / (MAXM / MG), m0 = (b % (MAXM / MG)) * MG;
      const int c = cset + q * CSETS;
      if (c < nchunks && m0 < mrows) {  // the same for the whole warp
        uint8_t* sb = smem + c * S::SLOT;
        const bool pair_ok = c * CHUNK_PAIRS + pc < npairs;
#pragma unroll
        for (int mm = 0; mm < MG; ++mm) {
          const int m = m0 + mm;
          if (m >= mrows) break;  // the same for every thread of the CTA
          convert_row4<C>(vc[mm], m, sb, kbase, s2, oa, ob, pc, (ct & 15) == 0, pair_ok);
        }
      }
    }
    __syncthreads();
   }
  }

  // accumulators [tile][rg][cg][row R0 / R1] as {column 2tq, column 2tq + 1}
  // pairs (packed fp32x2 updates)
  static_assert(!(R1 && RG), "row-group CTAs have two row groups per warp");
  unsigned long long acc[TPC][NRG][C][2];
#pragma unroll
  for (int tt = 0; tt < TPC; ++tt)
#pragma unroll
    for (int r = 0; r < NRG; ++r)
#pragma unroll
      for (int cg = 0; cg < C; ++cg) acc[tt][r][cg][0] = acc[tt][r][cg][1] = 0ull;

  if (compute) {
    const int g = lane >> 2, tq = lane & 3;
    const int lsw0 = (lane ^ ((sl & 1) * 4)) * 16;        // slot of this lane, h = 0
    const int lsw1 = (lane ^ ((sl & 1) * 4 + 1)) * 16;    // h = 1
    // the 16-byte words and scales of pair i of this warp, once they are in
    // (this lane's groups complete in order, WD - 1 may still fly; the warp
    // barrier makes lanes 0..7's scale copies visible to all lanes)
    auto load_pair = [&](int i, int tt, uint4 (&w)[2], uint2 (&sv)[2]) {
      if (tt == 0) {
        asm volatile("cp.async.wait_group %0;" ::"n"(WD - 1) : "memory");
        __syncwarp();
      }
      const uint8_t* srcp = smem + S::WR_OFF + warp * (WD * S::WSLOT * TPC) + (i % WD) * (S::WSLOT * TPC) +
                            tt * S::WSLOT;
#pragma unroll
      for (int r = 0; r < NRG; ++r) {
        w[r] = *reinterpret_cast<const uint4*>(srcp + r * 512 + lane * 16);
        sv[r] = *reinterpret_cast<const uint2*>(srcp + S::WSCL + r * 64 + g * 8);
      }
    };
#if Q4MM_UNROLL == 2
#pragma unroll 2
#elif Q4MM_UNROLL == 4
#pragma unroll 4
#endif
    for (int i = 0; i < n_i; ++i) {
      // chunk of this pair: slice sl's pairs are sl + NSL i
      const int c = RG ? 2 * i + (sl >> 3) : (R1 ? (i >> 2) : (i >> 1));
      const int slot = UP ? c : (c & (NSLOT - 1));
      if (!UP && (RG || (R1 ? (i & 3) == 0 : (i & 1) == 0)) &&
          !mbar_wait_bounded(smem_u32(&bfull[slot]), (uint32_t)((c / NSLOT) & 1), &s_err, a.wait_ns)) {
        s_err = 1;
        break;
      }
      const int pc = RG ? (sl & 7) : (R1 ? sl + 2 * (i & 3) : sl + 4 * (i & 1));  // pair within the chunk
      const uint8_t* sb = smem + slot * S::SLOT;
      // {1/s, 1/s} and {1/(16 s), 1/(16 s)} of token row 4 cg + tq (the
      // lane's two columns are that row's two terms; rows beyond the launch's
      // are not written: their columns are never read back)
      const uint8_t* sigp = sb + S::SIG_OFF + (pc * MAXM + tq) * 16;
#pragma unroll
      for (int tt = 0; tt < TPC; ++tt) {
        if (tt == 1 && !has1) break;  // the same for every thread of the CTA
        uint4 w[2];
        uint2 sv[2];  // .x = d(R0, b0), d(R0, b1); .y = d(R1, b0), d(R1, b1)
        load_pair(i, tt, w, sv);
        // this pair's sum d_0 D_0 + d_1 D_1 per [rg][cg][R0 / R1]
        unsigned long long pp[NRG][C][2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t af[NRG][2][4];  // [rg][k-step][register]
#pragma unroll
          for (int r = 0; r < NRG; ++r) {
            unpack_word(h ? w[r].z : w[r].x, af[r][0]);
            unpack_word(h ? w[r].w : w[r].y, af[r][1]);
          }
          // refill the slot once every lane has unpacked its words (the
          // shared loads have completed, so the copy cannot overtake them);
          // with two tiles, after the second tile's words (or the first's
          // when there is no second)
          if (h == 1 && (TPC == 1 || tt == 1 || !has1)) {
            __syncwarp();
            fetch();  // pair i + WD
          }
          unsigned long long dd[NRG][2];
#pragma unroll
          for (int r = 0; r < NRG; ++r) {
            const __half2* q = reinterpret_cast<const __half2*>(&sv[r]);
            dd[r][0] = dup2(h ? __high2float(q[0]) : __low2float(q[0]));
            dd[r][1] = dup2(h ? __high2float(q[1]) : __low2float(q[1]));
          }
          const uint8_t* bb = sb + (pc * C * 2 + h) * 512 + (h ? lsw1 : lsw0);
#pragma unroll
          for (int cg = 0; cg < C; ++cg) {
            const uint4 bf = *reinterpret_cast<const uint4*>(bb + cg * 1024);
#pragma unroll
            for (int r = 0; r < NRG; ++r) {
              float d[4];
              mma_f16_first(d, af[r][0], bf.x, bf.y);
              mma_f16_acc(d, af[r][1], bf.z, bf.w);
              if (h == 0) {
                pp[r][cg][0] = fmul2(dd[r][0], d[0], d[1]);
                pp[r][cg][1] = fmul2(dd[r][1], d[2], d[3]);
              } else {
                ffma2(pp[r][cg][0], dd[r][0], d[0], d[1]);
                ffma2(pp[r][cg][1], dd[r][1], d[2], d[3]);
              }
            }
          }
        }
        // acc += P / s (rows R1 also / 16)
#pragma unroll
        for (int cg = 0; cg < C; ++cg) {
          unsigned long long s0, s1;
          {
            const ulonglong2 sg = *reinterpret_cast<const ulonglong2*>(sigp + cg * 64);
            s0 = sg.x;
            s1 = sg.y;
          }
#pragma unroll
          for (int r = 0; r < NRG; ++r) {
            ffma2p(acc[tt][r][cg][0], s0, pp[r][cg][0]);
            ffma2p(acc[tt][r][cg][1], s1, pp[r][cg][1]);
          }
        }
      }
      if (!UP && (RG || (R1 ? (i & 3) == 3 : (i & 1))) && c + NSLOT < nchunks) {  // this warp is done with the slot
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bempty[slot]));
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");  // no copy into the ring outlives the loop
    // arrival number for the split-K epilogue (up-front conversion: drawn by
    // the first compute warp at the end of its loop, so CTAs draw in about
    // the order they finish)
    if (UP && tid == 0 && a.e.splits > 1 && !a.cluster) s_arrival = split_arrive(&a.e.counters[blockIdx.x]);
  } else if constexpr (!UP) {
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
      if (a.stall) break;  // (test setting) no chunk is handed over: the compute warps' waits run out
      const int slot = c & (NSLOT - 1);
      uint8_t* sb = smem + slot * S::SLOT;
      const uint8_t* xs = smem + S::XRAW_OFF + (c % S::XSTAGES) * S::XSLOT;
      const bool pair_ok = c * CHUNK_PAIRS + pc < npairs;
      const bool k_ok = pair_ok && (bp0 + (int64_t)c * CHUNK_PAIRS) * 64 + 4 * ct < a.K;
      // chunk c staged (the next XLEAD - 1 may be in flight)
      asm volatile("cp.async.wait_group %0;" ::"n"(XLEAD - 1) : "memory");
      stage(c + XLEAD);  // refills the slot read in the previous iteration
      if (c >= NSLOT &&
          !mbar_wait_bounded(smem_u32(&bempty[slot]), (uint32_t)(((c / NSLOT) + 1) & 1), &s_err, a.wait_ns)) {
        s_err = 1;
        break;
      }
      constexpr int MG = MAXM < 4 ? MAXM : 4;  // rows read back together
#pragma unroll
      for (int m0 = 0; m0 < MAXM; m0 += MG) {
        if (m0 >= mrows) break;  // the same for every thread of the CTA
        float4 v[MG];
        uint32_t u[MG];
#pragma unroll
        for (int mm = 0; mm < MG; ++mm) {
          v[mm] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
          if (m0 + mm < mrows && k_ok && xoff[m0 + mm] >= 0)
            v[mm] = *reinterpret_cast<const float4*>(xs + (m0 + mm) * (CHUNK_K * 4) + ct * 16);
          // largest |x| of the four (as bits: non-negative floats order like integers)
          u[mm] = __float_as_uint(fmaxf(fmaxf(fabsf(v[mm].x), fabsf(v[mm].y)), fmaxf(fabsf(v[mm].z), fabsf(v[mm].w))));
        }
        // the largest |x| per row over the warp's 128 elements (two block
        // pairs), one warp-wide reduction per row
#pragma unroll
        for (int mm = 0; mm < MG; ++mm)
          if (m0 + mm < mrows) asm volatile("redux.sync.max.u32 %0, %0, 0xffffffff;" : "+r"(u[mm]));
#pragma unroll
        for (int mm = 0; mm < MG; ++mm) {
          const int m = m0 + mm;
          if (m >= mrows) break;
          // s = 2^e with e = 14 - floor(log2 max|x|), kept within [-120, 120]:
          // |x s| < 2^15 for every finite x
          int e = 14 - ((int)(u[mm] >> 23) - 127);
          e = max(-120, min(120, e));
          const float s = __int_as_float((e + 127) << 23);
          if (pair_ok) {
            uint32_t ta[TERMS], tb[TERMS];
            split4(v[mm], s, ta, tb);
#pragma unroll
            for (int t = 0; t < TERMS; ++t) {
              const int col = TERMS * m + t;
              const int cg = col >> 3, gl = col & 7;
              uint8_t* base = sb + kbase + cg * 1024 + (gl ^ s2) * 64;
              *reinterpret_cast<uint32_t*>(base + oa) = ta[t];
              *reinterpret_cast<uint32_t*>(base + ob) = tb[t];
            }
            if ((ct & 15) == 0) {
              // 1/s, and 1/(16 s) for rows R1 (exact powers of two)
              const float r1 = __int_as_float((127 - e) << 23);
              const float r16 = __int_as_float((123 - e) << 23);
              *reinterpret_cast<float4*>(sb + S::SIG_OFF + (pc * MAXM + m) * 16) = make_float4(r1, r1, r16, r16);
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
    if (tid == 0) {
      atomicOr(a.status, STATUS_TIMEOUT);
      // the split-K counter still moves on to the next launch's epoch
      if (a.e.splits > 1 && arrival_last(s_arrival, a.e.splits))
        a.e.counters[blockIdx.x] = arrival_next(s_arrival);
    }
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
              const float2 pr = split2(acc[tt][r][cg][e >> 1]);
              red[sl * RS + (cg * 8 + 2 * tq + (e & 1)) * T2_LD + tt * TILE_N + (2 * rgp + r) * 16 + g +
                  8 * (e >> 1)] = (e & 1) ? pr.y : pr.x;
            }
    }
    __syncthreads();
    if (a.e.idx != nullptr) {
      // greedy pick: per tile, thread tid owns row tid % 128 for token rows
      // tid / 128 + 5k (as on the one-tile path), then the tile's maximum
      constexpr int MG = NT / TILE_N;
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
            float v = 0.0f;
#pragma unroll
            for (int t = 0; t < TERMS; ++t)
#pragma unroll
              for (int s = 0; s < SLICES; ++s) v += red[s * RS + (TERMS * m + t) * T2_LD + tt * TILE_N + row];
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
    if (a.gated) {
      // h = SiLU(g) * u for the tile's 128 rows: thread t < 512 takes row
      // t % 128 and token rows t / 128 + 4k; g and u are added up in the
      // same order as on the ungated path, so they carry the same bits
      if (tid < 4 * TILE_N) {
        const int row = tid & (TILE_N - 1);
        const int64_t n = tile * TILE_N + row;
        float* h = a.w[0].y;
        const int64_t N = a.w[0].N;
        if (n < N) {
          for (int m = tid >> 7; m < mrows; m += 4) {
            float g = 0.0f, u = 0.0f;
#pragma unroll
            for (int t = 0; t < TERMS; ++t)
#pragma unroll
              for (int s = 0; s < SLICES; ++s) g += red[s * RS + (TERMS * m + t) * T2_LD + row];
#pragma unroll
            for (int t = 0; t < TERMS; ++t)
#pragma unroll
              for (int s = 0; s < SLICES; ++s) u += red[s * RS + (TERMS * m + t) * T2_LD + TILE_N + row];
            h[(int64_t)m * N + n] = g / (1.0f + expf(-g)) * u;
          }
        }
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
            float v = 0.0f;
#pragma unroll
            for (int t = 0; t < TERMS; ++t)
#pragma unroll
              for (int s = 0; s < SLICES; ++s) v += red[s * RS + (TERMS * m + t) * T2_LD + row];
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
            const float2 pr = split2(acc[0][r][cg][e >> 1]);
            red[sl * RS + (cg * 8 + 2 * tq + (e & 1)) * RG_LD + r * 16 + g + 8 * (e >> 1)] =
                (e & 1) ? pr.y : pr.x;
          }
    }
    __syncthreads();
    // thread: row tid % 32 of the pair, token rows tid / 32 + 20k; fixed order
    // of terms and slices, as on the split path
    const int row = tid & 31;
    const int64_t n = tile * TILE_N + rgp * 32 + row;
    float* y = a.w[wi].y;
    if (n < a.w[wi].N) {
      for (int m = tid >> 5; m < mrows; m += NT / 32) {
        float v = 0.0f;
#pragma unroll
        for (int t = 0; t < TERMS; ++t)
#pragma unroll
          for (int s = 0; s < NSL; ++s) v += red[s * RS + (TERMS * m + t) * RG_LD + row];
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
          const float2 pr = split2(acc[0][r][cg][e >> 1]);
          red[sl * RS + (cg * 8 + 2 * tq + (e & 1)) * RED_LD + ((R1 ? (warp & 7) : 2 * rgp) + r) * 16 + g +
              8 * (e >> 1)] = (e & 1) ? pr.y : pr.x;
        }
  }
  __syncthreads();

  // all threads take part from here: thread tid owns tile row tid % 128 for
  // the token rows tid / 128 + 5k, so the split-K reads of the last CTA are
  // spread over the whole CTA and issued in a single round
  constexpr int MGROUPS = NT / TILE_N;
  constexpr int MT = (MAXM + MGROUPS - 1) / MGROUPS;
  static_assert(NT % TILE_N == 0, "whole groups of tile rows");
  const int row = tid % TILE_N, mfirst = tid / TILE_N;
  float val[MT];
#pragma unroll
  for (int k = 0; k < MT; ++k) {
    const int m = mfirst + k * MGROUPS;
    val[k] = 0.0f;
    if (m < mrows) {
      float v = 0.0f;
#pragma unroll
      for (int t = 0; t < TERMS; ++t)  // fixed order: term 0, 1, each slice 0..3
#pragma unroll
        for (int s = 0; s < S::NSL; ++s) v += red[s * RS + (TERMS * m + t) * RED_LD + row];
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
      for (int o = split * per + tid; o < o_end; o += NT) {
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
template <int C, bool RG, int TPC, bool UP>
int cluster_capacity(int device, int size) {
  static std::atomic<int> cache[64][9];  // value + 1; 0 = not yet asked
  if (size < 2 || size > 8) return 0;
  std::atomic<int>& slot = cache[device & 63][size];
  const int c = slot.load();
  if (c > 0) return c - 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1, (unsigned)size, 1);
  cfg.blockDim = dim3(MmaCfg<C, TPC, RG, UP>::THREADS);
  cfg.dynamicSmemBytes = MmaCfg<C, TPC, RG, UP>::BYTES;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = (unsigned)size;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, mma_kernel<C, RG, TPC, UP>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  slot.store(n + 1);
  return n;
}

// ---- pre-conversion pass ----
// Converts the activations of one launch once, into the chunk-slot image that
// the up-front launches copy into shared memory: CTA (c, split) writes chunk c
// of K split `split`, with the thread mapping and the operations of the
// up-front conversion (convert_row4), so the image holds the bytes every CTA
// would otherwise compute for itself.
struct XpreArgs {
  const float* x;       // [mrows, K] activations of the launch
  uint8_t* img;         // [splits][chunks] slots, `stride` bytes per split
  int64_t K, KBP, kbp_per_split, stride;
  int mrows;
};

template <int C>
__global__ void __launch_bounds__(128) xpre_kernel(const XpreArgs a) {
  constexpr int MAXM = C * 8 / TERMS;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int ct = threadIdx.x;
  const int c = blockIdx.x, split = blockIdx.y;
  const int64_t bp0 = (int64_t)split * a.kbp_per_split;
  const int64_t bp1 = min(a.KBP, bp0 + a.kbp_per_split);
  const int npairs = (int)(bp1 - bp0);
  const int pc = ct >> 4, h = (ct >> 3) & 1, j = (ct >> 1) & 3, tql = 2 * (ct & 1);
  const int kbase = (pc * C * 2 + h) * 512 + j * 4;
  const int s2 = pc & 1;
  const int oa = ((tql) ^ h) * 16, ob = ((tql + 1) ^ h) * 16;
  const bool pair_ok = c * CHUNK_PAIRS + pc < npairs;
  const bool k_ok = pair_ok && (bp0 + (int64_t)c * CHUNK_PAIRS) * 64 + 4 * ct < a.K;
  uint8_t* sb = a.img + split * a.stride + (int64_t)c * chunk_slot_bytes<C>();
  const float* xr = a.x + (bp0 + (int64_t)c * CHUNK_PAIRS) * 64 + 4 * ct;
  asm volatile("griddepcontrol.wait;" ::: "memory");  // x may come from the previous kernel
  float4 v[MAXM];
#pragma unroll
  for (int m = 0; m < MAXM; ++m) {
    v[m] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    if (k_ok && m < a.mrows) v[m] = __ldg(reinterpret_cast<const float4*>(xr + (int64_t)m * a.K));
  }
#pragma unroll
  for (int m = 0; m < MAXM; ++m) {
    if (m >= a.mrows) break;  // the same for every thread
    convert_row4<C>(v[m], m, sb, kbase, s2, oa, ob, pc, (ct & 15) == 0, pair_ok);
  }
}

// The image of a launch of `splits` K splits of `kbp` block pairs each.
int64_t xpre_split_bytes(int64_t kbp, int C) {
  const int64_t chunks = (kbp + CHUNK_PAIRS - 1) / CHUNK_PAIRS;
  return chunks * (C == 1 ? chunk_slot_bytes<1>() : chunk_slot_bytes<2>());
}

int launch_xpre(int C, const float* x, int mrows, int64_t K, int64_t KBP, int64_t kbp, int splits, uint8_t* img,
                cudaStream_t s) {
  XpreArgs a;
  a.x = x;
  a.img = img;
  a.K = K;
  a.KBP = KBP;
  a.kbp_per_split = kbp;
  a.stride = xpre_split_bytes(kbp, C);
  a.mrows = mrows;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((kbp + CHUNK_PAIRS - 1) / CHUNK_PAIRS), (unsigned)splits, 1);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = C == 1 ? cudaLaunchKernelEx(&cfg, xpre_kernel<1>, a) : cudaLaunchKernelEx(&cfg, xpre_kernel<2>, a);
  return e == cudaSuccess ? Q4_OK : Q4_ERR_CUDA;
}

// True when a launch of `mrows` token rows takes its activations from the
// pre-conversion pass (given scratch for the image): an up-front launch of
// one or two column groups reading x in row order, with at least the rows
// set for its kind.  rg / two: row-group or two-tile CTAs (whole K).
bool takes_xpre(int64_t KBP, const MmaPlan& plan, bool rg, bool two, int mrows, bool row_list) {
  const int cgs = (TERMS * mrows + 7) / 8;
  const int64_t chunks_split = (plan.kbp_per_split + CHUNK_PAIRS - 1) / CHUNK_PAIRS;
  const int64_t chunks_all = (KBP + CHUNK_PAIRS - 1) / CHUNK_PAIRS;
  if (!Q4MM_UPFRONT || cgs > 2 || row_list) return false;
  const int from = rg ? Q4MM_XPRE_RG_ROWS : (two ? Q4MM_XPRE_TWO_ROWS : Q4MM_XPRE_SPLIT_ROWS);
  const bool up = rg ? chunks_all <= UP_CHUNKS
                     : (two ? (Q4MM_UP_TWO && chunks_all <= UP_CHUNKS) : chunks_split <= UP_CHUNKS);
  const int64_t chunks = (rg || two) ? chunks_all : chunks_split;
  return up && from > 0 && mrows >= from && chunks >= Q4MM_XPRE_MIN_CHUNKS;
}

template <int C, bool RG, int TPC = 1, bool UP = false>
int launch_c(const MmaLaunch& L, const float* x, int mrows, int32_t* idx, float* maxval,
             const MmaPlan& plan, const Workspace& ws, int64_t mb, cudaStream_t s,
             const int32_t* xrows, int64_t x_rows, const uint8_t* xpre = nullptr, int64_t xpre_stride = 0) {
  using S = MmaCfg<C, TPC, RG, UP>;
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
  a.gated = L.gated ? (int)L.W[0]->tiles : 0;
  a.xpre = UP ? xpre : nullptr;
  a.xpre_stride = xpre_stride;
  a.status = ws.status;
  a.wait_ns = wait_limit_ns();
  a.stall = stall_for_test();
  a.e.poll_limit = poll_rounds();
  a.e.stall = a.stall;
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
    if (cudaFuncSetAttribute(mma_kernel<C, RG, TPC, UP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
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
              tiles <= cluster_capacity<C, RG, TPC, UP>(W0->device, plan.splits);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = RG ? dim3((unsigned)tiles * 4u, 1, 1)
                   : L.gated ? dim3((unsigned)L.W[0]->tiles, 1, 1)
                             : dim3((unsigned)((tiles + TPC - 1) / TPC), (unsigned)plan.splits, 1);
  cfg.blockDim = dim3(S::THREADS);
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
  return cudaLaunchKernelEx(&cfg, mma_kernel<C, RG, TPC, UP>, a) == cudaSuccess ? Q4_OK : Q4_ERR_CUDA;
}

// Rows per launch: 16 (four column groups of two terms per row) in default
// mode; 8 for launches that run as two-tile CTAs (one or two column groups),
// which stream two tiles per CTA in one wave where 16 rows would need one tile
// per CTA in two waves (measured on GB300 for the gate/up group of a 7B layer,
// two launches of 8 rows / one of 16: 42.6 / 53.0 us at M = 16); 8 for every
// batch-invariant launch (one or two column groups, so that every row count
// runs the same layout).
int rows_per_launch(bool batch_invariant, bool two_tiles = false) {
  return (two_tiles || batch_invariant) ? 8 : MAX_CG * 8 / TERMS;
}

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

size_t mma_xpre_bytes(int64_t KBP, const MmaPlan& p) {
  if (Q4MM_XPRE_RG_ROWS <= 0 && Q4MM_XPRE_SPLIT_ROWS <= 0 && Q4MM_XPRE_TWO_ROWS <= 0) return 0;
  const int64_t whole = xpre_split_bytes(KBP, 2);
  const int64_t split = (int64_t)p.splits * xpre_split_bytes(p.kbp_per_split, 2);
  return (size_t)(whole > split ? whole : split);
}

size_t mma_partial_bytes_tiles(int64_t tiles, const MmaPlan& p, int64_t M, bool batch_invariant) {
  if (p.splits <= 1) return 0;
  const int64_t rpl = rows_per_launch(batch_invariant);
  const int64_t ml = M < rpl ? M : rpl;
  return (size_t)p.splits * (size_t)ml * (size_t)(tiles * TILE_N) * sizeof(unsigned long long);
}

size_t mma_partial_bytes(const Weight* W, const MmaPlan& p, int64_t M, bool batch_invariant) {
  return mma_partial_bytes_tiles(W->tiles, p, M, batch_invariant);
}

bool mma_two_tiles(const MmaPlan& plan, int64_t tiles, bool) {
  return Q4MM_TWO_TILES && plan.splits == 1 && plan.num_sms > 0 && tiles > plan.num_sms;
}

int mma_rows_per_launch(bool batch_invariant, bool two_tiles) { return rows_per_launch(batch_invariant, two_tiles); }

int mma_call_launches(int64_t tiles, int64_t KBP, int64_t K, const MmaPlan& plan, int64_t M, bool batch_invariant,
                      bool greedy_pick) {
  const bool two = mma_two_tiles(plan, tiles, batch_invariant);
  const int64_t rpl = rows_per_launch(batch_invariant, two);
  int n = 0;
  for (int64_t mb = 0; mb < M; mb += rpl) {
    const int mrows = (int)((M - mb) < rpl ? (M - mb) : rpl);
    const bool rg = mma_row_groups(plan, K, batch_invariant, greedy_pick, mrows);
    n += 1 + (takes_xpre(KBP, plan, rg, two, mrows, false) ? 1 : 0);
  }
  return n;
}

int mma_launch_count(int64_t M, bool batch_invariant, bool two_tiles) {
  const int64_t rpl = rows_per_launch(batch_invariant, two_tiles);
  return (int)((M + rpl - 1) / rpl);
}

bool mma_row_groups(const MmaPlan& plan, int64_t K, bool batch_invariant, bool greedy_pick,
                    int64_t launch_rows) {
  (void)batch_invariant;
  return !greedy_pick && launch_rows <= Q4MM_RG_MAX_ROWS && plan.splits >= 4 && K <= Q4MM_RG_MAX_K;
}

int launch_mma_group(const MmaLaunch& L, const float* x, int64_t M, int32_t* idx, float* maxval,
                     const MmaPlan& plan, bool batch_invariant, const Workspace& ws, cudaStream_t s,
                     const int32_t* xrows, int64_t x_rows) {
  int64_t tiles = 0;
  for (int i = 0; i < L.count; ++i) tiles += L.W[i]->tiles;
  if (plan.splits > 1 && tiles > MAX_COUNTERS) return Q4_ERR_SHAPE;
  const int64_t K = L.W[0]->K;
  // row-group CTAs (per launch, below): no K split and so no cross-CTA
  // exchange, when four CTAs per tile fit on the SMs (the split plan has at
  // least 4 splits), K is short and the launch has at most 8 rows; the plan
  // depends on the shapes and that row count only (y output, default mode)
  // two tiles per CTA (whole K, no split): launches of more tiles than SMs
  // run as CTAs that stream two tiles each, for one or two column groups (up
  // to 8 rows) in default mode (y output or the greedy pick)
  const bool two = mma_two_tiles(plan, tiles, batch_invariant);
  const int64_t rpl = rows_per_launch(batch_invariant, two);
  // up-front conversion when every CTA's K range is at most UP_CHUNKS chunks
  // (row-group CTAs cover the whole K).  Measured on GB300 over the 7B layer
  // (8 layer copies per graph, us per call, up-front / converter warps):
  // q/k/v 4.79 / 5.68 at M = 1 and 7.68 / 9.76 at M = 8; down 17.13 / 18.90
  // at M = 8.
  const int64_t chunks_split = (plan.kbp_per_split + CHUNK_PAIRS - 1) / CHUNK_PAIRS;
  const int64_t chunks_all = (L.W[0]->KBP + CHUNK_PAIRS - 1) / CHUNK_PAIRS;
  const bool up_rg = Q4MM_UPFRONT && chunks_all <= UP_CHUNKS;
  const bool up_split = Q4MM_UPFRONT && chunks_split <= UP_CHUNKS;
  const bool up_two = Q4MM_UPFRONT && chunks_all <= UP_CHUNKS;
  for (int64_t mb = 0; mb < M; mb += rpl) {
    const int mrows = (int)((M - mb) < rpl ? (M - mb) : rpl);
    const bool rg = mma_row_groups(plan, K, batch_invariant, idx != nullptr || xrows != nullptr, mrows);
    const float* xs = xrows ? x : x + mb * K;
    const int32_t* xr = xrows ? xrows + mb : nullptr;
    int st;
    // batch-invariant mode takes the same kernels as the default mode in
    // launches of at most 8 rows (one or two column groups): their layout
    // depends on the shapes only (row-group, two-tile or split CTAs, the K
    // partition of the shapes), every MMA output column depends on its own B
    // column only, and a column's scaling, slice and split sums are the same
    // operations in the same order whatever the column count
    const int cgs = (TERMS * mrows + 7) / 8;  // column groups of this launch
    // up-front launches take their activations from the pre-conversion pass
    // (takes_xpre) when the scratch holds its image; the slot bytes are the
    // same either way
    const uint8_t* xp = nullptr;
    int64_t xstride = 0;
    if (takes_xpre(L.W[0]->KBP, plan, rg, two, mrows, xrows != nullptr) && ws.xpre != nullptr) {
      const int64_t kbp = (rg || two) ? L.W[0]->KBP : plan.kbp_per_split;
      const int sp = (rg || two) ? 1 : plan.splits;
      const int64_t stride = xpre_split_bytes(kbp, cgs);
      if ((size_t)(stride * sp) <= ws.xpre_bytes) {
        st = launch_xpre(cgs, xs, mrows, K, L.W[0]->KBP, kbp, sp, ws.xpre, s);
        if (st) return st;
        xp = ws.xpre;
        xstride = stride;
      }
    }
    if (cgs >= 3) {  // 9 to 16 rows: one row group per warp, K splits
      st = cgs == 3 ? launch_c<3, false>(L, xs, mrows, idx, maxval, plan, ws, mb, s, xr, x_rows)
                    : launch_c<4, false>(L, xs, mrows, idx, maxval, plan, ws, mb, s, xr, x_rows);
    } else if (rg) {
      if (up_rg) st = cgs == 1 ? launch_c<1, true, 1, true>(L, xs, mrows, idx, maxval, plan, ws, mb, s, xr, x_rows, xp, xstride)
                               : launch_c<2, true, 1, true>(L, xs, mrows, idx, maxval, plan, ws, mb, s, xr, x_rows, xp, xstride);
      else st = cgs == 1 ? launch_c<1, true>(L, xs, mrows, idx, maxval, plan, ws, mb, s, xr, x_rows, xp, xstride)
                         : launch_c<2, true>(L, xs, mrows, idx, maxval, plan, ws, mb, s, xr, x_rows, xp, xstride);
    } else if (two) {
      if (Q4MM_UP_TWO && up_two)
        st = cgs == 1 ? launch_c<1, false, 2, true>(L, xs, mrows, idx, maxval, plan, ws, mb, s, xr, x_rows, xp, xstride)
                      : launch_c<2, false, 2, true>(L, xs, mrows, idx, maxval, plan, ws, mb, s, xr, x_rows, xp, xstride);
      else
        st = cgs == 1 ? launch_c<1, false, 2>(L, xs, mrows, idx, maxval, plan, ws, mb, s, xr, x_rows)
                      : launch_c<2, false, 2>(L, xs, mrows, idx, maxval, plan, ws, mb, s, xr, x_rows);
    } else {
      if (up_split)
        st = cgs == 1 ? launch_c<1, false, 1, true>(L, xs, mrows, idx, maxval, plan, ws, mb, s, xr, x_rows, xp, xstride)
                      : launch_c<2, false, 1, true>(L, xs, mrows, idx, maxval, plan, ws, mb, s, xr, x_rows, xp, xstride);
      else
        st = cgs == 1 ? launch_c<1, false>(L, xs, mrows, idx, maxval, plan, ws, mb, s, xr, x_rows)
                      : launch_c<2, false>(L, xs, mrows, idx, maxval, plan, ws, mb, s, xr, x_rows);
    }
    if (st) return st;
  }
  return Q4_OK;
}

int launch_mma_gated(const Weight* Wg, const Weight* Wu, const float* x, int64_t M, float* h,
                     const Workspace& ws, cudaStream_t s) {
  // two-tile CTAs over the pair (gate tile b, up tile b), whole K, up to 8
  // token rows per launch
  MmaLaunch L;
  L.count = 2;
  L.W[0] = Wg;
  L.W[1] = Wu;
  L.y[0] = h;
  L.y[1] = nullptr;
  L.gated = true;
  MmaPlan plan;
  plan.splits = 1;
  plan.kbp_per_split = Wg->KBP;
  plan.num_sms = 0;
  for (int64_t mb = 0; mb < M; mb += 8) {
    const int mrows = (int)((M - mb) < 8 ? (M - mb) : 8);
    const float* xs = x + mb * Wg->K;
    const int cgs = mrows <= 4 ? 1 : 2;
    const uint8_t* xp = nullptr;
    int64_t xstride = 0;
    if (takes_xpre(Wg->KBP, plan, false, true, mrows, false) && ws.xpre != nullptr &&
        (size_t)xpre_split_bytes(Wg->KBP, cgs) <= ws.xpre_bytes) {
      const int st = launch_xpre(cgs, xs, mrows, Wg->K, Wg->KBP, Wg->KBP, 1, ws.xpre, s);
      if (st) return st;
      xp = ws.xpre;
      xstride = xpre_split_bytes(Wg->KBP, cgs);
    }
    const int st = cgs == 1
        ? launch_c<1, false, 2, true>(L, xs, mrows, nullptr, nullptr, plan, ws, mb, s, nullptr, 0, xp, xstride)
        : launch_c<2, false, 2, true>(L, xs, mrows, nullptr, nullptr, plan, ws, mb, s, nullptr, 0, xp, xstride);
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
