// q4mm_epilogue.cuh — output stage shared by the matmul kernels.
//
// Each CTA ends with the fp32 results of one 128-row tile for up to MAXM
// token rows over its K range.  finish_tile() then
//   - with one K split: writes y (or feeds the greedy pick);
//   - with several: stores its partial sums, and the last CTA of the tile to
//     arrive (an atomic counter; no CTA ever waits for another) adds all the
//     partials in ascending split order, so the sum does not depend on which
//     CTA finished first;
//   - for the greedy pick (§"Same Prompt, Different Story" of "Why Continuous
//     Batching Slowed Down My LLM Inference Engine": greedy decoding takes the
//     largest logit) folds the tile's per-row maximum into a 64-bit key with an
//     atomic max — value in the high word, complemented index in the low word,
//     so equal values prefer the lower index and NaN never wins — and the last
//     tile to arrive writes idx / maxval and resets the keys and counters for
//     the next launch.
#pragma once

#include <cstdint>

#include "q4mm_internal.h"

namespace q4 {

struct EpiArgs {
  int64_t N, N_pad;
  int64_t M;            // token rows in this launch
  float* y;             // [M, N] or null
  int32_t* idx;         // [M] or null (greedy pick instead of y)
  float* maxval;        // [M] or null
  int splits;
  float* partial;       // [splits][M][N_pad]
  unsigned int* counters;
  unsigned long long* keys;  // [M]
  unsigned int* argmax_done;
  int tiles;            // tiles x m-tiles of this launch (greedy-pick completion count)
};

__device__ __forceinline__ unsigned long long argmax_key(float v, uint32_t n) {
  if (v != v) return 0ull;
  if (v == 0.0f) v = 0.0f;  // -0 and +0 are the same logit
  uint32_t u = __float_as_uint(v);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((unsigned long long)u << 32) | (unsigned long long)(0xFFFFFFFFu - n);
}

__device__ __forceinline__ float key_value(unsigned long long k) {
  const uint32_t u = (uint32_t)(k >> 32);
  if (u == 0u) return __uint_as_float(0x7FC00000u);
  return __uint_as_float((u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u);
}

// Called by every thread of the participating group; `row` in [0, 128) for
// the 128 threads that own the tile's rows and -1 for the others (they only
// take part in the barriers).  `sync` is a barrier over the whole group.
// `val[m]` holds the result of row `row` for token row m0 + m (m < mcount).
// `counter_slot` identifies (tile, m-tile) among this launch's counters.
template <int MAXM, class Sync>
__device__ __forceinline__ void finish_tile(const EpiArgs& e, float (&val)[MAXM], int row,
                                            int64_t tile, int64_t m0, int mcount, int split,
                                            int counter_slot, int* s_flag,
                                            unsigned long long (*red)[MAXM], Sync sync) {
  const int64_t n = tile * TILE_N + row;
  if (e.splits > 1) {
    if (row >= 0) {
#pragma unroll
      for (int m = 0; m < MAXM; ++m)
        if (m < mcount) e.partial[((int64_t)split * e.M + m0 + m) * e.N_pad + n] = val[m];
      __threadfence();  // the writers' partial sums are visible before the count
    }
    sync();
    if (row == 0) {
      const unsigned prev = atomicAdd(&e.counters[counter_slot], 1u);
      *s_flag = (prev == (unsigned)(e.splits - 1));
    }
    sync();
    if (!*s_flag) return;
    if (row >= 0) {
      __threadfence();
      // ascending split order per output; the loads of a batch of splits for
      // every token row are issued before any of them is added
      constexpr int SB = MAXM <= 2 ? 8 : (MAXM <= 5 ? 4 : 2);  // splits loaded per batch
      const int64_t sstride = e.M * e.N_pad;
      const float* pp = e.partial + (m0 * e.N_pad + n);
#pragma unroll
      for (int m = 0; m < MAXM; ++m) val[m] = 0.0f;
      for (int s0 = 0; s0 < e.splits; s0 += SB) {
        float t[MAXM][SB];
#pragma unroll
        for (int m = 0; m < MAXM; ++m)
#pragma unroll
          for (int j = 0; j < SB; ++j)
            t[m][j] = (m < mcount && s0 + j < e.splits)
                          ? __ldcg(pp + (int64_t)(s0 + j) * sstride + (int64_t)m * e.N_pad)
                          : 0.0f;
#pragma unroll
        for (int m = 0; m < MAXM; ++m)
#pragma unroll
          for (int j = 0; j < SB; ++j)
            if (s0 + j < e.splits) val[m] += t[m][j];
      }
    }
    if (row == 0) e.counters[counter_slot] = 0u;  // ready for the next launch
  }

  if (e.idx == nullptr) {
    if (row >= 0 && n < e.N) {
#pragma unroll
      for (int m = 0; m < MAXM; ++m)
        if (m < mcount) e.y[(m0 + m) * e.N + n] = val[m];
    }
    return;
  }

  // greedy pick: tile maximum per token row, then a global atomic max
  const int lane = threadIdx.x & 31;
  const int wq = row >= 0 ? (row >> 5) : -1;
#pragma unroll
  for (int m = 0; m < MAXM; ++m) {
    unsigned long long k =
        (row >= 0 && m < mcount && n < e.N) ? argmax_key(val[m], (uint32_t)n) : 0ull;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const unsigned long long o = __shfl_xor_sync(0xFFFFFFFFu, k, off);
      k = o > k ? o : k;
    }
    if (wq >= 0 && lane == 0) red[wq][m] = k;
  }
  sync();
  if (row >= 0 && row < mcount) {
    unsigned long long k = red[0][row];
#pragma unroll
    for (int w = 1; w < 4; ++w) k = red[w][row] > k ? red[w][row] : k;
    atomicMax(&e.keys[m0 + row], k);
  }
  __threadfence();
  sync();
  if (row == 0) {
    const unsigned prev = atomicAdd(e.argmax_done, 1u);
    *s_flag = (prev == (unsigned)(e.tiles - 1));
  }
  sync();
  if (!*s_flag) return;
  __threadfence();
  if (row >= 0) {
    for (int64_t m = row; m < e.M; m += TILE_N) {
      const unsigned long long k = atomicExch(&e.keys[m], 0ull);
      e.idx[m] = k == 0ull ? 0 : (int32_t)(0xFFFFFFFFu - (uint32_t)(k & 0xFFFFFFFFull));
      if (e.maxval) e.maxval[m] = key_value(k);
    }
  }
  if (row == 0) *e.argmax_done = 0u;
}

}  // namespace q4
