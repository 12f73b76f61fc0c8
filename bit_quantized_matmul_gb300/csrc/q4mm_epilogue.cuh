// q4mm_epilogue.cuh — output stage shared by the matmul kernels.
//
// Each CTA ends with the fp32 results of one 128-row tile for up to MAXM
// token rows over its K range.  finish_tile() then
//   - with one K split: writes y (or feeds the greedy pick);
//   - with several: the CTAs of a tile draw arrival numbers from the tile's
//     counter (the kernels draw them early, as soon as they start).  Every
//     CTA but the one with the last number stores its partial sums, each
//     value in one 64-bit word together with a launch flag, and is done: no
//     fence, no wait.  The CTA with the last number polls its peers' words
//     until every flag is the one of this launch (a bounded wait; the peers
//     all drew their numbers, so all of them are running and none waits for
//     anything) and adds the partials in ascending split order, so the sum
//     does not depend on which CTA finished first.  It clears the words it
//     read and advances the counter's epoch for the next launch;
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
  unsigned long long* partial;  // [splits][M][N_pad] flagged words, zero when idle
  unsigned int* counters;  // split-K arrival words, one per slot
  unsigned int* status;    // device status word (STATUS_TIMEOUT)
  unsigned long long* keys;  // [M]
  unsigned int* argmax_done;
  int tiles;            // tiles x m-tiles of this launch (greedy-pick completion count)
  unsigned poll_limit;  // rounds of re-reads of a batch of partial sums before giving up
  int stall;            // test setting: CTAs that are not last leave their partial sums unstored
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

// Split-K arrival word, one per slot (tile, or tile and token tile): the low
// ARRIVAL_BITS count the CTAs of the running launch that arrived, the bits
// above are the slot's epoch, advanced once per launch that uses the slot.
// The flag of a partial-sum word is the epoch with the top bit set, so it is
// never zero, and idle words are zero.
constexpr int ARRIVAL_BITS = 10;
constexpr int MAX_SPLITS = (1 << ARRIVAL_BITS) - 1;

__device__ __forceinline__ unsigned split_arrive(unsigned* counter) {
  return atomicAdd(counter, 1u);
}
__device__ __forceinline__ bool arrival_last(unsigned word, int splits) {
  return (int)(word & ((1u << ARRIVAL_BITS) - 1u)) == splits - 1;
}
__device__ __forceinline__ unsigned arrival_flag(unsigned word) {
  return (word >> ARRIVAL_BITS) | 0x80000000u;
}
__device__ __forceinline__ unsigned arrival_next(unsigned word) {
  return ((word >> ARRIVAL_BITS) + 1u) << ARRIVAL_BITS;  // next epoch, no arrivals
}

// flag in the high word, the fp32 bits in the low word: one single-copy
// atomic 64-bit access carries both
__device__ __forceinline__ void st_flagged(unsigned long long* p, unsigned flag, float v) {
  const unsigned long long w = ((unsigned long long)flag << 32) | __float_as_uint(v);
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}
__device__ __forceinline__ unsigned long long ld_flagged(const unsigned long long* p) {
  unsigned long long w;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(w) : "l"(p) : "memory");
  return w;
}

// Called by every thread of the participating group; `row` in [0, 128) for
// the threads that own one of the tile's rows and -1 for the others (they
// only take part in the barriers).  `sync` is a barrier over the whole
// group.  A row's token rows may be spread over several threads: the thread
// holds in val[k] the result of row `row` for token row m0 + mfirst +
// k * MSTRIDE (counted when that is below mcount); every token row belongs to
// one thread per tile row, and the thread with mfirst = 0 also does the
// single-thread steps.  `red` has a column per token row of the call (MAXM).
// `arrival` is the CTA's arrival word for this tile (any value with one K
// split); the CTA with the last arrival resets the word at `counter_slot`
// when that is >= 0 (the last call for the slot in this CTA).
template <int MT, int MSTRIDE, int MAXM, class Sync>
__device__ __forceinline__ void finish_tile(const EpiArgs& e, float (&val)[MT], int row, int mfirst,
                                            int64_t tile, int64_t m0, int mcount, int split,
                                            unsigned arrival, int counter_slot, int* s_flag,
                                            unsigned long long (*red)[MAXM], Sync sync) {
  const int64_t n = tile * TILE_N + (row >= 0 ? row : 0);
  const bool lead = row >= 0 && mfirst == 0;
  auto owned = [&](int k) { return row >= 0 && mfirst + k * MSTRIDE < mcount; };
  if (e.splits > 1) {
    const unsigned flag = arrival_flag(arrival);
    const int64_t sstride = e.M * e.N_pad;
    unsigned long long* pp = e.partial + ((m0 + mfirst) * e.N_pad + n);
    constexpr int64_t KSTEP = MSTRIDE;  // token rows between a thread's values
    if (!arrival_last(arrival, e.splits)) {
      if (e.stall) return;  // (test setting) the last CTA then waits for words nothing writes
#pragma unroll
      for (int k = 0; k < MT; ++k)
        if (owned(k)) st_flagged(pp + (int64_t)split * sstride + k * KSTEP * e.N_pad, flag, val[k]);
      return;
    }
    // ascending split order per output, this CTA's own sums in its place;
    // the reads of a batch of splits for every value are issued together and
    // whatever is not yet from this launch is read again in the next round
    constexpr int SB = MT <= 1 ? 16 : (MT <= 2 ? 8 : (MT <= 5 ? 4 : 2));  // splits per batch
    float own[MT];
#pragma unroll
    for (int k = 0; k < MT; ++k) {
      own[k] = val[k];
      val[k] = 0.0f;
    }
    unsigned rounds = 0;
    for (int s0 = 0; s0 < e.splits; s0 += SB) {
      auto peer = [&](int k, int j) { return owned(k) && s0 + j < e.splits && s0 + j != split; };
      auto addr = [&](int k, int j) { return pp + (int64_t)(s0 + j) * sstride + k * KSTEP * e.N_pad; };
      unsigned long long t[MT][SB];
#pragma unroll
      for (int k = 0; k < MT; ++k)
#pragma unroll
        for (int j = 0; j < SB; ++j) t[k][j] = peer(k, j) ? ld_flagged(addr(k, j)) : 0ull;
      for (;;) {
        bool ready = true;
#pragma unroll
        for (int k = 0; k < MT; ++k)
#pragma unroll
          for (int j = 0; j < SB; ++j)
            if (peer(k, j) && (unsigned)(t[k][j] >> 32) != flag) ready = false;
        if (ready || rounds >= e.poll_limit) break;
        ++rounds;
#pragma unroll
        for (int k = 0; k < MT; ++k)
#pragma unroll
          for (int j = 0; j < SB; ++j)
            if (peer(k, j) && (unsigned)(t[k][j] >> 32) != flag) t[k][j] = ld_flagged(addr(k, j));
      }
#pragma unroll
      for (int k = 0; k < MT; ++k)
#pragma unroll
        for (int j = 0; j < SB; ++j) {
          if (peer(k, j)) *addr(k, j) = 0ull;  // idle again
          if (s0 + j < e.splits)
            val[k] += (s0 + j == split) ? own[k] : __uint_as_float((uint32_t)t[k][j]);
        }
    }
    if (rounds >= e.poll_limit) atomicOr(e.status, STATUS_TIMEOUT);
    if (lead && row == 0 && counter_slot >= 0) e.counters[counter_slot] = arrival_next(arrival);
  }

  if (e.idx == nullptr) {
    if (row >= 0 && n < e.N) {
#pragma unroll
      for (int k = 0; k < MT; ++k)
        if (owned(k)) e.y[(m0 + mfirst + k * MSTRIDE) * e.N + n] = val[k];
    }
    return;
  }

  // greedy pick: tile maximum per token row, then a global atomic max
  const int lane = threadIdx.x & 31;
  const int wq = row >= 0 ? (row >> 5) : -1;
#pragma unroll
  for (int k = 0; k < MT; ++k) {
    unsigned long long key = (owned(k) && n < e.N) ? argmax_key(val[k], (uint32_t)n) : 0ull;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const unsigned long long o = __shfl_xor_sync(0xFFFFFFFFu, key, off);
      key = o > key ? o : key;
    }
    const int m = mfirst + k * MSTRIDE;
    if (wq >= 0 && lane == 0 && m < MAXM) red[wq][m] = key;
  }
  sync();
  if (lead && row < mcount) {
    unsigned long long key = red[0][row];
#pragma unroll
    for (int w = 1; w < 4; ++w) key = red[w][row] > key ? red[w][row] : key;
    atomicMax(&e.keys[m0 + row], key);
  }
  __threadfence();
  sync();
  if (lead && row == 0) {
    const unsigned prev = atomicAdd(e.argmax_done, 1u);
    *s_flag = (prev == (unsigned)(e.tiles - 1));
  }
  sync();
  if (!*s_flag) return;
  __threadfence();
  if (lead) {
    for (int64_t m = row; m < e.M; m += TILE_N) {
      const unsigned long long k = atomicExch(&e.keys[m], 0ull);
      e.idx[m] = k == 0ull ? 0 : (int32_t)(0xFFFFFFFFu - (uint32_t)(k & 0xFFFFFFFFull));
      if (e.maxval) e.maxval[m] = key_value(k);
    }
  }
  if (lead && row == 0) *e.argmax_done = 0u;
}

}  // namespace q4
