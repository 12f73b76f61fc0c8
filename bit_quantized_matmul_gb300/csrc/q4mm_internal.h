// q4mm_internal.h — device layout, workspace and launcher declarations shared
// by the library's translation units (not part of the public ABI).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "q4mm.h"

namespace q4 {

// ---------------------------------------------------------------------------
// Device weight layout ("fragment layout").
//
// Rows are grouped in tiles of TILE_N = 128 (N is padded to a multiple of 128
// with zero-scale rows); blocks of 32 weights along K are grouped in pairs
// (KB is padded to an even count with zero blocks).  A tile is 8 row groups
// of 16 rows.  For tile t, block pair bp, row group rg and lane L = 4g + tq
// (g = 0..7, tq = 0..3) there are 16 bytes: four 32-bit words, word 2h + s for
// block b = 2bp + h and k-step s (16 weights of the block).  Lane L holds the
// weights of rows R0 = 16rg + g and R1 = R0 + 8 at k0 = 16s + 2tq, k0 + 1,
// k0 + 8, k0 + 9 of the block.  In each word, nibble pair p (bits 4p..4p+3 and
// 16+4p..19+4p) holds row (p & 1 ? R1 : R0) at k = k0 + 8(p >> 1) and k + 1.
// So (w >> 4p) & 0x000F000F is pair p, and pairs 0..3 are exactly the A
// fragment registers a0..a3 of an m16n8k16 MMA over that k-step.  The 16-byte
// groups of a (tile, block pair) are contiguous (4 KB), so a warp's 32 lanes
// read 512 consecutive bytes and consecutive block pairs of a tile are one
// contiguous range.
//
// Scales: for tile t, block pair bp, row group rg and g, four binary16 values
// (8 bytes): d(R0, 2bp), d(R0, 2bp+1), d(R1, 2bp), d(R1, 2bp+1); 512 bytes per
// (tile, block pair).
// ---------------------------------------------------------------------------
constexpr int TILE_N = 128;
constexpr int BLOCK_K = 32;
constexpr int CANON_BLOCK_BYTES = 18;
constexpr int PAIR_NIB_BYTES = 4096;   // nibbles of one (tile, block pair)
constexpr int PAIR_SCL_BYTES = 512;    // scales of one (tile, block pair)

inline int64_t pad_n(int64_t N) { return (N + TILE_N - 1) / TILE_N * TILE_N; }

// 32-bit word index of (tile t, block pair bp, row group rg, lane, half h, k-step s).
__host__ __device__ inline int64_t nib_word_index(int64_t KBP, int64_t t, int64_t bp, int rg, int lane,
                                                  int h, int s) {
  return ((((t * KBP + bp) * 8 + rg) * 32 + lane) * 4) + h * 2 + s;
}

// binary16 index of the scale of (tile t, block pair bp, row group rg, g, upper, h).
__host__ __device__ inline int64_t scale_index(int64_t KBP, int64_t t, int64_t bp, int rg, int g,
                                               int upper, int h) {
  return ((((t * KBP + bp) * 8 + rg) * 8 + g) * 4) + upper * 2 + h;
}

struct Weight {
  int64_t N = 0, K = 0, N_pad = 0, KB = 0, KBP = 0, tiles = 0;
  int device = 0;
  uint8_t* nib = nullptr;   // tiles * KBP * 4096 bytes (fragment layout)
  uint16_t* d = nullptr;    // tiles * KBP * 256 binary16 scales
  void* alloc = nullptr;    // single allocation backing nib and d
  size_t alloc_bytes = 0;
};

// Per-device scratch shared by all handles on that device.
struct Workspace {
  unsigned int* status = nullptr;      // device status word: STATUS_* bits
  unsigned int* counters = nullptr;    // split-K arrival counters, self-resetting
  unsigned long long* keys = nullptr;  // argmax keys [Q4MM_M_MAX], self-resetting
  unsigned int* argmax_done = nullptr; // argmax completion counter
  unsigned long long* partial = nullptr;  // split-K partial sums (flagged words, zero when idle)
  size_t partial_bytes = 0;
  void* xop = nullptr;                 // tensor-core activation operand
  size_t xop_bytes = 0;
  float* gu = nullptr;                 // gate and up outputs of an unfused gated call
  size_t gu_bytes = 0;
  uint8_t* xpre = nullptr;             // chunk-slot image of the pre-conversion pass
  size_t xpre_bytes = 0;
};
constexpr int MAX_COUNTERS = 1 << 16;

// Bits of the device status word (read and cleared by q4_device_status).
constexpr unsigned STATUS_TIMEOUT = 1u;   // a bounded wait ran out
constexpr unsigned STATUS_BAD_ROW = 2u;   // a row index of q4mm_argmax_rows was out of range
constexpr unsigned STATUS_KV_RANGE = 4u;  // a q4_kv_append request was out of range (not written)

// Returns Q4_OK and fills *ws with at least the requested capacities.
int workspace_get(int device, size_t partial_bytes, size_t xop_bytes, Workspace* ws, size_t gu_bytes = 0,
                  size_t xpre_bytes = 0);

// ---- launchers (return a Q4 status; launch errors map to Q4_ERR_CUDA) ----
// Quantize fp32 W (device) into canonical blocks in canon_dev, then repack.
int launch_quantize(const float* w, int64_t N, int64_t K, uint8_t* canon_dev, Weight* W,
                    unsigned int* flag, cudaStream_t s);
int launch_import(const uint8_t* canon_dev, Weight* W, unsigned int* flag, cudaStream_t s);
int launch_export(const Weight* W, uint8_t* canon_dev, cudaStream_t s);
int quantize_flag_status(unsigned flag);

// K partition of the streaming kernels (from N and K only, never from M).
struct MmaPlan {
  int splits;
  int64_t kbp_per_split;  // block pairs per split
  int num_sms = 0;        // SMs the plan was made for (0: unknown)
};

// mma.sync streaming kernel (small and medium M).  One launch may cover up to
// MMA_GROUP_MAX weights that share K and the activations; the K partition is
// planned from their total tile count.
constexpr int MMA_GROUP_MAX = Q4MM_GROUP_MAX;
struct MmaLaunch {
  int count = 0;
  const Weight* W[MMA_GROUP_MAX] = {};
  float* y[MMA_GROUP_MAX] = {};
  bool gated = false;  // W[0], W[1] = gate, up: y[0] = SiLU(x W0^T) * (x W1^T)
};
MmaPlan mma_plan(const Weight* W, int num_sms);
// Bytes of the pre-conversion image for any launch of this plan (whole K or
// its K splits); 0 when the pass is built out.
size_t mma_xpre_bytes(int64_t KBP, const MmaPlan& p);
// True when a launch of `launch_rows` token rows with this plan uses row-group
// CTAs (one 32-row group pair of a tile over the whole K, no K split) instead
// of the split plan: four CTAs per tile fit on the SMs, K is short and the
// launch has at most 8 rows, for y output in default mode.
bool mma_row_groups(const MmaPlan& plan, int64_t K, bool batch_invariant, bool greedy_pick,
                    int64_t launch_rows);
// Launches of more tiles than SMs with one K split run as two-tile CTAs in
// default mode, and then take at most 8 token rows each (16 otherwise).
bool mma_two_tiles(const MmaPlan& plan, int64_t tiles, bool batch_invariant);
int mma_rows_per_launch(bool batch_invariant, bool two_tiles);
MmaPlan mma_plan_tiles(int64_t tiles, int64_t KBP, int num_sms);
size_t mma_partial_bytes(const Weight* W, const MmaPlan& p, int64_t M, bool batch_invariant);
size_t mma_partial_bytes_tiles(int64_t tiles, const MmaPlan& p, int64_t M, bool batch_invariant);
int mma_launch_count(int64_t M, bool batch_invariant, bool two_tiles);
// Kernel launches of a streaming call over `tiles` tiles (main launches and
// their pre-conversion passes), as launch_mma_group makes them.
int mma_call_launches(int64_t tiles, int64_t KBP, int64_t K, const MmaPlan& plan, int64_t M, bool batch_invariant,
                      bool greedy_pick);
int launch_mma(const Weight* W, const float* x, int64_t M, float* y, int32_t* idx, float* maxval,
               const MmaPlan& plan, bool batch_invariant, const Workspace& ws, cudaStream_t s);
int launch_mma_group(const MmaLaunch& L, const float* x, int64_t M, int32_t* idx, float* maxval,
                     const MmaPlan& plan, bool batch_invariant, const Workspace& ws, cudaStream_t s,
                     const int32_t* xrows = nullptr, int64_t x_rows = 0);

// h = SiLU(x Wg^T) * (x Wu^T) on the streaming kernel: two-tile CTAs that
// pair tile b of Wg with tile b of Wu over the whole K, up to 8 token rows per
// launch (Wg and Wu of one shape).
int launch_mma_gated(const Weight* Wg, const Weight* Wu, const float* x, int64_t M, float* h,
                     const Workspace& ws, cudaStream_t s);
// h[i] = SiLU(g[i]) * u[i] for i < n (the gated step after a grouped call).
int launch_silu_mul(const float* g, const float* u, float* h, int64_t n, cudaStream_t s);

// KV-cache append of one step (see q4_kv_append); sizes in elements except
// row_bytes and the source strides (bytes: K layer, token, head, then V's).
int launch_kv_append(uint8_t* k_cache, uint8_t* v_cache, const uint8_t* k_new, const uint8_t* v_new,
                     int64_t layers, int64_t slots, int64_t heads, int64_t row_bytes, int64_t capacity,
                     const int64_t (&stride)[6], const int32_t* offsets,
                     const int32_t* slot, const int32_t* pos, int S, int64_t total, unsigned* status,
                     int num_sms, cudaStream_t s);

// Greedy verification of draft tokens per request (see q4_verify_greedy).
int launch_verify(const int32_t* idx, const int32_t* draft, int64_t total, const int32_t* offsets,
                  int S, int32_t* accepted, cudaStream_t s);

// CUDA-core streaming kernel.
MmaPlan simt_plan(const Weight* W, int num_sms);
size_t simt_partial_bytes(const Weight* W, const MmaPlan& p, int64_t M);
int simt_launch_count(int64_t M);
int launch_simt(const Weight* W, const float* x, int64_t M, float* y, int32_t* idx,
                float* maxval, const MmaPlan& plan, const Workspace& ws, cudaStream_t s);

// tcgen05 kernel (large M).
struct TcPlan {
  int splits;
  int64_t kbp_per_split;  // block pairs per split
  int m_tile;             // MMA N (3 x token rows per CTA)
  int num_sms;            // SMs of the device (one CTA per SM)
};
TcPlan tc_plan(const Weight* W, int64_t M, int num_sms, bool batch_invariant);
TcPlan tc_plan_tiles(int64_t tiles, int64_t KBP, int64_t M, int num_sms, bool batch_invariant);
size_t tc_partial_bytes_tiles(int64_t tiles, const TcPlan& p, int64_t M);
size_t tc_xop_bytes_kbp(int64_t KBP, const TcPlan& p, int64_t M);
// One tcgen05 launch (pair) over the tiles of up to MMA_GROUP_MAX weights that
// share K and the activations.
int launch_tc_group(const MmaLaunch& L, const float* x, int64_t M, int32_t* idx, float* maxval,
                    const TcPlan& plan, const Workspace& ws, cudaStream_t s);
size_t tc_partial_bytes(const Weight* W, const TcPlan& p, int64_t M);
size_t tc_xop_bytes(const Weight* W, const TcPlan& p, int64_t M);
int tc_launch_count(const TcPlan& p, int64_t M);
int64_t tc_rows_per_launch();  // token rows per launch pair
int launch_tc(const Weight* W, const float* x, int64_t M, float* y, int32_t* idx,
              float* maxval, const TcPlan& plan, const Workspace& ws, cudaStream_t s);

int device_num_sms(int device);
// Test settings (q4mm_set_wait_limit_ns, q4mm_set_stall_for_test): the bound
// of every wait a kernel makes on another role or CTA, in ns (default 1 s),
// the split-K poll rounds that match it, and whether launches withhold their
// first hand-off so that the waiting side times out.
unsigned long long wait_limit_ns();
unsigned poll_rounds();
int stall_for_test();
// Read and clear the status word of q4mm_forward_noalloc's fixed scratch on
// `device` (0 if that call never ran there).
int noalloc_status_take(int device, unsigned* bits);
bool tc_kernel_built();

}  // namespace q4
