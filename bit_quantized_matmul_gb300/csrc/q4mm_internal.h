// q4mm_internal.h — device layout, workspace and launcher declarations shared
// by the library's translation units (not part of the public ABI).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "q4mm.h"

namespace q4 {

// ---------------------------------------------------------------------------
// Device weight layout ("tiled Q4").
//
// Rows are grouped in tiles of TILE_N = 128 (one row per TMEM lane / thread);
// N is padded to a multiple of 128 with zero-scale rows.  For tile t, block b
// (32 weights along K) and row r of the tile:
//   nibbles: 16 bytes at  ((t * KB + b) * 128 + r) * 16
//   scale:   binary16 at   (t * KB + b) * 128 + r
// so one block column of a tile is 2 KB of nibbles plus 256 B of scales, both
// contiguous: a warp's 32 rows read 512 consecutive bytes, and a bulk copy of
// B consecutive blocks of one tile is one contiguous range.
//
// Nibble order inside the 16 bytes (four little-endian 32-bit words w_i, word
// i covering k = 8i .. 8i+7): the nibble at bit 4p (p = 0..3) holds
// k = 8i + 2p and the nibble at bit 16 + 4p holds k = 8i + 2p + 1.  Then
// (w_i >> 4p) & 0x000F000F puts the pair (k = 8i+2p, 8i+2p+1) in the low and
// high 16-bit halves, which is what both kernels unpack.
// ---------------------------------------------------------------------------
constexpr int TILE_N = 128;
constexpr int BLOCK_K = 32;
constexpr int CANON_BLOCK_BYTES = 18;

inline int64_t pad_n(int64_t N) { return (N + TILE_N - 1) / TILE_N * TILE_N; }

struct Weight {
  int64_t N = 0, K = 0, N_pad = 0, KB = 0, tiles = 0;
  int device = 0;
  uint8_t* nib = nullptr;   // [tiles][KB][128][16]
  uint16_t* d = nullptr;    // [tiles][KB][128] binary16 bits
  void* alloc = nullptr;    // single allocation backing nib and d
  size_t alloc_bytes = 0;
};

// Per-device scratch shared by all handles on that device.
struct Workspace {
  unsigned int* status = nullptr;      // device status word (Q4_ERR_TIMEOUT ...)
  unsigned int* counters = nullptr;    // split-K arrival counters, self-resetting
  unsigned long long* keys = nullptr;  // argmax keys [Q4MM_M_MAX], self-resetting
  unsigned int* argmax_done = nullptr; // argmax completion counter
  float* partial = nullptr;            // split-K partial sums
  size_t partial_bytes = 0;
  void* xop = nullptr;                 // tensor-core activation operand
  size_t xop_bytes = 0;
};
constexpr int MAX_COUNTERS = 1 << 16;

// Returns Q4_OK and fills *ws with at least the requested capacities.
int workspace_get(int device, size_t partial_bytes, size_t xop_bytes, Workspace* ws);

// ---- launchers (return a Q4 status; launch errors map to Q4_ERR_CUDA) ----
int launch_quantize(const float* w, int64_t N, int64_t K, Weight* W, unsigned int* flag,
                    cudaStream_t s);
int launch_import(const uint8_t* canon_dev, Weight* W, unsigned int* flag, cudaStream_t s);
int launch_export(const Weight* W, uint8_t* canon_dev, cudaStream_t s);
int quantize_flag_status(unsigned flag);

struct SimtPlan {
  int splits;          // K partition count (depends on N and K only)
  int64_t kb_per_split;
};
SimtPlan simt_plan(const Weight* W, int num_sms);
size_t simt_partial_bytes(const Weight* W, const SimtPlan& p, int64_t M);
int simt_launch_count(int64_t M);

// Mode: y output, or argmax (idx/maxval).
int launch_simt(const Weight* W, const float* x, int64_t M, float* y, int32_t* idx,
                float* maxval, const SimtPlan& plan, const Workspace& ws, cudaStream_t s);

struct TcPlan {
  int splits;
  int64_t kb_per_split;
  int m_tile;          // token rows per CTA pass (MMA N), multiple of 16
};
TcPlan tc_plan(const Weight* W, int64_t M, int num_sms, bool batch_invariant);
size_t tc_partial_bytes(const Weight* W, const TcPlan& p, int64_t M);
size_t tc_xop_bytes(const Weight* W, const TcPlan& p, int64_t M);
int tc_launch_count(const TcPlan& p, int64_t M);
int launch_tc(const Weight* W, const float* x, int64_t M, float* y, int32_t* idx,
              float* maxval, const TcPlan& plan, const Workspace& ws, cudaStream_t s);

int device_num_sms(int device);
bool tc_kernel_built();

}  // namespace q4
