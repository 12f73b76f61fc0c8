// q4mm_api.cu — the C ABI: argument checks, handle and scratch management,
// and the choice of kernel path.
//
// The path choice follows the lesson of "Why Continuous Batching Slowed Down
// My LLM Inference Engine" (§"Row-by-Row GEMV to the Rescue", §"Takeaways"):
// the switch between the streaming small-M kernel and the tensor-core kernel
// is a measured M threshold, not "one row vs. more than one"; and in
// batch-invariant mode the path and the K partition never depend on M
// (§"The Other Request Already Finished — So Why Is It Still Having an
// Effect?").
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "q4mm_internal.h"

struct q4_weight {
  q4::Weight w;
};

namespace q4 {
namespace {

constexpr int MAX_DEVICES = 64;

struct DeviceScratch {
  std::mutex mu;
  bool init = false;
  Workspace ws;
  unsigned int* format_flag = nullptr;
  int num_sms = 0;
  int cc_major = 0, cc_minor = 0;
};
DeviceScratch g_dev[MAX_DEVICES];

// Below this M the streaming mma.sync kernel is used, at or above it the
// tcgen05 kernel.  Measured on GB300 over one Qwen2.5-7B decoder layer (q/k/v
// group, o, gate/up group, down; 8 layer copies in a CUDA graph), with the
// streaming kernel taking up to 16 rows per launch: streaming is faster up to
// M = 16 (o 13.7 against 16.9 us, down 33.2 against 40.3 us), the tensor-core
// kernel from M = 17, where streaming needs a second launch (o 17.2 against
// 17.9 us, down 40.5 against 44.5 us; the layer 142.4 against 148.7 us).
constexpr int64_t DEFAULT_M_THRESHOLD = 17;
std::atomic<int64_t> g_m_threshold{DEFAULT_M_THRESHOLD};
// Grouped calls (q4mm_forward_group) run one launch over the whole group on
// either path (the gate/up group's streaming launches take 8 rows each, as
// two-tile CTAs).  Measured on GB300 over a layer's q/k/v and gate/up groups
// (8 layer copies in a graph, us for the two groups, streaming / tensor
// cores): 75.2 / 85.3 at M = 20, 83.7 / 85.3 at M = 24, 99.8 / 85.7 at
// M = 25 and 109.2 / 86.0 at M = 32.
constexpr int64_t DEFAULT_GROUP_M_THRESHOLD = 25;
std::atomic<int64_t> g_group_m_threshold{DEFAULT_GROUP_M_THRESHOLD};

// Test settings (q4mm_set_wait_limit_ns, q4mm_set_stall_for_test).
constexpr unsigned long long DEFAULT_WAIT_NS = 1000000000ull;  // 1 s
std::atomic<unsigned long long> g_wait_ns{DEFAULT_WAIT_NS};
std::atomic<int> g_stall{0};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int init_device_locked(int dev, DeviceScratch& ds) {
  if (ds.init) return Q4_OK;
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return Q4_ERR_CUDA;
  ds.num_sms = prop.multiProcessorCount;
  ds.cc_major = prop.major;
  ds.cc_minor = prop.minor;
  const size_t small = 256 + MAX_COUNTERS * sizeof(unsigned) + Q4MM_M_MAX * sizeof(unsigned long long) + 256;
  char* base = nullptr;
  if (cudaMalloc(&base, small) != cudaSuccess) return Q4_ERR_NOMEM;
  if (cudaMemset(base, 0, small) != cudaSuccess) return Q4_ERR_CUDA;
  ds.ws.status = reinterpret_cast<unsigned*>(base);
  ds.ws.argmax_done = reinterpret_cast<unsigned*>(base + 4);
  ds.format_flag = reinterpret_cast<unsigned*>(base + 8);
  ds.ws.keys = reinterpret_cast<unsigned long long*>(base + 256);
  ds.ws.counters = reinterpret_cast<unsigned*>(base + 256 + Q4MM_M_MAX * sizeof(unsigned long long));
  if (cudaDeviceSynchronize() != cudaSuccess) return Q4_ERR_CUDA;
  ds.init = true;
  return Q4_OK;
}

int current_device(int* dev) {
  if (cudaGetDevice(dev) != cudaSuccess) return Q4_ERR_CUDA;
  if (*dev < 0 || *dev >= MAX_DEVICES) return Q4_ERR_UNSUPPORTED;
  return Q4_OK;
}

bool tc_supported(const DeviceScratch& ds) {
  return tc_kernel_built() && ds.cc_major == 10 && ds.cc_minor == 3;
}

int alloc_weight(int64_t N, int64_t K, int dev, Weight* W) {
  W->N = N;
  W->K = K;
  W->N_pad = pad_n(N);
  W->KB = K / BLOCK_K;
  W->KBP = (W->KB + 1) / 2;
  W->tiles = W->N_pad / TILE_N;
  W->device = dev;
  const size_t nib_bytes = (size_t)W->tiles * W->KBP * PAIR_NIB_BYTES;
  const size_t d_bytes = (size_t)W->tiles * W->KBP * PAIR_SCL_BYTES;
  const size_t off = (nib_bytes + 255) / 256 * 256;
  W->alloc_bytes = off + d_bytes;
  if (cudaMalloc(&W->alloc, W->alloc_bytes) != cudaSuccess) {
    cudaGetLastError();
    return Q4_ERR_NOMEM;
  }
  W->nib = static_cast<uint8_t*>(W->alloc);
  W->d = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(W->alloc) + off);
  return Q4_OK;
}

int check_shape(int64_t N, int64_t K) {
  if (N < 1 || K < BLOCK_K || (K % BLOCK_K) != 0) return Q4_ERR_SHAPE;
  // grid limits: K/32 blocks and N/128 tiles are grid dimensions of 65535 max
  if (pad_n(N) / TILE_N > 65535 || K / BLOCK_K > 65535) return Q4_ERR_SHAPE;
  return Q4_OK;
}

// Path choice.  Deterministic in (flags, M, device); in batch-invariant mode
// it ignores M entirely (always the streaming MMA kernel with one token row
// per column group).
int choose_path(const DeviceScratch& ds, int64_t M, uint32_t flags) {
  const bool tc = tc_supported(ds);
  if (flags & Q4MM_ROW_BY_ROW) return Q4MM_PATH_ROW_BY_ROW;
  if (flags & Q4MM_FORCE_SIMT) return Q4MM_PATH_SIMT;
  if (flags & Q4MM_FORCE_MMA) return Q4MM_PATH_MMA;
  if (flags & Q4MM_FORCE_TC) return tc ? Q4MM_PATH_TC : -Q4_ERR_UNSUPPORTED;
  if (flags & Q4MM_BATCH_INVARIANT) return Q4MM_PATH_MMA;
  return (tc && M >= g_m_threshold.load()) ? Q4MM_PATH_TC : Q4MM_PATH_MMA;
}

constexpr uint32_t KNOWN_FLAGS = Q4MM_BATCH_INVARIANT | Q4MM_FORCE_SIMT | Q4MM_FORCE_TC |
                                 Q4MM_ROW_BY_ROW | Q4MM_FORCE_MMA;

int run(const q4_weight* Wh, const float* x, float* y, int32_t* idx, float* maxval, int64_t M,
        uint32_t flags, cudaStream_t s) {
  if (!Wh || !x || (!y && !idx)) return Q4_ERR_INVALID_ARG;
  if (flags & ~KNOWN_FLAGS) return Q4_ERR_INVALID_ARG;
  const int forced = !!(flags & Q4MM_FORCE_SIMT) + !!(flags & Q4MM_FORCE_TC) +
                     !!(flags & Q4MM_ROW_BY_ROW) + !!(flags & Q4MM_FORCE_MMA);
  if (forced > 1) return Q4_ERR_INVALID_ARG;
  if (M < 0) return Q4_ERR_INVALID_ARG;
  if (M > Q4MM_M_MAX) return Q4_ERR_SHAPE;
  if (M == 0) return Q4_OK;
  if (!aligned16(x) || (y && !aligned16(y)) || (idx && !aligned16(idx)) ||
      (maxval && !aligned16(maxval)))
    return Q4_ERR_ALIGN;
  const Weight* W = &Wh->w;
  int dev;
  int st = current_device(&dev);
  if (st) return st;
  if (dev != W->device) return Q4_ERR_INVALID_ARG;
  DeviceScratch& ds = g_dev[dev];
  std::lock_guard<std::mutex> lock(ds.mu);
  st = init_device_locked(dev, ds);
  if (st) return st;
  const int path = choose_path(ds, M, flags);
  if (path < 0) return -path;
  const bool inv = (flags & Q4MM_BATCH_INVARIANT) != 0;
  if (path == Q4MM_PATH_TC) {
    const TcPlan plan = tc_plan(W, M, ds.num_sms, inv);
    Workspace ws;
    st = workspace_get(dev, tc_partial_bytes(W, plan, M), tc_xop_bytes(W, plan, M), &ws);
    if (st) return st;
    return launch_tc(W, x, M, y, idx, maxval, plan, ws, s);
  }
  if (path == Q4MM_PATH_MMA) {
    const MmaPlan plan = mma_plan(W, ds.num_sms);
    Workspace ws;
    st = workspace_get(dev, mma_partial_bytes(W, plan, M, inv), 0, &ws, 0, mma_xpre_bytes(W->KBP, plan));
    if (st) return st;
    return launch_mma(W, x, M, y, idx, maxval, plan, inv, ws, s);
  }
  const MmaPlan plan = simt_plan(W, ds.num_sms);
  Workspace ws;
  if (path == Q4MM_PATH_ROW_BY_ROW) {
    st = workspace_get(dev, simt_partial_bytes(W, plan, 1), 0, &ws);
    if (st) return st;
    for (int64_t m = 0; m < M; ++m) {
      st = launch_simt(W, x + m * W->K, 1, y ? y + m * W->N : nullptr, idx ? idx + m : nullptr,
                       (idx && maxval) ? maxval + m : nullptr, plan, ws, s);
      if (st) return st;
    }
    return Q4_OK;
  }
  st = workspace_get(dev, simt_partial_bytes(W, plan, M), 0, &ws);
  if (st) return st;
  return launch_simt(W, x, M, y, idx, maxval, plan, ws, s);
}

}  // namespace

// Caller holds g_dev[device].mu.
int workspace_get(int device, size_t partial_bytes, size_t xop_bytes, Workspace* out, size_t gu_bytes,
                  size_t xpre_bytes) {
  DeviceScratch& ds = g_dev[device];
  if (xpre_bytes > ds.ws.xpre_bytes) {
    size_t want = xpre_bytes + xpre_bytes / 2;
    if (ds.ws.xpre) cudaFree(ds.ws.xpre);
    ds.ws.xpre = nullptr;
    ds.ws.xpre_bytes = 0;
    if (cudaMalloc(&ds.ws.xpre, want) != cudaSuccess) {
      cudaGetLastError();
      return Q4_ERR_NOMEM;
    }
    ds.ws.xpre_bytes = want;
  }
  if (gu_bytes > ds.ws.gu_bytes) {
    size_t want = gu_bytes + gu_bytes / 2;
    if (ds.ws.gu) cudaFree(ds.ws.gu);
    ds.ws.gu = nullptr;
    ds.ws.gu_bytes = 0;
    if (cudaMalloc(&ds.ws.gu, want) != cudaSuccess) {
      cudaGetLastError();
      return Q4_ERR_NOMEM;
    }
    ds.ws.gu_bytes = want;
  }
  if (partial_bytes > ds.ws.partial_bytes) {
    size_t want = partial_bytes + partial_bytes / 2;
    if (ds.ws.partial) cudaFree(ds.ws.partial);  // cudaFree waits for work in flight
    ds.ws.partial = nullptr;
    ds.ws.partial_bytes = 0;
    if (cudaMalloc(&ds.ws.partial, want) != cudaSuccess) {
      cudaGetLastError();
      return Q4_ERR_NOMEM;
    }
    // idle partial-sum words are zero (q4mm_epilogue.cuh)
    if (cudaMemset(ds.ws.partial, 0, want) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess)
      return Q4_ERR_CUDA;
    ds.ws.partial_bytes = want;
  }
  if (xop_bytes > ds.ws.xop_bytes) {
    size_t want = xop_bytes + xop_bytes / 2;
    if (ds.ws.xop) cudaFree(ds.ws.xop);
    ds.ws.xop = nullptr;
    ds.ws.xop_bytes = 0;
    if (cudaMalloc(&ds.ws.xop, want) != cudaSuccess) {
      cudaGetLastError();
      return Q4_ERR_NOMEM;
    }
    ds.ws.xop_bytes = want;
  }
  *out = ds.ws;
  return Q4_OK;
}

// The largest scratch any single-weight call on W can ask for, reserved when W
// is created (a synchronous step) so that q4mm_forward / q4mm_argmax on a
// created weight never allocate or synchronize.  Every path's scratch stops
// growing at its rows per launch (16 streaming, 256 tensor-core, the SIMT
// launch size), so the maxima are taken at M = Q4MM_M_MAX, and over all
// tensor-core launch sizes since its K partition depends on the token tiles.
// Caller holds g_dev[device].mu.
int workspace_reserve_for(int device, const Weight* W) {
  const DeviceScratch& ds = g_dev[device];
  size_t partial = mma_partial_bytes(W, mma_plan(W, ds.num_sms), Q4MM_M_MAX, false);
  partial = std::max(partial, simt_partial_bytes(W, simt_plan(W, ds.num_sms), Q4MM_M_MAX));
  size_t xop = 0;
  if (tc_supported(ds)) {
    for (int inv = 0; inv < 2; ++inv)
      for (int64_t m = 1; m <= tc_rows_per_launch(); ++m) {
        const TcPlan plan = tc_plan(W, m, ds.num_sms, inv != 0);
        partial = std::max(partial, tc_partial_bytes(W, plan, m));
        xop = std::max(xop, tc_xop_bytes(W, plan, m));
      }
  }
  Workspace ws;
  return workspace_get(device, partial, xop, &ws, 0, mma_xpre_bytes(W->KBP, mma_plan(W, ds.num_sms)));
}

int device_num_sms(int device) { return g_dev[device].num_sms; }

unsigned long long wait_limit_ns() { return g_wait_ns.load(); }
// one round of re-reads of a batch of partial sums takes about 1 us
unsigned poll_rounds() {
  const unsigned long long r = g_wait_ns.load() / 1024ull;
  return (unsigned)(r < 16ull ? 16ull : (r > (1ull << 24) ? (1ull << 24) : r));
}
int stall_for_test() { return g_stall.load(); }

}  // namespace q4

using namespace q4;

extern "C" {

int q4_quantize(const float* w, int64_t N, int64_t K, q4_weight** out, cudaStream_t stream) {
  if (!w || !out) return Q4_ERR_INVALID_ARG;
  int st = check_shape(N, K);
  if (st) return st;
  if (!aligned16(w)) return Q4_ERR_ALIGN;
  int dev;
  st = current_device(&dev);
  if (st) return st;
  DeviceScratch& ds = g_dev[dev];
  std::lock_guard<std::mutex> lock(ds.mu);
  st = init_device_locked(dev, ds);
  if (st) return st;
  q4_weight* h = new (std::nothrow) q4_weight;
  if (!h) return Q4_ERR_NOMEM;
  st = alloc_weight(N, K, dev, &h->w);
  if (st) {
    delete h;
    return st;
  }
  uint8_t* canon = nullptr;  // canonical blocks, repacked into the device layout
  if (cudaMalloc(&canon, (size_t)N * (size_t)(K / BLOCK_K) * CANON_BLOCK_BYTES) != cudaSuccess) {
    cudaGetLastError();
    cudaFree(h->w.alloc);
    delete h;
    return Q4_ERR_NOMEM;
  }
  unsigned flag = 0;
  st = Q4_OK;
  if (cudaMemsetAsync(ds.format_flag, 0, sizeof(unsigned), stream) != cudaSuccess) st = Q4_ERR_CUDA;
  if (!st) st = launch_quantize(w, N, K, canon, &h->w, ds.format_flag, stream);
  if (!st && cudaMemcpyAsync(&flag, ds.format_flag, sizeof(unsigned), cudaMemcpyDeviceToHost,
                             stream) != cudaSuccess)
    st = Q4_ERR_CUDA;
  if (!st && cudaStreamSynchronize(stream) != cudaSuccess) st = Q4_ERR_CUDA;
  cudaFree(canon);
  if (!st) st = quantize_flag_status(flag);
  if (!st) st = workspace_reserve_for(dev, &h->w);
  if (st) {
    cudaFree(h->w.alloc);
    delete h;
    return st;
  }
  *out = h;
  return Q4_OK;
}

int q4_import_blocks(const void* host_blocks, int64_t N, int64_t K, q4_weight** out,
                     cudaStream_t stream) {
  if (!host_blocks || !out) return Q4_ERR_INVALID_ARG;
  int st = check_shape(N, K);
  if (st) return st;
  int dev;
  st = current_device(&dev);
  if (st) return st;
  DeviceScratch& ds = g_dev[dev];
  std::lock_guard<std::mutex> lock(ds.mu);
  st = init_device_locked(dev, ds);
  if (st) return st;
  q4_weight* h = new (std::nothrow) q4_weight;
  if (!h) return Q4_ERR_NOMEM;
  st = alloc_weight(N, K, dev, &h->w);
  if (st) {
    delete h;
    return st;
  }
  const size_t bytes = (size_t)N * (size_t)(K / BLOCK_K) * CANON_BLOCK_BYTES;
  uint8_t* staging = nullptr;
  if (cudaMalloc(&staging, bytes) != cudaSuccess) {
    cudaGetLastError();
    cudaFree(h->w.alloc);
    delete h;
    return Q4_ERR_NOMEM;
  }
  unsigned flag = 0;
  if (cudaMemsetAsync(ds.format_flag, 0, sizeof(unsigned), stream) != cudaSuccess ||
      cudaMemcpyAsync(staging, host_blocks, bytes, cudaMemcpyHostToDevice, stream) != cudaSuccess)
    st = Q4_ERR_CUDA;
  if (!st) st = launch_import(staging, &h->w, ds.format_flag, stream);
  if (!st && cudaMemcpyAsync(&flag, ds.format_flag, sizeof(unsigned), cudaMemcpyDeviceToHost,
                             stream) != cudaSuccess)
    st = Q4_ERR_CUDA;
  if (!st && cudaStreamSynchronize(stream) != cudaSuccess) st = Q4_ERR_CUDA;
  cudaFree(staging);
  if (!st) st = quantize_flag_status(flag);
  if (!st) st = workspace_reserve_for(dev, &h->w);
  if (st) {
    cudaFree(h->w.alloc);
    delete h;
    return st;
  }
  *out = h;
  return Q4_OK;
}

int q4_export_blocks(const q4_weight* W, void* host_blocks, size_t bytes) {
  if (!W || !host_blocks) return Q4_ERR_INVALID_ARG;
  const size_t need = (size_t)W->w.N * (size_t)W->w.KB * CANON_BLOCK_BYTES;
  if (bytes < need) return Q4_ERR_INVALID_ARG;
  int dev;
  int st = current_device(&dev);
  if (st) return st;
  if (dev != W->w.device) return Q4_ERR_INVALID_ARG;
  uint8_t* staging = nullptr;
  if (cudaMalloc(&staging, need) != cudaSuccess) {
    cudaGetLastError();
    return Q4_ERR_NOMEM;
  }
  st = launch_export(&W->w, staging, 0);
  if (!st && cudaMemcpy(host_blocks, staging, need, cudaMemcpyDeviceToHost) != cudaSuccess)
    st = Q4_ERR_CUDA;
  cudaFree(staging);
  return st;
}

int q4_weight_free(q4_weight* W) {
  if (!W) return Q4_ERR_INVALID_ARG;
  const cudaError_t e = cudaFree(W->w.alloc);
  delete W;
  return e == cudaSuccess ? Q4_OK : Q4_ERR_CUDA;
}

int q4_weight_shape(const q4_weight* W, int64_t* N, int64_t* K) {
  if (!W || !N || !K) return Q4_ERR_INVALID_ARG;
  *N = W->w.N;
  *K = W->w.K;
  return Q4_OK;
}

int q4_weight_device_bytes(const q4_weight* W, size_t* bytes) {
  if (!W || !bytes) return Q4_ERR_INVALID_ARG;
  *bytes = W->w.alloc_bytes;
  return Q4_OK;
}

int q4mm_forward(const q4_weight* W, const float* x, float* y, int64_t M, cudaStream_t stream) {
  if (!y) return Q4_ERR_INVALID_ARG;
  return run(W, x, y, nullptr, nullptr, M, 0u, stream);
}

int q4mm_forward_ex(const q4_weight* W, const float* x, float* y, int64_t M, uint32_t flags,
                    cudaStream_t stream) {
  if (!y) return Q4_ERR_INVALID_ARG;
  return run(W, x, y, nullptr, nullptr, M, flags, stream);
}

int q4mm_forward_group(const q4_weight* const* W, int count, const float* x, float* const* y,
                       int64_t M, uint32_t flags, cudaStream_t stream) {
  if (!W || !x || !y || count < 1 || count > Q4MM_GROUP_MAX) return Q4_ERR_INVALID_ARG;
  if (flags & ~(Q4MM_BATCH_INVARIANT | Q4MM_FORCE_MMA | Q4MM_FORCE_TC)) return Q4_ERR_INVALID_ARG;
  if ((flags & Q4MM_FORCE_MMA) && (flags & Q4MM_FORCE_TC)) return Q4_ERR_INVALID_ARG;
  for (int i = 0; i < count; ++i) {
    if (!W[i] || !y[i]) return Q4_ERR_INVALID_ARG;
    if (W[i]->w.K != W[0]->w.K || W[i]->w.device != W[0]->w.device) return Q4_ERR_INVALID_ARG;
  }
  if (M < 0) return Q4_ERR_INVALID_ARG;
  if (M > Q4MM_M_MAX) return Q4_ERR_SHAPE;
  if (M == 0) return Q4_OK;
  if (!aligned16(x)) return Q4_ERR_ALIGN;
  for (int i = 0; i < count; ++i)
    if (!aligned16(y[i])) return Q4_ERR_ALIGN;
  int dev;
  int st = current_device(&dev);
  if (st) return st;
  if (dev != W[0]->w.device) return Q4_ERR_INVALID_ARG;
  {
    DeviceScratch& ds = g_dev[dev];
    std::lock_guard<std::mutex> lock(ds.mu);
    st = init_device_locked(dev, ds);
    if (st) return st;
    const bool inv = (flags & Q4MM_BATCH_INVARIANT) != 0;
    const bool force_tc = (flags & Q4MM_FORCE_TC) != 0;
    if (force_tc && !tc_supported(ds)) return Q4_ERR_UNSUPPORTED;
    const bool streaming = !force_tc && ((flags & (Q4MM_FORCE_MMA | Q4MM_BATCH_INVARIANT)) != 0 ||
                                         !tc_supported(ds) || M < g_group_m_threshold.load());
    MmaLaunch L;
    L.count = count;
    int64_t tiles = 0;
    for (int i = 0; i < count; ++i) {
      L.W[i] = &W[i]->w;
      L.y[i] = y[i];
      tiles += W[i]->w.tiles;
    }
    Workspace ws;
    if (streaming) {
      const MmaPlan plan = mma_plan_tiles(tiles, W[0]->w.KBP, ds.num_sms);
      st = workspace_get(dev, mma_partial_bytes_tiles(tiles, plan, M, inv), 0, &ws, 0, mma_xpre_bytes(W[0]->w.KBP, plan));
      if (st) return st;
      return launch_mma_group(L, x, M, nullptr, nullptr, plan, inv, ws, stream);
    }
    // tensor-core path: one launch pair over the tiles of the whole group (in
    // batch-invariant mode with the plan of one token tile, as single calls)
    const TcPlan plan = tc_plan_tiles(tiles, W[0]->w.KBP, M, ds.num_sms, inv);
    st = workspace_get(dev, tc_partial_bytes_tiles(tiles, plan, M), tc_xop_bytes_kbp(W[0]->w.KBP, plan, M), &ws);
    if (st) return st;
    return launch_tc_group(L, x, M, nullptr, nullptr, plan, ws, stream);
  }
}

int q4mm_forward_gated(const q4_weight* Wg, const q4_weight* Wu, const float* x, float* h, int64_t M,
                       uint32_t flags, cudaStream_t stream) {
  if (!Wg || !Wu || !x || !h) return Q4_ERR_INVALID_ARG;
  if (flags & ~(Q4MM_BATCH_INVARIANT | Q4MM_FORCE_MMA | Q4MM_FORCE_TC)) return Q4_ERR_INVALID_ARG;
  if ((flags & Q4MM_FORCE_MMA) && (flags & Q4MM_FORCE_TC)) return Q4_ERR_INVALID_ARG;
  if (Wg->w.N != Wu->w.N || Wg->w.K != Wu->w.K || Wg->w.device != Wu->w.device) return Q4_ERR_INVALID_ARG;
  if (M < 0) return Q4_ERR_INVALID_ARG;
  if (M > Q4MM_M_MAX) return Q4_ERR_SHAPE;
  if (M == 0) return Q4_OK;
  if (!aligned16(x) || !aligned16(h)) return Q4_ERR_ALIGN;
  int dev;
  int st = current_device(&dev);
  if (st) return st;
  if (dev != Wg->w.device) return Q4_ERR_INVALID_ARG;
  DeviceScratch& ds = g_dev[dev];
  std::lock_guard<std::mutex> lock(ds.mu);
  st = init_device_locked(dev, ds);
  if (st) return st;
  const bool inv = (flags & Q4MM_BATCH_INVARIANT) != 0;
  const bool force_tc = (flags & Q4MM_FORCE_TC) != 0;
  if (force_tc && !tc_supported(ds)) return Q4_ERR_UNSUPPORTED;
  const bool streaming = !force_tc && ((flags & (Q4MM_FORCE_MMA | Q4MM_BATCH_INVARIANT)) != 0 ||
                                       !tc_supported(ds) || M < g_group_m_threshold.load());
  Workspace ws;
  if (streaming && !inv) {
    // fused: the gate and up tiles of a row range in one CTA, h written directly
    MmaPlan whole;  // one K split: the gated launches cover the whole K
    whole.splits = 1;
    whole.kbp_per_split = Wg->w.KBP;
    st = workspace_get(dev, 0, 0, &ws, 0, mma_xpre_bytes(Wg->w.KBP, whole));
    if (st) return st;
    return launch_mma_gated(&Wg->w, &Wu->w, x, M, h, ws, stream);
  }
  // grouped call into scratch, then the elementwise step
  const size_t out_bytes = (size_t)M * (size_t)Wg->w.N * sizeof(float);
  MmaLaunch L;
  L.count = 2;
  L.W[0] = &Wg->w;
  L.W[1] = &Wu->w;
  const int64_t tiles = Wg->w.tiles + Wu->w.tiles;
  if (streaming) {
    const MmaPlan plan = mma_plan_tiles(tiles, Wg->w.KBP, ds.num_sms);
    st = workspace_get(dev, mma_partial_bytes_tiles(tiles, plan, M, inv), 0, &ws, 2 * out_bytes,
                       mma_xpre_bytes(Wg->w.KBP, plan));
    if (st) return st;
    L.y[0] = ws.gu;
    L.y[1] = ws.gu + M * Wg->w.N;
    st = launch_mma_group(L, x, M, nullptr, nullptr, plan, inv, ws, stream);
  } else {
    const TcPlan plan = tc_plan_tiles(tiles, Wg->w.KBP, M, ds.num_sms, inv);
    st = workspace_get(dev, tc_partial_bytes_tiles(tiles, plan, M), tc_xop_bytes_kbp(Wg->w.KBP, plan, M), &ws,
                       2 * out_bytes);
    if (st) return st;
    L.y[0] = ws.gu;
    L.y[1] = ws.gu + M * Wg->w.N;
    st = launch_tc_group(L, x, M, nullptr, nullptr, plan, ws, stream);
  }
  if (st) return st;
  return launch_silu_mul(ws.gu, ws.gu + M * Wg->w.N, h, M * Wg->w.N, stream);
}

int q4mm_argmax_rows(const q4_weight* Wh, const float* x, int64_t x_rows, const int32_t* rows,
                     int64_t R, int32_t* idx, float* maxval, cudaStream_t stream) {
  if (!Wh || !x || !rows || !idx) return Q4_ERR_INVALID_ARG;
  if (R < 0 || x_rows < 1 || x_rows > INT32_MAX) return Q4_ERR_INVALID_ARG;
  if (R > Q4MM_M_MAX) return Q4_ERR_SHAPE;
  if (R == 0) return Q4_OK;
  if (!aligned16(x) || !aligned16(idx) || (maxval && !aligned16(maxval))) return Q4_ERR_ALIGN;
  const Weight* W = &Wh->w;
  int dev;
  int st = current_device(&dev);
  if (st) return st;
  if (dev != W->device) return Q4_ERR_INVALID_ARG;
  DeviceScratch& ds = g_dev[dev];
  std::lock_guard<std::mutex> lock(ds.mu);
  st = init_device_locked(dev, ds);
  if (st) return st;
  const MmaPlan plan = mma_plan(W, ds.num_sms);
  Workspace ws;
  st = workspace_get(dev, mma_partial_bytes(W, plan, R, false), 0, &ws);
  if (st) return st;
  MmaLaunch L;
  L.count = 1;
  L.W[0] = W;
  L.y[0] = nullptr;
  return launch_mma_group(L, x, R, idx, maxval, plan, false, ws, stream, rows, x_rows);
}

int q4_verify_greedy(const int32_t* idx, const int32_t* draft, int64_t total, const int32_t* offsets,
                     int64_t S, int32_t* accepted, cudaStream_t stream) {
  if (!idx || !draft || !offsets || !accepted || total < 0 || S < 0 || S > INT32_MAX - 128)
    return Q4_ERR_INVALID_ARG;
  if (S == 0) return Q4_OK;
  return launch_verify(idx, draft, total, offsets, (int)S, accepted, stream);
}

int q4_kv_append(void* k_cache, void* v_cache, const void* k_new, const void* v_new, int64_t layers,
                 int64_t slots, int64_t heads, int64_t head_dim, int64_t capacity, int elem_bytes,
                 const int64_t* k_strides, const int64_t* v_strides, const int32_t* offsets,
                 const int32_t* slot, const int32_t* pos, int64_t S, int64_t total, cudaStream_t stream) {
  constexpr int64_t LIM = (int64_t)1 << 31;
  if (layers < 1 || slots < 1 || heads < 1 || head_dim < 1 || capacity < 1 || layers >= LIM ||
      slots >= LIM || heads >= LIM || head_dim >= LIM || capacity >= LIM ||
      (elem_bytes != 2 && elem_bytes != 4) || S < 0 || S >= INT32_MAX || total < 0 || total >= INT32_MAX ||
      !k_strides || !v_strides)
    return Q4_ERR_INVALID_ARG;
  int64_t stride[6];
  for (int i = 0; i < 3; ++i) {
    if (k_strides[i] < 0 || v_strides[i] < 0 || k_strides[i] >= (LIM << 28) || v_strides[i] >= (LIM << 28))
      return Q4_ERR_INVALID_ARG;
    stride[i] = k_strides[i] * elem_bytes;
    stride[3 + i] = v_strides[i] * elem_bytes;
  }
  if (S == 0 || total == 0) return Q4_OK;
  if (!k_cache || !v_cache || !k_new || !v_new || !offsets || !slot || !pos) return Q4_ERR_INVALID_ARG;
  const int64_t row_bytes = head_dim * elem_bytes;
  if (total * ((row_bytes + 15) / 16) >= INT32_MAX || 2 * layers * heads >= INT32_MAX)
    return Q4_ERR_INVALID_ARG;  // the kernel's 32-bit item index within a plane
  bool aligned = row_bytes % 16 == 0 && aligned16(k_cache) && aligned16(v_cache) && aligned16(k_new) &&
                 aligned16(v_new);
  for (int i = 0; i < 6; ++i) aligned = aligned && stride[i] % 16 == 0;
  if (!aligned) return Q4_ERR_ALIGN;
  int dev;
  int st = current_device(&dev);
  if (st) return st;
  DeviceScratch& ds = g_dev[dev];
  std::lock_guard<std::mutex> lock(ds.mu);
  st = init_device_locked(dev, ds);  // the status word the kernel reports to
  if (st) return st;
  return launch_kv_append(static_cast<uint8_t*>(k_cache), static_cast<uint8_t*>(v_cache),
                          static_cast<const uint8_t*>(k_new), static_cast<const uint8_t*>(v_new), layers,
                          slots, heads, row_bytes, capacity, stride, offsets, slot, pos, (int)S, total,
                          ds.ws.status, ds.num_sms, stream);
}

int q4mm_argmax(const q4_weight* W, const float* x, int32_t* idx, float* maxval, int64_t M,
                cudaStream_t stream) {
  if (!idx) return Q4_ERR_INVALID_ARG;
  return run(W, x, nullptr, idx, maxval, M, 0u, stream);
}

int q4mm_argmax_ex(const q4_weight* W, const float* x, int32_t* idx, float* maxval, int64_t M,
                   uint32_t flags, cudaStream_t stream) {
  if (!idx) return Q4_ERR_INVALID_ARG;
  return run(W, x, nullptr, idx, maxval, M, flags, stream);
}

int q4mm_select_path(const q4_weight* W, int64_t M, uint32_t flags) {
  if (!W || M < 0 || (flags & ~KNOWN_FLAGS)) return -Q4_ERR_INVALID_ARG;
  int dev;
  int st = current_device(&dev);
  if (st) return -st;
  DeviceScratch& ds = g_dev[dev];
  std::lock_guard<std::mutex> lock(ds.mu);
  st = init_device_locked(dev, ds);
  if (st) return -st;
  return choose_path(ds, M, flags);
}

int q4mm_plan_info(const q4_weight* W, int64_t M, uint32_t flags, int* path, int* launches,
                   int* splits) {
  if (!W || M < 0 || M > Q4MM_M_MAX || (flags & ~KNOWN_FLAGS)) return Q4_ERR_INVALID_ARG;
  int dev;
  int st = current_device(&dev);
  if (st) return st;
  DeviceScratch& ds = g_dev[dev];
  std::lock_guard<std::mutex> lock(ds.mu);
  st = init_device_locked(dev, ds);
  if (st) return st;
  const int p = choose_path(ds, M, flags);
  if (p < 0) return -p;
  int l = 0, sp = 1;
  if (p == Q4MM_PATH_TC) {
    const TcPlan plan = tc_plan(&W->w, M, ds.num_sms, (flags & Q4MM_BATCH_INVARIANT) != 0);
    l = tc_launch_count(plan, M);
    sp = plan.splits;
  } else if (p == Q4MM_PATH_MMA) {
    const MmaPlan plan = mma_plan(&W->w, ds.num_sms);
    const bool inv = (flags & Q4MM_BATCH_INVARIANT) != 0;
    const bool two = mma_two_tiles(plan, W->w.tiles, inv);
    l = mma_call_launches(W->w.tiles, W->w.KBP, W->w.K, plan, M, inv, false);
    const int64_t rows0 = M < mma_rows_per_launch(inv, two) ? M : mma_rows_per_launch(inv, two);  // first launch
    sp = mma_row_groups(plan, W->w.K, inv, false, rows0) ? 1 : plan.splits;
  } else {
    const MmaPlan plan = simt_plan(&W->w, ds.num_sms);
    l = p == Q4MM_PATH_ROW_BY_ROW ? (int)M : simt_launch_count(M);
    sp = plan.splits;
  }
  if (M == 0) l = 0;
  if (path) *path = p;
  if (launches) *launches = l;
  if (splits) *splits = sp;
  return Q4_OK;
}

int q4mm_set_m_threshold(int64_t m) {
  if (m < 1 || m > Q4MM_M_MAX + 1) return Q4_ERR_INVALID_ARG;
  g_m_threshold.store(m);
  return Q4_OK;
}

int64_t q4mm_get_m_threshold(void) { return g_m_threshold.load(); }

int q4mm_set_group_m_threshold(int64_t m) {
  if (m < 1 || m > Q4MM_M_MAX + 1) return Q4_ERR_INVALID_ARG;
  g_group_m_threshold.store(m);
  return Q4_OK;
}

int64_t q4mm_get_group_m_threshold(void) { return g_group_m_threshold.load(); }

int q4mm_set_wait_limit_ns(uint64_t ns) {
  g_wait_ns.store(ns == 0 ? DEFAULT_WAIT_NS : (unsigned long long)ns);
  return Q4_OK;
}

int q4mm_set_stall_for_test(int on) {
  g_stall.store(on ? 1 : 0);
  return Q4_OK;
}

int q4_scratch_bytes(size_t* partial, size_t* xop, size_t* gu, size_t* xpre) {
  if (!partial || !xop || !gu || !xpre) return Q4_ERR_INVALID_ARG;
  int dev;
  int st = current_device(&dev);
  if (st) return st;
  DeviceScratch& ds = g_dev[dev];
  std::lock_guard<std::mutex> lock(ds.mu);
  *partial = ds.ws.partial_bytes;
  *xop = ds.ws.xop_bytes;
  *gu = ds.ws.gu_bytes;
  *xpre = ds.ws.xpre_bytes;
  return Q4_OK;
}

int q4_device_status(void) {
  int dev;
  int st = current_device(&dev);
  if (st) return st;
  if (cudaDeviceSynchronize() != cudaSuccess) return Q4_ERR_CUDA;
  unsigned v = 0;
  {
    DeviceScratch& ds = g_dev[dev];
    std::lock_guard<std::mutex> lock(ds.mu);
    if (ds.init) {
      if (cudaMemcpy(&v, ds.ws.status, sizeof(unsigned), cudaMemcpyDeviceToHost) != cudaSuccess)
        return Q4_ERR_CUDA;
      if (v) {
        const unsigned zero = 0;
        if (cudaMemcpy(ds.ws.status, &zero, sizeof(unsigned), cudaMemcpyHostToDevice) != cudaSuccess)
          return Q4_ERR_CUDA;
      }
      if (v & STATUS_TIMEOUT) {
        // a kernel gave up part-way: its split-K counters, partial-sum words and
        // greedy-pick keys may be left mid-launch; the device is idle, so reset
        // them to the state every launch expects
        if (cudaMemset(ds.ws.argmax_done, 0, sizeof(unsigned)) != cudaSuccess ||
            cudaMemset(ds.ws.keys, 0, Q4MM_M_MAX * sizeof(unsigned long long)) != cudaSuccess ||
            cudaMemset(ds.ws.counters, 0, MAX_COUNTERS * sizeof(unsigned)) != cudaSuccess ||
            (ds.ws.partial && cudaMemset(ds.ws.partial, 0, ds.ws.partial_bytes) != cudaSuccess) ||
            cudaDeviceSynchronize() != cudaSuccess)
          return Q4_ERR_CUDA;
      }
    }
  }
  // the fixed scratch of q4mm_forward_noalloc keeps its own status word
  unsigned na = 0;
  st = noalloc_status_take(dev, &na);
  if (st) return st;
  v |= na;
  if (v) return (v & STATUS_TIMEOUT) ? Q4_ERR_TIMEOUT : Q4_ERR_INVALID_ARG;
  return Q4_OK;
}

const char* q4_status_string(int status) {
  switch (status) {
    case Q4_OK: return "ok";
    case Q4_ERR_INVALID_ARG: return "invalid argument";
    case Q4_ERR_SHAPE: return "unsupported shape";
    case Q4_ERR_ALIGN: return "pointer not 16-byte aligned";
    case Q4_ERR_NONFINITE: return "non-finite weight or scale";
    case Q4_ERR_RANGE: return "block scale out of binary16 range";
    case Q4_ERR_CUDA: return "CUDA runtime error";
    case Q4_ERR_TIMEOUT: return "device-side wait timed out";
    case Q4_ERR_NOMEM: return "device allocation failed";
    case Q4_ERR_UNSUPPORTED: return "unsupported device or path";
    default: return "unknown status";
  }
}

}  // extern "C"
