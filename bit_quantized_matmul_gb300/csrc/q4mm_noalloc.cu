// q4mm_noalloc.cu — q4mm_forward_noalloc: the streaming matmul with its
// scratch in a fixed, statically sized device array instead of the
// library's growable per-device workspace.
//
// Why it exists: the other compute calls create (and grow) their scratch with
// cudaMalloc / cudaFree on the first call that needs more.  Some callers must
// not allocate at that point: a serving loop that handed all free device
// memory to its own pool (the allocation would fail), or one that cannot
// afford the device-wide wait that cudaFree implies in the middle of a step.
// This call never allocates; its only device memory besides the caller's
// buffers and the weight handle is the array below, created with the module.
//
// The kernel is the same streaming mma.sync kernel, launch sequence and K
// partition as q4mm_forward_ex(..., Q4MM_FORCE_MMA), so the results are
// bit-identical to that call.
#include <cuda_runtime.h>

#include <mutex>

#include "q4mm_internal.h"

namespace q4 {
namespace {

// Scratch layout (byte offsets):
//   [0, 256)          status word, argmax completion counter
//   [256, +16 KiB)    split-K arrival counters, one per weight tile
//   next 32 KiB       argmax keys (kept valid; this call never uses them)
//   the rest          split-K partial sums
constexpr size_t NA_HEAD = 256;
constexpr int NA_COUNTERS = 4096;
constexpr size_t NA_COUNTER_OFF = NA_HEAD;
constexpr size_t NA_KEYS_OFF = NA_COUNTER_OFF + NA_COUNTERS * sizeof(unsigned);
constexpr size_t NA_PARTIAL_OFF = NA_KEYS_OFF + Q4MM_M_MAX * sizeof(unsigned long long);
constexpr size_t NA_TOTAL = NA_PARTIAL_OFF + Q4MM_NOALLOC_PARTIAL_BYTES;
static_assert(NA_PARTIAL_OFF % 256 == 0, "partial sums must stay 256-byte aligned");

static __device__ __align__(256) unsigned char g_noalloc_scratch[NA_TOTAL];

constexpr int NA_MAX_DEVICES = 64;

struct NoAllocDevice {
  std::mutex mu;
  bool ready = false;
  unsigned char* base = nullptr;  // device address of g_noalloc_scratch on this device
  int num_sms = 0;
};
NoAllocDevice g_na[NA_MAX_DEVICES];

// Once per device, with that device current: find the array's address, read
// the SM count the K partition depends on, and clear the array: counters,
// keys and partial-sum words start at zero (and every launch leaves them so,
// up to the counters' epochs).
int setup_locked(int dev, NoAllocDevice& d) {
  if (d.ready) return Q4_OK;
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) {
    cudaGetLastError();
    return Q4_ERR_CUDA;
  }
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
    return Q4_ERR_CUDA;
  if (cudaMemset(p, 0, NA_TOTAL) != cudaSuccess) return Q4_ERR_CUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return Q4_ERR_CUDA;
  d.base = static_cast<unsigned char*>(p);
  d.num_sms = sms;
  d.ready = true;
  return Q4_OK;
}

}  // namespace

// The status word of the fixed array on `dev`: read and cleared (two 4-byte
// copies, no allocation).  0 when no q4mm_forward_noalloc call has set the
// array up on that device.
int noalloc_status_take(int dev, unsigned* bits) {
  *bits = 0;
  if (dev < 0 || dev >= NA_MAX_DEVICES) return Q4_OK;
  NoAllocDevice& d = g_na[dev];
  std::lock_guard<std::mutex> lock(d.mu);
  if (!d.ready) return Q4_OK;
  unsigned v = 0;
  if (cudaMemcpy(&v, d.base, sizeof(unsigned), cudaMemcpyDeviceToHost) != cudaSuccess) return Q4_ERR_CUDA;
  if (v) {
    const unsigned zero = 0;
    if (cudaMemcpy(d.base, &zero, sizeof(unsigned), cudaMemcpyHostToDevice) != cudaSuccess) return Q4_ERR_CUDA;
  }
  if (v & STATUS_TIMEOUT) {
    // a kernel gave up part-way: counters, keys and partial-sum words back to zero
    if (cudaMemset(d.base + 4, 0, NA_TOTAL - 4) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess)
      return Q4_ERR_CUDA;
  }
  *bits = v;
  return Q4_OK;
}

}  // namespace q4

struct q4_weight {
  q4::Weight w;
};

using namespace q4;

extern "C" int q4mm_forward_noalloc(const q4_weight* Wh, const float* x, float* y, int64_t M,
                                    cudaStream_t stream) {
  if (!Wh || !x || !y) return Q4_ERR_INVALID_ARG;
  if (M < 0) return Q4_ERR_INVALID_ARG;
  if (M > Q4MM_M_MAX) return Q4_ERR_SHAPE;
  if (M == 0) return Q4_OK;
  if ((reinterpret_cast<uintptr_t>(x) & 15u) || (reinterpret_cast<uintptr_t>(y) & 15u))
    return Q4_ERR_ALIGN;
  const Weight* W = &Wh->w;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return Q4_ERR_CUDA;
  if (dev < 0 || dev >= NA_MAX_DEVICES) return Q4_ERR_UNSUPPORTED;
  if (dev != W->device) return Q4_ERR_INVALID_ARG;
  NoAllocDevice& d = g_na[dev];
  std::lock_guard<std::mutex> lock(d.mu);
  int st = setup_locked(dev, d);
  if (st) return st;

  const MmaPlan plan = mma_plan(W, d.num_sms);
  // reject, before any launch, a call whose scratch would not fit
  if (mma_partial_bytes(W, plan, M, false) > (size_t)Q4MM_NOALLOC_PARTIAL_BYTES) return Q4_ERR_SHAPE;
  if (plan.splits > 1 && W->tiles > NA_COUNTERS) return Q4_ERR_SHAPE;

  Workspace ws;
  ws.status = reinterpret_cast<unsigned*>(d.base);
  ws.argmax_done = reinterpret_cast<unsigned*>(d.base + 4);
  ws.counters = reinterpret_cast<unsigned*>(d.base + NA_COUNTER_OFF);
  ws.keys = reinterpret_cast<unsigned long long*>(d.base + NA_KEYS_OFF);
  ws.partial = reinterpret_cast<unsigned long long*>(d.base + NA_PARTIAL_OFF);
  ws.partial_bytes = Q4MM_NOALLOC_PARTIAL_BYTES;
  ws.xop = nullptr;
  ws.xop_bytes = 0;
  return launch_mma(W, x, M, y, nullptr, nullptr, plan, false, ws, stream);
}
