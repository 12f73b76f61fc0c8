// q4_kv.cu — KV-cache append of one continuous-batching step into a
// preallocated, contiguous cache.
//
// "A non-contiguous KV cache cuts Qwen2 decode speed by 59 % at 2k context in
// Candle on Metal" (§"Why it matters", §"Cause and workaround") traces slow
// decode to a cache that grows by concatenation: when the new V rows are a
// strided view, every append re-copies the whole cache.  The fast variants it
// measures write only the new rows into a buffer that is already in place
// (`slice_set` into a preallocated cache, or a contiguous copy first).  Here
// one launch writes the new K and V rows of every layer and every request of
// the step straight into their cache positions, reading the new rows through
// their strides, so a transposed or otherwise strided view needs no staging
// copy and nothing already cached is touched.
//
// Cache layout: [layers][slots][heads][capacity][head_dim], so a request's
// consecutive positions of one (layer, head) are contiguous.  The work is cut
// into 16-byte vectors: one grid row per (K/V, layer, head) plane, and inside
// it (packed row, vector), so the threads of a warp write consecutive bytes of
// one request's rows.
#include "q4mm_internal.h"

namespace q4 {
namespace {

struct KvArgs {
  uint8_t* cache[2];        // K, V caches
  const uint8_t* src[2];    // K, V new rows
  int64_t layers, slots, heads, capacity, total;
  int64_t row_bytes;        // head_dim * element bytes (a multiple of 16)
  int64_t s_layer[2], s_token[2], s_head[2];  // source strides in bytes (K, V)
  const int32_t* offsets;   // [S + 1]
  const int32_t* slot;      // [S]
  const int32_t* pos;       // [S]
  int S;
  unsigned* status;
};

// the request whose packed rows contain row t: the last s with offsets[s] <= t
// (offsets are expected to be non-decreasing; the caller checks the result)
__device__ __forceinline__ int find_request(const int32_t* __restrict__ offsets, int S, int64_t t) {
  int lo = 0, hi = S;  // invariant: answer in [lo, hi)
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if ((int64_t)__ldg(offsets + mid) <= t) lo = mid;
    else hi = mid;
  }
  return lo;
}

// grid.y runs over the (K/V, layer, head) planes; inside a plane the items
// are (packed row t, 16-byte vector v) with 32-bit index arithmetic
__global__ void __launch_bounds__(256) kv_append_kernel(const KvArgs a, uint32_t vpr, int planes) {
  const uint32_t items = (uint32_t)a.total * vpr;
  for (int plane = blockIdx.y; plane < planes; plane += gridDim.y) {
    const int kv = plane / (int)(a.layers * a.heads);
    const int64_t lh = plane - (int64_t)kv * a.layers * a.heads;
    const int64_t l = lh / a.heads, h = lh - l * a.heads;
    const uint8_t* src_plane = a.src[kv] + l * a.s_layer[kv] + h * a.s_head[kv];
    uint8_t* dst_plane = a.cache[kv] + (l * a.slots * a.heads + h) * a.capacity * a.row_bytes;
    const int64_t slot_stride = a.heads * a.capacity * a.row_bytes;  // bytes between slots
    for (uint32_t it = blockIdx.x * blockDim.x + threadIdx.x; it < items; it += gridDim.x * blockDim.x) {
      const uint32_t t = it / vpr, v = it - t * vpr;
      const int s = find_request(a.offsets, a.S, t);
      const int64_t b = __ldg(a.offsets + s), e = __ldg(a.offsets + s + 1);
      if ((int64_t)t < b || (int64_t)t >= e) continue;  // a packed row that belongs to no request
      const int64_t sl = __ldg(a.slot + s), p0 = __ldg(a.pos + s);
      if (sl < 0 || sl >= a.slots || p0 < 0 || e > a.total || p0 + (e - b) > a.capacity) {
        // the whole request is left unwritten; one thread per row reports it
        if (plane == 0 && v == 0) atomicOr(a.status, STATUS_KV_RANGE);
        continue;
      }
      const int64_t p = p0 + ((int64_t)t - b);
      const uint4* src = reinterpret_cast<const uint4*>(src_plane + (int64_t)t * a.s_token[kv]) + v;
      uint4* dst = reinterpret_cast<uint4*>(dst_plane + sl * slot_stride + p * a.row_bytes) + v;
      *dst = __ldg(src);
    }
  }
}

}  // namespace

int launch_kv_append(uint8_t* k_cache, uint8_t* v_cache, const uint8_t* k_new, const uint8_t* v_new,
                     int64_t layers, int64_t slots, int64_t heads, int64_t row_bytes, int64_t capacity,
                     const int64_t (&stride)[6], const int32_t* offsets,
                     const int32_t* slot, const int32_t* pos, int S, int64_t total, unsigned* status,
                     int num_sms, cudaStream_t s) {
  KvArgs a;
  a.cache[0] = k_cache;
  a.cache[1] = v_cache;
  a.src[0] = k_new;
  a.src[1] = v_new;
  a.layers = layers;
  a.slots = slots;
  a.heads = heads;
  a.capacity = capacity;
  a.total = total;
  a.row_bytes = row_bytes;
  for (int kv = 0; kv < 2; ++kv) {
    a.s_layer[kv] = stride[3 * kv];
    a.s_token[kv] = stride[3 * kv + 1];
    a.s_head[kv] = stride[3 * kv + 2];
  }
  a.offsets = offsets;
  a.slot = slot;
  a.pos = pos;
  a.S = S;
  a.status = status;
  const uint32_t vpr = (uint32_t)(row_bytes >> 4);  // 16-byte vectors per row
  const int64_t planes = 2 * layers * heads;
  const int64_t per_plane = (total * vpr + 255) / 256;  // blocks that cover one plane
  const int64_t gy = planes < 65535 ? planes : 65535;
  int64_t gx = ((int64_t)num_sms * 8 + gy - 1) / gy;     // about 8 blocks per SM in all
  if (gx > per_plane) gx = per_plane;
  if (gx < 1) gx = 1;
  kv_append_kernel<<<dim3((unsigned)gx, (unsigned)gy), 256, 0, s>>>(a, vpr, (int)(planes < INT32_MAX ? planes : INT32_MAX));
  return cudaGetLastError() == cudaSuccess ? Q4_OK : Q4_ERR_CUDA;
}

}  // namespace q4
