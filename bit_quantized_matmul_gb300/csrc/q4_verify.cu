// q4_verify.cu — greedy verification of draft tokens in a continuous-batching
// step.
//
// A step packs the rows of several requests into one batch ("What continuous
// batching changes: reading three LLM inference traces": prefill, decode and
// verify rows of different requests share one forward pass).  For a request
// verifying speculative draft tokens, the greedy pick of its verify rows
// (§"Same Prompt, Different Story" of "Why Continuous Batching Slowed Down My
// LLM Inference Engine": greedy decoding takes the largest logit) is compared
// with the drafts: the request keeps the longest prefix on which they agree.
#include "q4mm_internal.h"

namespace q4 {
namespace {

// One thread per request: accepted[s] = number of leading positions j of the
// segment [offsets[s], offsets[s+1]) with idx == draft; -1 if the segment is
// malformed (decreasing offsets or outside [0, total)).
__global__ void __launch_bounds__(128) verify_kernel(const int32_t* __restrict__ idx,
                                                     const int32_t* __restrict__ draft,
                                                     int64_t total,
                                                     const int32_t* __restrict__ offsets, int S,
                                                     int32_t* __restrict__ accepted) {
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= S) return;
  const int32_t b = offsets[s], e = offsets[s + 1];
  if (b < 0 || e < b || (int64_t)e > total) {
    accepted[s] = -1;
    return;
  }
  int32_t n = 0;
  while (b + n < e && idx[b + n] == draft[b + n]) ++n;
  accepted[s] = n;
}

}  // namespace

int launch_verify(const int32_t* idx, const int32_t* draft, int64_t total, const int32_t* offsets,
                  int S, int32_t* accepted, cudaStream_t s) {
  verify_kernel<<<(S + 127) / 128, 128, 0, s>>>(idx, draft, total, offsets, S, accepted);
  return cudaGetLastError() == cudaSuccess ? Q4_OK : Q4_ERR_CUDA;
}

}  // namespace q4
