/*
 * q4mm.h — C ABI of the GB300 (sm_103a) Q4_0 block-quantized matmul library.
 *
 * The operation is the linear layer of LLM decode and continuous batching:
 * M activation rows (token rows: decode, prefill and verify rows merged into
 * one batch) times a weight matrix stored in 4-bit blocks and dequantized on
 * the fly,
 *
 *     y[m, n] = sum_k x[m, k] * w[n, k],   w[n, k] = (q[n, k] - 8) * d[n, k/32]
 *
 * ("Why Continuous Batching Slowed Down My LLM Inference Engine: A Metal
 * Kernel Investigation", §"Two Rows of Input, Two Different Kernels": the
 * quantized matmul whose one-row (GEMV) and many-row (GEMM) kernels the
 * investigation compares; "Why LLM Decoding Is Slow, and Why Batching Is
 * (Almost) Free", §3 "Two Ceilings" and §4 "Share the Weights Across Users":
 * every token row that shares one pass over the weights is nearly free while
 * the step stays memory-bound).
 *
 * Q4_0 block format (the pages say only "4-bit"; this library fixes it):
 * 32 consecutive weights along K share one fp16 scale d = m / -8, where m is
 * the first element of largest magnitude, and q = clamp(round(w/d) + 8, 0, 15)
 * with IEEE fp32 division and round-half-away-from-zero; an all-zero block has
 * d = 0 and q = 8.  The canonical serialized block is 18 bytes: d as binary16
 * little-endian, then 16 bytes where byte j holds q_j in its low nibble and
 * q_{j+16} in its high nibble.  Blocks of row n follow in ascending K; rows in
 * ascending n.  Inside the library the weights live in a private device layout
 * (tiled for coalesced, 16-byte-aligned streaming); only the canonical form is
 * exchanged across this boundary.
 *
 * Conventions for every entry point:
 *  - All functions return an int status (Q4_OK on success), never throw and
 *    never trap the device.  Invalid arguments are rejected on the host before
 *    any launch.
 *  - "device" pointers are CUDA global-memory pointers on the current device;
 *    "host" pointers are ordinary CPU memory.  The caller owns x, y, idx,
 *    maxval and all host buffers.  A q4_weight is owned by the library from
 *    its creation (q4_quantize / q4_import_blocks) until q4_weight_free.
 *  - Compute calls are asynchronous on `stream` (0 = the legacy default
 *    stream) and do not synchronize the host.  A kernel fault from an earlier
 *    call surfaces as Q4_ERR_CUDA on a later call.
 *  - Compute calls use a per-device scratch area owned by the library (split-K
 *    partial sums, the activation operand of the tensor-core path, argmax
 *    keys).  Creating a weight (q4_quantize, q4_import_blocks) reserves the
 *    largest scratch that any single-weight call on it can need, at any M and
 *    with any flags, so q4mm_forward, q4mm_forward_ex and q4mm_argmax on a
 *    created weight never allocate.  A grouped or gated call (its weights'
 *    tiles summed) grows the scratch on its first call of a larger shape
 *    (cudaFree, cudaMalloc, a device synchronize): make one such call of each
 *    shape before capturing a CUDA graph.  Calls that
 *    share that scratch must be ordered on one stream; calls on different
 *    streams that overlap on the GPU race on it.
 *  - Every device-side wait in the kernels is bounded; a wait that runs out
 *    records Q4_ERR_TIMEOUT in a device status word that q4_device_status()
 *    returns.
 */
#ifndef Q4MM_H
#define Q4MM_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define Q4_API __attribute__((visibility("default")))
#else
#define Q4_API
#endif

/* ---- status codes ---- */
#define Q4_OK 0
#define Q4_ERR_INVALID_ARG 1  /* null pointer, negative size, wrong device, bad flag */
#define Q4_ERR_SHAPE 2        /* K not a multiple of 32 in [32, 32*65535], N not in [1, 128*65535], M above Q4MM_M_MAX */
#define Q4_ERR_ALIGN 3        /* a device pointer not 16-byte aligned */
#define Q4_ERR_NONFINITE 4    /* a weight is NaN or infinite (quantize), or a stored scale is */
#define Q4_ERR_RANGE 5        /* a block scale does not fit binary16 (|d| >= 65520) */
#define Q4_ERR_CUDA 6         /* a CUDA runtime error (launch failure, sticky fault) */
#define Q4_ERR_TIMEOUT 7      /* a bounded device-side wait ran out */
#define Q4_ERR_NOMEM 8        /* device allocation failed */
#define Q4_ERR_UNSUPPORTED 9  /* the device is not sm_103 / requested path unavailable */

/* ---- flags for the _ex entry points ---- */
/* Bit-identical output rows: row r of y depends only on x[r,:] and W, never on
 * M, on r's position in the batch or on the other rows' values.  The calls
 * then run the streaming kernel for every M, in launches of at most 8 rows,
 * with the CTA layout and the K partition fixed per weight shape; a row's
 * operations do not depend on the MMA column it occupies (§"The Other Request
 * Already Finished": a 120-prefill + 4-verify batch crossed the kernel-switch
 * threshold and changed the cached numbers).
 * With Q4MM_FORCE_TC as well, the calls run the tensor-core kernel for every
 * M instead, with one instruction shape (token tiles of 64 rows) and a K
 * partition fixed per weight shape: rows are again bit-identical whatever M
 * is (but not equal to the streaming mode's), large batches read the weights
 * once per 256 rows instead of once per 8, and small ones pay the tensor-core
 * kernel's fixed cost. */
#define Q4MM_BATCH_INVARIANT 0x1u
/* Force the CUDA-core streaming kernel (no tensor cores). */
#define Q4MM_FORCE_SIMT 0x2u
/* Force the tcgen05/TMEM tensor-core kernel (the large-M path). */
#define Q4MM_FORCE_TC 0x4u
/* Ablation: one launch per activation row with the CUDA-core kernel, the
 * row-by-row fallback of §"Row-by-Row GEMV to the Rescue". */
#define Q4MM_ROW_BY_ROW 0x8u
/* Force the streaming mma.sync kernel (the measured small/medium-M path). */
#define Q4MM_FORCE_MMA 0x10u

/* Largest M accepted by one call. */
#define Q4MM_M_MAX 4096

/* Kernel paths reported by q4mm_select_path. */
#define Q4MM_PATH_SIMT 1
#define Q4MM_PATH_TC 2
#define Q4MM_PATH_ROW_BY_ROW 3
#define Q4MM_PATH_MMA 4

typedef struct q4_weight q4_weight;

/* Quantize an fp32 weight matrix already on the device.
 *   w      device, fp32 [N, K] row-major, 16-byte aligned; read only.
 *   N, K   N >= 1 output rows; K >= 32 and a multiple of 32.
 *   out    receives a new handle (library-owned) on Q4_OK; untouched otherwise.
 * Synchronizes `stream` to report Q4_ERR_NONFINITE / Q4_ERR_RANGE (this is an
 * off-step operation), and reserves the device scratch of the single-weight
 * calls on the new weight (Q4_ERR_NOMEM, with no handle, if that fails).  The
 * blocks are byte-identical to the canonical rule in the file header. */
Q4_API int q4_quantize(const float* w, int64_t N, int64_t K, q4_weight** out, cudaStream_t stream);

/* Create a handle from canonical blocks in host memory (N*K/32*18 bytes).
 * Rejects blocks whose scale is not finite (Q4_ERR_NONFINITE).  Synchronous;
 * reserves scratch as q4_quantize does. */
Q4_API int q4_import_blocks(const void* host_blocks, int64_t N, int64_t K, q4_weight** out,
                     cudaStream_t stream);

/* Write the canonical blocks (N*K/32*18 bytes) of W to host memory.
 * bytes must be at least that size.  Synchronous. */
Q4_API int q4_export_blocks(const q4_weight* W, void* host_blocks, size_t bytes);

/* Release a handle and its device memory (after the work that uses it). */
Q4_API int q4_weight_free(q4_weight* W);

/* Shape and device footprint of a handle. */
Q4_API int q4_weight_shape(const q4_weight* W, int64_t* N, int64_t* K);
Q4_API int q4_weight_device_bytes(const q4_weight* W, size_t* bytes);

/* y = x @ W^T.
 *   x   device, fp32 [M, K] row-major, 16-byte aligned.
 *   y   device, fp32 [M, N] row-major, 16-byte aligned; fully overwritten.
 *   M   0 <= M <= Q4MM_M_MAX; M = 0 is a no-op returning Q4_OK.
 * Picks the kernel from the measured M threshold (q4mm_get_m_threshold).
 * Result per element within 1e-5 * sum_k |w x| + 1e-6 of the exact value. */
Q4_API int q4mm_forward(const q4_weight* W, const float* x, float* y, int64_t M, cudaStream_t stream);

/* q4mm_forward with Q4MM_* flags (batch-invariant mode, forced path, ablation). */
Q4_API int q4mm_forward_ex(const q4_weight* W, const float* x, float* y, int64_t M, uint32_t flags,
                    cudaStream_t stream);

/* Greedy pick per row (the LM-head use, §"Same Prompt, Different Story"):
 * idx[m] = argmax_n y[m, n] with the lowest index on exact ties and NaN never
 * winning, without writing y.
 *   idx     device, int32 [M].
 *   maxval  device, fp32 [M] receiving y[m, idx[m]], or NULL. */
Q4_API int q4mm_argmax(const q4_weight* W, const float* x, int32_t* idx, float* maxval, int64_t M,
                cudaStream_t stream);
Q4_API int q4mm_argmax_ex(const q4_weight* W, const float* x, int32_t* idx, float* maxval, int64_t M,
                   uint32_t flags, cudaStream_t stream);

/* Most weights one q4mm_forward_group call takes. */
#define Q4MM_GROUP_MAX 4

/* y_i = x @ W_i^T for up to Q4MM_GROUP_MAX weights that share K and the same
 * activations (the q, k and v projections, or the gate and up projections, of
 * one decoder layer), in one kernel launch per 16 token rows (8 when the
 * group's tiles outnumber the SMs) instead of one per weight: the activations
 * are staged once and the fixed cost of a launch is
 * paid once ("Why LLM Decoding Is Slow, and Why Batching Is (Almost) Free",
 * §4: every weight is still read exactly once per call).
 *   W       host array of `count` handles, all with the same K, on the current
 *           device; 1 <= count <= Q4MM_GROUP_MAX.
 *   x       device, fp32 [M, K] row-major, 16-byte aligned.
 *   y       host array of `count` device pointers, y[i] fp32 [M, N_i],
 *           16-byte aligned, fully overwritten; distinct, non-overlapping.
 *   flags   0, Q4MM_FORCE_MMA, Q4MM_FORCE_TC and/or Q4MM_BATCH_INVARIANT
 *           (others, or FORCE_MMA with FORCE_TC: INVALID_ARG; FORCE_TC off
 *           sm_103: UNSUPPORTED).
 * Each y_i is within the q4mm_forward tolerance.  The K partition depends on
 * the group's shapes (not on M), so in batch-invariant mode row r of every y_i
 * is bit-identical whatever M is; it may differ in the last bits from a
 * single-weight call of the same W_i.  At or above the group M threshold
 * (q4mm_get_group_m_threshold; without flags) the call runs the tensor-core
 * kernel instead, again as one launch (with its activation pre-pass) over the
 * tiles of the whole group. */
Q4_API int q4mm_forward_group(const q4_weight* const* W, int count, const float* x, float* const* y,
                              int64_t M, uint32_t flags, cudaStream_t stream);

/* The hidden state of a gated MLP in one call:
 *   h[M,N] = SiLU(x Wg^T) * (x Wu^T),  SiLU(z) = z / (1 + exp(-z)),
 * with Wg, Wu the gate and up projections (same N and K, same device) and x
 * fp32 [M,K] as for q4mm_forward; h fp32 [M,N] row-major, device, 16-byte
 * aligned, caller-owned, fully overwritten.  The pages name the gate/up/down
 * projections of Qwen2.5-7B but not the step between them; this is that
 * model's gated MLP.  Fusing it into the matmul follows "Why LLM Decoding Is
 * Slow, and Why Batching Is (Almost) Free" (§3 "The Real Constraint: Two
 * Ceilings": small elementwise ops around the matmuls cost time of their
 * own): on the streaming path (M below the group M threshold) each CTA
 * computes the gate and up rows of the same row range and writes only h; g
 * and u never reach memory.  On the tensor-core path and in batch-invariant
 * mode the grouped call writes g and u to library scratch and one elementwise
 * pass forms h.
 *   flags   as for q4mm_forward_group.
 * Each element is within the gate and up tolerances propagated through SiLU
 * (SiLU is 1.1-Lipschitz) plus fp32 rounding; in batch-invariant mode row r
 * of h is bit-identical whatever M is.  The streaming path takes up to 8
 * token rows per launch.  Errors as for q4mm_forward_group; mismatched shapes
 * or devices: INVALID_ARG. */
Q4_API int q4mm_forward_gated(const q4_weight* Wg, const q4_weight* Wu, const float* x, float* h,
                              int64_t M, uint32_t flags, cudaStream_t stream);

/* Capacity of the split-K partial sums of q4mm_forward_noalloc (2400 KiB). */
#define Q4MM_NOALLOC_PARTIAL_BYTES 2457600

/* y = x @ W^T without allocating any device memory.  (The pages have no
 * counterpart: this is a library concern.)
 *
 * The other compute calls draw on a library scratch that is reserved with
 * cudaMalloc when a weight is created and, for grouped and gated calls, grown
 * (cudaFree, cudaMalloc) on the first call that needs more.  Callers that
 * cannot allocate at those moments use this call instead: a serving process
 * that gave all free device memory to its own pool (the allocation would
 * fail), or a step that must not wait for the whole device, as cudaFree does.  Its scratch is one
 * fixed device array in the library (about 2.5 MB per device, created when the
 * library's device code is loaded), so this call allocates nothing.  (As for
 * any CUDA library, the runtime may still load kernel code on first use.)
 *
 *   x, y, M   as q4mm_forward; y is fully overwritten.
 * Always runs the streaming mma.sync kernel with its usual K partition: the
 * results are bit-identical to q4mm_forward_ex(W, x, y, M, Q4MM_FORCE_MMA).
 * Returns Q4_ERR_SHAPE, before any launch, if the call's split-K partial
 * sums (splits x min(M, 16) x N rounded up to 128 x 8 bytes) exceed
 * Q4MM_NOALLOC_PARTIAL_BYTES.  On a 152-SM GB300 every linear layer of a
 * 7B decoder (N, K up to 18944) fits at any M; q4mm_forward has no such limit.
 *
 * The first call on each device sets up: it looks up the array's address,
 * clears the counters that must start at zero and synchronizes the device
 * once.  Make that first call before any stream capture begins.
 * All calls on one device share the one array: calls whose kernels overlap on
 * the GPU (other streams, other host threads) race on it and give wrong
 * results.  Order them on one stream.  A bounded device-side wait that runs
 * out is recorded in this array's own status word (y is then unspecified);
 * q4_device_status reads and clears that word together with the ordinary
 * one, with two 4-byte copies and no allocation. */
Q4_API int q4mm_forward_noalloc(const q4_weight* W, const float* x, float* y, int64_t M,
                                cudaStream_t stream);

/* Greedy pick for selected rows of a ragged continuous-batching step: only
 * the rows that need logits (the last prefill row of a request, its verify
 * rows, decode rows) go through the LM head, without gathering them first.
 *   x       device, fp32 [x_rows, K] row-major, 16-byte aligned (the step's
 *           hidden states); 1 <= x_rows <= INT32_MAX.
 *   rows    device, int32 [R]: the x row of each output; an index outside
 *           [0, x_rows) reads zeros and makes the next q4_device_status()
 *           return Q4_ERR_INVALID_ARG (it is checked on the device, never read
 *           out of bounds).
 *   idx     device, int32 [R]; maxval device, fp32 [R] or NULL.
 *   R       0 <= R <= Q4MM_M_MAX.
 * Same result as q4mm_argmax on the gathered rows (streaming kernel). */
Q4_API int q4mm_argmax_rows(const q4_weight* W, const float* x, int64_t x_rows, const int32_t* rows,
                            int64_t R, int32_t* idx, float* maxval, cudaStream_t stream);

/* Greedy verification of speculative draft tokens, one result per request:
 * accepted[s] = the number of leading positions j of request s's segment
 * [offsets[s], offsets[s+1]) with idx[j] == draft[j] (the request keeps the
 * drafts up to the first disagreement), or -1 if the segment is malformed
 * (decreasing offsets, or outside [0, total)).
 *   idx, draft  device, int32 [total] (idx from q4mm_argmax / _rows; draft[j]
 *               the token proposed at the position idx[j] predicts).
 *   offsets     device, int32 [S + 1].  accepted: device, int32 [S]. */
Q4_API int q4_verify_greedy(const int32_t* idx, const int32_t* draft, int64_t total,
                            const int32_t* offsets, int64_t S, int32_t* accepted,
                            cudaStream_t stream);

/* KV-cache append of one continuous-batching step into a preallocated cache
 * ("A non-contiguous KV cache cuts Qwen2 decode speed by 59 % at 2k context in
 * Candle on Metal", §"Cause and workaround": a cache that grows by
 * concatenation re-copies itself on every append when the new V rows are a
 * strided view; writing only the new rows into a buffer that is already in
 * place does not).  One launch writes the new K and V rows of every layer and
 * every request; nothing already cached is read or moved.
 *   k_cache, v_cache  device, [layers][slots][heads][capacity][head_dim]
 *                     elements of elem_bytes (2 or 4) each, contiguous,
 *                     caller-owned; slot sl's position p of (layer, head) is
 *                     one head_dim row.
 *   k_new, v_new      device, the step's new rows: K element (l, t, h, d) at
 *                     k_new + l*k_strides[0] + t*k_strides[1] +
 *                     h*k_strides[2] + d (host arrays of 3 strides, in
 *                     elements, head_dim contiguous), V likewise with
 *                     v_strides; t over the step's packed rows [0, total).  A
 *                     transposed or otherwise strided view (such as V after
 *                     prefill) is read in place.
 *   offsets           device, int32 [S + 1], non-decreasing: request s owns
 *                     packed rows [offsets[s], offsets[s+1]); rows outside
 *                     every request are not cached.
 *   slot, pos         device, int32 [S]: request s's cache slot and the
 *                     position of its first new row (its current length).
 *                     Row offsets[s] + j goes to position pos[s] + j; the
 *                     caller advances its lengths.
 * Host-checked: sizes >= 1 (layers, slots, heads, head_dim, capacity below
 * 2^31; S and total below 2^31 - 1; total * head_dim * elem_bytes / 16 and
 * 2 * layers * heads below 2^31 - 1), elem_bytes 2 or 4, stride arrays given
 * and every stride in [0, 2^59) (INVALID_ARG); head_dim * elem_bytes, every
 * stride * elem_bytes and every base address multiples of 16 bytes (ALIGN).  S = 0 or total = 0: a no-op.
 * On the device, a request whose slot is outside [0, slots), whose position
 * is negative, or whose rows would pass capacity or total is not written at
 * all (the other requests are) and q4_device_status then reports
 * Q4_ERR_INVALID_ARG.  Asynchronous on stream; the same bytes as the source,
 * whatever the element type. */
Q4_API int q4_kv_append(void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                        int64_t layers, int64_t slots, int64_t heads, int64_t head_dim,
                        int64_t capacity, int elem_bytes, const int64_t* k_strides,
                        const int64_t* v_strides, const int32_t* offsets, const int32_t* slot,
                        const int32_t* pos, int64_t S, int64_t total, cudaStream_t stream);

/* The kernel path (Q4MM_PATH_*) a call with these arguments would take, or a
 * negative status. */
Q4_API int q4mm_select_path(const q4_weight* W, int64_t M, uint32_t flags);

/* Plan of a call with these arguments, without running it: *path receives
 * the Q4MM_PATH_* value, *launches the number of kernel launches the call
 * makes (on the streaming path including the passes that convert the
 * activations of a launch once for all its CTAs), *splits the K partition
 * count of the first launch of a
 * q4mm_forward_ex call (1 when the streaming kernel gives each CTA one 32-row
 * group pair over the whole K, which it does for launches of up to 8 rows).
 * Any output pointer may be NULL. */
Q4_API int q4mm_plan_info(const q4_weight* W, int64_t M, uint32_t flags, int* path, int* launches,
                          int* splits);

/* The M threshold: calls with M >= threshold take the tcgen05 path, smaller M
 * the streaming mma.sync path (the kernel-switch threshold that
 * §"Row-by-Row GEMV to the Rescue" says must be measured, not assumed).
 * The default is the value measured on GB300; set_m_threshold overrides it for
 * the process (1 = always tensor cores; Q4MM_M_MAX + 1 = never). */
Q4_API int q4mm_set_m_threshold(int64_t m);
Q4_API int64_t q4mm_get_m_threshold(void);

/* The M threshold of q4mm_forward_group: at or above it one tcgen05 launch
 * covers the whole group, below it one streaming launch per 16 token rows (8
 * when the group's tiles outnumber the SMs).
 * The default is the crossover measured on GB300 over a 7B layer's q/k/v and
 * gate/up groups.  Same range and errors as set_m_threshold. */
Q4_API int q4mm_set_group_m_threshold(int64_t m);
Q4_API int64_t q4mm_get_group_m_threshold(void);

/* Test settings for the bounded waits (process-wide; the defaults are the
 * library's normal behaviour).  Every wait a kernel makes on another of its
 * roles or CTAs gives up after a bound, 1 s by default, records
 * Q4_ERR_TIMEOUT for q4_device_status and lets the kernel return instead of
 * hanging.
 *   q4mm_set_wait_limit_ns  sets that bound (0 restores 1 s) for later
 *                           launches; the split-K polls scale with it.
 *   q4mm_set_stall_for_test when on, later launches withhold their first
 *                           hand-off (the converter warps hand over no chunk,
 *                           the CTAs of a K split store no partial sum, the
 *                           tensor-core producer issues no copy), so that the
 *                           waiting side waits for something nothing sets and
 *                           its bound runs out.  Outputs are then unspecified.
 * Launches with no wait (one K split with the activations converted up front)
 * are unaffected.  Only tests need these. */
Q4_API int q4mm_set_wait_limit_ns(uint64_t ns);
Q4_API int q4mm_set_stall_for_test(int on);

/* Synchronize the current device and return (then clear) the device status
 * words (the library's scratch and, once q4mm_forward_noalloc has run on the
 * device, its fixed array): Q4_OK; Q4_ERR_TIMEOUT if a bounded wait in a kernel ran out
 * (the library's scratch words are then reset for the calls that follow);
 * Q4_ERR_INVALID_ARG if q4mm_argmax_rows met a row index out of range; or
 * Q4_ERR_CUDA if the device reports an error. */
Q4_API int q4_device_status(void);

/* Bytes of the library's device scratch on the current device, as now held:
 * split-K partial sums, the tensor-core activation operand, the grouped or
 * gated calls' g/u outputs and the streaming kernel's pre-converted
 * activations.  All four pointers must be non-null (else Q4_ERR_INVALID_ARG);
 * zeros before the device's first call.  Host-only. */
Q4_API int q4_scratch_bytes(size_t* partial, size_t* xop, size_t* gu, size_t* xpre);

/* Human-readable name of a status code (static storage). */
Q4_API const char* q4_status_string(int status);

#ifdef __cplusplus
}
#endif
#endif /* Q4MM_H */
