/*
 * l3.h — C ABI of a Large Lookup Layer (L³) library for NVIDIA B300 (sm_103a).
 *
 * The layer is the one described in "L³: Large Lookup Layers" (Tseng, De Sa;
 * arXiv:2601.21461). Its gist.science explainer, Technical Summary:
 *   - "Core Architecture": the layer takes a hidden state x and a token id t. Static
 *     routing maps t to a fixed subset of a large embedding table (here: the contiguous
 *     CSR row range offs[t] .. offs[t+1]-1 of a key table K and a value table V). The
 *     output is  y = W_mix [ LayerNorm( W_up( V_tᵀ Softmax(K_t x) ) ) ; x ].
 *   - "Information-Theoretic Embedding Allocation": a budget of v rows is spread over
 *     the vocabulary; every token gets at least 1 and at most k rows.
 *   - "Systems-Friendly Design", batch sorting: sorting a batch by token id makes the
 *     layer's attention mask block-diagonal; the library sorts every batch and works
 *     on the segments of equal ids.
 *
 * Conventions shared by every entry point:
 *   - All pointers named *_host are host memory; every other pointer is device memory
 *     on the current CUDA device. The caller owns all memory. The library never
 *     allocates device memory: scratch comes from a caller-provided workspace sized by
 *     l3_workspace_size (l3_route_noalloc alone uses a fixed array the library declares).
 *   - Device work is enqueued asynchronously on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream). Argument errors are returned before anything is enqueued.
 *   - Matrices are dense row-major. Element types: L3_F32 (float) or L3_BF16 (bfloat16,
 *     accumulation in fp32).
 *   - Errors found on the device (a token id outside [0, vocab), a bad offsets table, a
 *     bounded wait that ran out) never trap: a kernel records them in the workspace's
 *     status words, and l3_get_error reports them. Every call clears the status words of
 *     its workspace when it starts, so l3_get_error reports the most recent call. The
 *     output rows concerned are then unspecified.
 *   - A workspace (and a saved-state buffer) must not be used by two calls that can run
 *     at the same time. No C++ exception crosses this interface.
 */
#ifndef L3_H_
#define L3_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define L3_ABI_VERSION 2

typedef struct CUstream_st* l3_stream_t; /* = cudaStream_t */
typedef struct CUevent_st* l3_event_t;   /* = cudaEvent_t  */

typedef enum l3_status {
  L3_OK = 0,
  L3_ERR_INVALID_ARG = 1, /* null pointer, bad size or shape                          */
  L3_ERR_INFEASIBLE = 2,  /* allocation: vocab*n_min <= v <= vocab*n_max does not hold */
  L3_ERR_UNSUPPORTED = 3, /* shape outside what the kernels handle (see l3_layer)       */
  L3_ERR_WORKSPACE = 4,   /* workspace smaller than l3_workspace_size, or (device-found)
                             a row output smaller than the rows a batch touches           */
  L3_ERR_TOKEN_RANGE = 5, /* a token id was outside [0, vocab)          (device-found)  */
  L3_ERR_CUDA = 6,        /* a CUDA runtime call failed                                 */
  L3_ERR_LAYER = 7,       /* offsets not 0 = offs[0] < ... < offs[vocab] = v, or a range
                             longer than k_max                           (device-found) */
  L3_ERR_TIMEOUT = 8      /* a bounded device-side wait gave up, or a kernel found its
                             work plan inconsistent and stopped          (device-found) */
} l3_status;

enum { L3_F32 = 0, L3_BF16 = 1 };

/*
 * A layer: its shapes and its parameters (device pointers, caller-owned).
 *   offs   [vocab+1] int32   CSR offsets; token id t owns rows offs[t] .. offs[t+1]-1.
 *                            Must hold 0 = offs[0] < offs[1] < ... < offs[vocab] = v and
 *                            offs[t+1] - offs[t] <= k_max (l3_check_layer verifies).
 *   K      [v, d]     dtype  key table
 *   V      [v, d_v]   dtype  value table
 *   W_up   [d, d_v]   dtype  (out x in): u = W_up a
 *   W_mix  [d, 2d]    dtype  (out x in): y = W_mix [h; x]; columns 0..d-1 act on the
 *                            LayerNorm output h, columns d..2d-1 on x.
 * Supported: 1 <= k_max <= 512; d and d_v multiples of 64 with 64 <= d <= 2048 and
 * 64 <= d_v <= 512; v < 2^31; vocab < 2^31. LayerNorm is over the d features, biased
 * variance, no affine, epsilon ln_eps (> 0; 1e-5 is the usual value).
 */
typedef struct l3_layer {
  int64_t vocab;
  int64_t v;
  int64_t d;
  int64_t d_v;
  int32_t k_max;
  int32_t dtype; /* L3_F32 or L3_BF16 */
  float ln_eps;
  int32_t reserved; /* set to 0 */
  const int32_t* offs;
  const void* K;
  const void* V;
  const void* W_up;
  const void* W_mix;
} l3_layer;

/* Passes for l3_workspace_size. */
enum {
  L3_PASS_FORWARD = 0,
  L3_PASS_BACKWARD = 1,
  L3_PASS_FORWARD_HOST = 2,
  L3_PASS_BACKWARD_ROWS = 3,
  L3_PASS_STAGE = 4
};

/* Stages of l3_forward, for l3_forward_timed. */
enum {
  L3_STAGE_ROUTE = 0,       /* sort the batch by token id, build segments and work plan */
  L3_STAGE_ATTEND = 1,      /* a = V_tᵀ softmax(K_t x), tokens of short segments        */
  L3_STAGE_ATTEND_LONG = 2, /* the same for tokens of long segments (large bf16 batches) */
  L3_STAGE_UP = 3,          /* u = W_up a, LayerNorm statistics                         */
  L3_STAGE_MIX = 4,         /* y = W_mix [LayerNorm(u); x]                              */
  L3_FWD_STAGES = 5
};

/*
 * Row allocation (host only, synchronous; touches no GPU). Explainer, Technical Summary,
 * "Information-Theoretic Embedding Allocation": each of the vocab token ids gets n_t rows
 * with n_min <= n_t <= n_max and sum n_t = v; frequent ids get more. The corpus-driven
 * Algorithm 1 is not given on the pages; this is the frequency rule the library uses:
 *   w_t = pow(freq[t], power); a water level c solves sum_t clamp(c w_t, n_min, n_max) = v
 *   (200 bisection steps locate the clamped sets, then c is solved exactly for them, the
 *   free weights summed in increasing id order); the real targets are rounded by largest
 *   remainder (among ids below n_max; ties go to the lower id).
 * Writes offs_out[0..vocab] (exclusive prefix sum of n_t: offs_out[0] = 0,
 * offs_out[vocab] = v). freq: [vocab] positive finite values (any scale).
 * Errors: L3_ERR_INVALID_ARG (null pointer, vocab < 1, n_min < 1, n_max < n_min,
 * non-positive or non-finite freq, non-finite power, v >= 2^31), L3_ERR_INFEASIBLE.
 */
l3_status l3_alloc_offsets(const double* freq, int64_t vocab, int64_t v, int32_t n_min,
                           int32_t n_max, double power, int32_t* offs_out);

/*
 * Token frequencies of a stream of token ids, the statistic the allocation follows
 * (explainer, "Information-Theoretic Embedding Allocation": frequent tokens get more
 * rows). A stream of ids stands in for the training corpus; the corpus-driven Algorithm 1
 * itself is not on the pages.
 *   ids     [n] int32 token ids (device), 0 <= n < 2^31
 *   counts  [vocab] int64 out (device): counts[t] = occurrences of id t (overwritten)
 *   ws      >= 256 bytes of device memory for the status words
 * Ids outside [0, vocab) are not counted; l3_get_error(ws, stream) then reports
 * L3_ERR_TOKEN_RANGE. The counts are exact (integer atomics) and independent of order.
 */
l3_status l3_count_ids(const int32_t* ids, int64_t n, int64_t vocab, int64_t* counts, void* ws,
                       size_t ws_bytes, l3_stream_t stream);

/*
 * l3_alloc_offsets with freq[t] = counts_host[t] + smoothing (host only, synchronous).
 * Add-smoothing gives ids that never occurred a positive frequency (they end up with the
 * fewest rows). counts_host: [vocab] int64 >= 0 (from l3_count_ids); smoothing >= 0, and
 * with smoothing = 0 every count must be positive. Errors as l3_alloc_offsets.
 */
l3_status l3_alloc_offsets_counts(const int64_t* counts_host, int64_t vocab, int64_t v,
                                  int32_t n_min, int32_t n_max, double power, double smoothing,
                                  int32_t* offs_out);

/* Bytes of workspace a call needs (pass: L3_PASS_*), 0 if the layer is invalid. */
size_t l3_workspace_size(const l3_layer* layer, int64_t T, int32_t pass);

/* Bytes of the saved-state buffer l3_forward fills for l3_backward. */
size_t l3_saved_size(const l3_layer* layer, int64_t T);

/*
 * Check the offsets table on the device (static routing must map every id to a
 * non-empty range of at most k_max rows inside [0, v)). Synchronises `stream`.
 * Returns L3_OK, L3_ERR_LAYER, or an argument/CUDA error. ws: >= l3_workspace_size(
 * layer, 0, L3_PASS_FORWARD) bytes.
 */
l3_status l3_check_layer(const l3_layer* layer, void* ws, size_t ws_bytes, l3_stream_t stream);

/*
 * Batch sorting (explainer, "Systems-Friendly Design"): stable sort of the T token ids
 * and the segments of equal ids.
 *   ids        [T]    int32 token ids (device)
 *   perm       [T]    int32 out: perm[q] = original index of the q-th token in sorted order
 *                     (equal ids keep their batch order)
 *   seg_start  [T+1]  int32 out: segment s spans sorted positions seg_start[s] ..
 *                     seg_start[s+1]-1; entries past n_seg are unspecified
 *   seg_id     [T]    int32 out: token id of segment s (increasing in s)
 *   n_seg      [1]    int32 out: number of segments (distinct ids)
 * Any output pointer may be NULL to skip that copy. T may be 0.
 */
l3_status l3_route(const l3_layer* layer, const int32_t* ids, int64_t T, int32_t* perm,
                   int32_t* seg_start, int32_t* seg_id, int32_t* n_seg, void* ws,
                   size_t ws_bytes, l3_stream_t stream);

/*
 * l3_route_noalloc: l3_route without a workspace. The paper has no counterpart to this
 * entry point; it exists for callers that cannot allocate device memory when they need
 * the sort — for example a plugin inside a host program that owns every device
 * allocation and offers no hook for more, or a latency-critical loop that must not enter
 * an allocator. Its scratch is a fixed array of about 1 MiB declared by the library in
 * device memory (each GPU that loads the library holds it until the process exits);
 * nothing is allocated or freed by this call.
 *   ids, perm, seg_start, seg_id: as for l3_route (perm, seg_start, seg_id may be NULL)
 *   n_seg  [1] int32 out, required: the number of segments, or -1 if some token id was
 *          outside [0, vocab) (the other outputs are then unspecified)
 * Only layer->vocab is read. T may be 0; T > 65536 returns L3_ERR_WORKSPACE. The first
 * call on a device looks up the array's device address with that device current, so
 * make that first call before any stream capture. That address is kept for the life of
 * the process: after a cudaDeviceReset of a device, this entry point must not be called
 * on it again (the array may then live elsewhere). Every call shares the one array and
 * clears its status words on entry; calls whose GPU work overlaps (on streams with no
 * ordering between them) race on it.
 */
l3_status l3_route_noalloc(const l3_layer* layer, const int32_t* ids, int64_t T,
                           int32_t* perm, int32_t* seg_start, int32_t* seg_id,
                           int32_t* n_seg, l3_stream_t stream);

/*
 * Forward pass (explainer, "Core Architecture", the layer formula), for each token i:
 *   s = K_t x_i (t = ids[i]); p = softmax(s) (no temperature); a_i = V_tᵀ p;
 *   u_i = W_up a_i; h_i = LayerNorm(u_i); y_i = W_mix [h_i; x_i].
 *   ids   [T]    int32 (device)
 *   x     [T, d] layer dtype, 16-byte aligned
 *   y     [T, d] y_dtype (L3_F32, or the layer dtype), 16-byte aligned
 *   saved nullable; if given, l3_saved_size(layer, T) bytes that l3_backward reads
 *   ws    >= l3_workspace_size(layer, T, L3_PASS_FORWARD) bytes
 * x and y rows are moved by TMA tensor copies, whose global addresses must be 16-byte
 * aligned; a misaligned x or y returns L3_ERR_INVALID_ARG.
 * T may be 0 (nothing is enqueued). Errors: L3_ERR_INVALID_ARG, L3_ERR_UNSUPPORTED,
 * L3_ERR_WORKSPACE, L3_ERR_CUDA; token ids out of range are reported by l3_get_error.
 */
l3_status l3_forward(const l3_layer* layer, const int32_t* ids, int64_t T, const void* x,
                     void* y, int32_t y_dtype, void* saved, void* ws, size_t ws_bytes,
                     l3_stream_t stream);

/*
 * l3_forward, recording events[k] on `stream` before stage k (k < L3_FWD_STAGES) and
 * events[L3_FWD_STAGES] after the last stage: the elapsed time between events[k] and
 * events[k+1] is stage k. events: L3_FWD_STAGES+1 created cudaEvent_t handles.
 */
l3_status l3_forward_timed(const l3_layer* layer, const int32_t* ids, int64_t T,
                           const void* x, void* y, int32_t y_dtype, void* saved, void* ws,
                           size_t ws_bytes, l3_stream_t stream, l3_event_t* events);

/*
 * l3_forward on HOST buffers: copies ids_host [T] int32 and x_host [T, d] (layer dtype)
 * to the device, runs the forward and copies y back to y_host [T, d] (y_dtype), all
 * enqueued on `stream` (one cudaMemcpyAsync per buffer). Host buffers should be pinned
 * for asynchronous copies; the caller synchronises `stream` before reading y_host.
 * ws: >= l3_workspace_size(layer, T, L3_PASS_FORWARD_HOST) bytes (holds the device
 * copies as well as the forward's scratch).
 */
l3_status l3_forward_host(const l3_layer* layer, const int32_t* ids_host, int64_t T,
                          const void* x_host, void* y_host, int32_t y_dtype, void* ws,
                          size_t ws_bytes, l3_stream_t stream);

/*
 * Backward pass: gradients of sum(dy * y) for the layer formula, given the `saved` state
 * of an l3_forward call on the same layer, ids and x.
 *   dy       [T, d]      layer dtype
 *   dx       [T, d]      fp32 out
 *   dK       [v, d]      fp32 out; rows of ids absent from the batch are zero
 *   dV       [v, d_v]    fp32 out; likewise
 *   dW_up    [d, d_v]    fp32 out
 *   dW_mix   [d, 2d]     fp32 out
 * Every output is overwritten, not accumulated. dK and dV are deterministic segmented
 * sums: for each id, its rows' gradients are summed over that id's tokens in batch order,
 * with no floating-point atomics, so repeated calls give bitwise-identical results.
 * ws: >= l3_workspace_size(layer, T, L3_PASS_BACKWARD) bytes.
 */
l3_status l3_backward(const l3_layer* layer, const int32_t* ids, int64_t T, const void* x,
                      const void* dy, const void* saved, float* dx, float* dK, float* dV,
                      float* dW_up, float* dW_mix, void* ws, size_t ws_bytes,
                      l3_stream_t stream);

/*
 * Backward pass at batch scale for bf16 layers, with the table gradients of the rows the
 * batch touches only (a dense dK/dV of a large table would be mostly zeros): the gradients
 * of sum(dy * y) for the layer formula (explainer, "Core Architecture"), given the `saved`
 * state of an l3_forward call on the same layer, ids and x. Batch sorting (explainer,
 * "Systems-Friendly Design") makes each id's tokens one segment; each touched row's
 * gradient is the sum over its id's segment, in batch order.
 *   dy         [T, d]          bf16
 *   dx         [T, d]          fp32 out
 *   row_index  [max_rows]      int32 out: the touched table rows, ascending (the ranges
 *                              offs[t] .. offs[t+1]-1 of the batch's distinct ids)
 *   dK_rows    [max_rows, d]   fp32 out: row r holds dK of table row row_index[r]
 *   dV_rows    [max_rows, d_v] fp32 out
 *   n_rows     [1]             int32 out: touched rows (entries past it are unspecified)
 *   max_rows   capacity of the row outputs; min(v, T * k_max) always suffices. If the batch
 *              touches more rows, the rows past max_rows are not written and l3_get_error
 *              reports L3_ERR_WORKSPACE.
 *   dW_up      [d, d_v]        fp32 out;  dW_mix [d, 2d] fp32 out
 * Arithmetic: every product accumulates in fp32 on tensor cores. u = W_up a is recomputed
 * in fp32 (a split into bf16 hi + lo) with its LayerNorm statistics; du and da enter the
 * products that lead to the softmax gradients as bf16 hi + lo, and the weights p and their
 * gradients ds are fp32, entering the row-gradient products as bf16 hi + lo; h, x and dy
 * enter the weight gradients as bf16. Every output is overwritten and the result is
 * bitwise repeatable.
 * The plain products with the weight matrices and the weight gradients run on cuBLASLt
 * (its scratch inside `ws`); everything else runs in this library's kernels.
 * ws: >= l3_workspace_size(layer, T, L3_PASS_BACKWARD_ROWS) bytes. fp32 layers:
 * L3_ERR_UNSUPPORTED (l3_backward covers them).
 */
l3_status l3_backward_rows(const l3_layer* layer, const int32_t* ids, int64_t T, const void* x,
                           const void* dy, const void* saved, float* dx, int32_t* row_index,
                           float* dK_rows, float* dV_rows, int32_t* n_rows, int64_t max_rows,
                           float* dW_up, float* dW_mix, void* ws, size_t ws_bytes,
                           l3_stream_t stream);

/*
 * Staging of a batch's rows for tables kept in host memory (explainer, "Systems-Friendly
 * Design": the tables may live in CPU memory; static routing tells from the token ids alone
 * which rows a batch needs, so they can be fetched ahead, e.g. while earlier layers run).
 * Copies the rows of the batch's distinct ids into compact device tables and describes them
 * as a staged layer over which l3_forward gives the same outputs as over the full tables:
 *   layer       the full layer; K and V may be pinned host memory the device can address
 *               (cudaHostAlloc / cudaMallocHost, or cudaHostRegister'ed), or device memory;
 *               offs, W_up, W_mix are device memory
 *   ids         [T] int32 token ids of the batch (device), T >= 1
 *   K_stage     [max_rows, d], V_stage [max_rows, d_v] (device, layer dtype) out: the
 *               distinct ids' rows, in increasing id order
 *   max_rows    capacity, T <= max_rows <= T * k_max; the batch's touched rows plus T always
 *               suffice (the rows past the staged ones are given zeros, up to 128 of them).
 *               If the batch touches more rows, l3_get_error reports L3_ERR_WORKSPACE and
 *               the staged tables are incomplete.
 *   offs_stage  [T + 1] int32 out (device): staged offsets (staged id s = the s-th distinct
 *               id); ids_stage [T] int32 out (device): each token's staged id
 *   n_rows      [1] int32 out (device): rows staged
 *   staged      out (host struct): the staged layer: vocab T, v max_rows, offs offs_stage,
 *               K K_stage, V V_stage, the rest as `layer`; only ids_stage's ids are valid
 *               in it (the unused staged ids have one-row ranges past the staged rows)
 * ws: >= l3_workspace_size(layer, T, L3_PASS_STAGE) bytes. Asynchronous on `stream`.
 * Errors: L3_ERR_INVALID_ARG (also pageable host tables), L3_ERR_WORKSPACE, L3_ERR_CUDA.
 */
l3_status l3_stage_rows(const l3_layer* layer, const int32_t* ids, int64_t T, void* K_stage,
                        void* V_stage, int64_t max_rows, int32_t* offs_stage, int32_t* ids_stage,
                        int32_t* n_rows, l3_layer* staged, void* ws, size_t ws_bytes,
                        l3_stream_t stream);

/*
 * Synchronise `stream`, then read and clear the status words that the kernels of the
 * most recent call on `ws` wrote there. Returns L3_OK, L3_ERR_TOKEN_RANGE, L3_ERR_LAYER,
 * L3_ERR_TIMEOUT, L3_ERR_WORKSPACE or L3_ERR_CUDA (the first that applies, in that order
 * of priority after L3_ERR_CUDA).
 */
l3_status l3_get_error(void* ws, l3_stream_t stream);

/* Static string naming a status. */
const char* l3_status_string(l3_status status);

/*
 * Self-test of the bounded waits every kernel uses: enqueues one small kernel whose single
 * thread waits on a shared-memory barrier that nothing completes, with a limit of
 * limit_ns nanoseconds (1e3 .. 1e10). The wait gives up, records a timeout in the status
 * words at the start of `ws`, and the kernel returns; l3_get_error(ws, stream) then
 * reports L3_ERR_TIMEOUT and the device stays usable. ws_bytes must be at least 256.
 * Returns L3_ERR_INVALID_ARG (null ws, ws_bytes < 256, limit out of range), L3_ERR_CUDA,
 * or L3_OK once the kernel is enqueued.
 */
l3_status l3_selftest_wait_timeout(void* ws, size_t ws_bytes, int64_t limit_ns,
                                   l3_stream_t stream);

/* Kernels this library has launched in this process so far (host-side counter). */
uint64_t l3_launch_count(void);

/* L3_ABI_VERSION of the built library. */
int32_t l3_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* L3_H_ */
