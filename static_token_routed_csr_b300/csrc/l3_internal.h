// Internal interfaces between the C-ABI layer (l3_api.cu) and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "l3_common.cuh"

namespace l3 {

void count_launch(int n = 1);

// Raises `kernel`'s dynamic shared-memory limit to `bytes` for the current device. The
// attribute belongs to the device's context, so it is set once per (kernel, device) pair.
cudaError_t ensure_smem_attr(const void* kernel, int bytes);
template <typename K>
inline cudaError_t ensure_smem_attr(K* kernel, int bytes) {
  return ensure_smem_attr(reinterpret_cast<const void*>(kernel), bytes);
}
// Streaming multiprocessors of the current device (looked up once per device).
int device_sm_count();

// ---- routing (l3_route.cu) ---------------------------------------------------------------
struct RouteOut {
  int32_t* perm;       // [T]
  int32_t* seg_start;  // [T+1]
  int32_t* seg_id;     // [T]
  int32_t* n_seg;      // [1]
};
// Work plan of the gather-attend, built by the routing pass. Segments of equal ids with
// fewer than `th` tokens go to the split-row CUDA-core kernel: each is cut into groups of at
// most kPlanMT tokens, and each group's n_t rows into chunks of `ch` rows; groups are
// numbered in sorted order and their chunks prefix-summed. Segments of at least `th`
// tokens go to the tensor-core kernel as items of at most kTcNT tokens.
constexpr int kPlanMT = 8;
constexpr int kTcNT = 64;
struct alignas(16) AttendGroup {
  int32_t q0;    // first sorted position of the group's tokens
  int32_t mt;    // tokens in the group (1..mt_max)
  int32_t t;     // token id
  int32_t row0;  // offs[t]
  int32_t n;     // rows n_t (0 if the offsets were invalid for t: the group is skipped)
  int32_t c0;    // index of the group's first chunk among all chunks
  int32_t w0;    // cost units of all chunks before c0 (see PlanOut::w_chunk)
  int32_t pad;
  int32_t tok[kPlanMT];  // batch index of each token (0 past mt)
};
// The group that holds the first chunk of a CTA's range in the split-row kernel, copied
// out by the plan so that the kernel can issue its first copies after a single read.
struct alignas(16) CtaHead {
  int32_t g;    // group index
  int32_t q0, mt, n, row0, c0;
  int32_t c1;   // the group's end chunk (the next group's c0)
  int32_t row;  // table row of the range's first chunk
  int32_t tok[kPlanMT];
  int32_t cb, ce;  // the CTA's chunk range [cb, ce) (cta_start[b], cta_start[b + 1])
  int32_t pad[2];
};
struct AttendItem {
  int32_t q0;  // first sorted position
  int32_t nt;  // tokens (1..kTcNT)
  int32_t t;   // token id
  int32_t pad;
};
// hdr words written by the plan
enum { kPlanGroups = 0, kPlanChunks = 1, kPlanItems = 2, kPlanHdrWords = 4 };
struct PlanOut {
  AttendGroup* groups;  // [T + 1]; entry n_groups carries only c0 = total chunks
  int32_t* hdr;         // [kPlanHdrWords]
  int32_t* counters;    // [T]: zeroed here, counted up by the split-row kernel
  AttendItem* items;    // [T / th + 1] (may be null when th > T)
  const int32_t* offs;
  int64_t v;
  int k_max;
  int ch;      // rows per chunk
  int mt_max;  // tokens per group (<= kPlanMT)
  int th;      // segments with at least th tokens go to the tensor-core kernel
  // Split of the chunk list over the n_cta CTAs of the split-row kernel, balanced by cost:
  // a chunk costs w_chunk units and each group start w_group more (the per-group work of
  // loading x and writing a). CTA b takes chunks [cta_start[b], cta_start[b+1]), which may
  // be empty; cta_group[b] is the group holding chunk cta_start[b].
  int32_t* cta_start;  // [n_cta + 1]
  int32_t* cta_group;  // [n_cta]
  CtaHead* cta_head;   // [n_cta]: the group holding chunk cta_start[b]
  int n_cta;
  int w_chunk, w_group;
};
size_t route_scratch_bytes(int64_t T);
cudaError_t launch_route(const int32_t* ids, int64_t T, int64_t vocab, void* scratch,
                         RouteOut out, DevStatus* st, cudaStream_t stream,
                         const uint64_t** sorted_keys, const PlanOut* plan = nullptr);

// ---- gather-attend, split rows (l3_attend.cu) ----------------------------------------------
struct AttendArgs {
  const uint64_t* sorted_keys;  // [T] (id << 32 | batch index), ascending
  int64_t T;
  const AttendGroup* groups;
  const int32_t* hdr;
  int32_t* counters;
  const void* K;
  const void* V;
  const void* x;
  int64_t v;             // table rows
  int d, d_v, ch;
  int dtype;             // L3_F32 / L3_BF16
  float* a_f32;          // [T, d_v] nullable, batch order
  __nv_bfloat16* a_bf16; // [T, d_v] nullable, batch order
  float* ml;             // [T, 2] nullable: (max score, softmax denominator)
  float* part;           // attend_part_floats(T, d_v) floats: partial (m, l, acc) per slot
  const int32_t* cta_start;  // the plan's split of the chunk list (PlanOut)
  const int32_t* cta_group;
  const CtaHead* cta_head;
  int n_cta;                 // grid of the split-row kernel
  DevStatus* st;
};
// Rows per chunk for a layer shape: 8 or 16 for bf16 layers (warp-MMA kernel), else as
// many as fit 40 KB of K and V rows (at most 8).
int attend_rows_per_chunk(int d, int d_v, int dtype);
int attend_mma_rows_per_chunk(int d, int d_v);
// Tokens per group of the split-row plan for a layer dtype.
int attend_group_tokens(int dtype);
size_t attend_part_floats(int d_v);
// Grid of the split-row kernel (at most kPlanMaxCtas) and the plan's cost weights for it.
constexpr int kPlanMaxCtas = 512;
int attend_split_ctas(int d, int d_v, int dtype);
void attend_split_weights(int d, int d_v, int dtype, int* w_chunk, int* w_group);
cudaError_t launch_attend_fwd(const AttendArgs& a, cudaStream_t stream);

// ---- gather-attend on tensor cores (l3_attend_tc.cu), the long segments of bf16 batches ----
struct AttendTcArgs {
  const uint64_t* sorted_keys;
  const AttendItem* items;
  const int32_t* hdr;       // plan header (item count)
  int64_t T;
  const int32_t* offs;
  const void* K;
  const void* V;
  const void* x;             // [T, d] bf16, 16-byte aligned (gathered by TMA)
  int64_t v;
  int d, d_v;
  int max_items;            // upper bound of the item count (0: no items)
  __nv_bfloat16* a_bf16;    // [T, d_v]
  float* a_f32;             // nullable
  float* ml;                // nullable
  DevStatus* st;
};
// Tokens per segment from which the tensor-core kernel takes a segment (0: never).
int attend_tc_threshold(int64_t T, int d, int d_v, int dtype);
cudaError_t launch_attend_tc(const AttendTcArgs& a, cudaStream_t stream);

// ---- SIMT GEMM and row kernels (l3_gemm_simt.cu) -------------------------------------------
// C[m, n] (fp32, row stride ldc) = alpha * sum_k A(m, k) B(k, n) + beta * C[m, n]
// with A(m, k) = A[m*a_sm + k*a_sk], B(k, n) = B[k*b_sk + n*b_sn].
struct SimtGemm {
  int64_t M, N, K;
  const void* A;
  int a_dtype;
  int64_t a_sm, a_sk;
  const void* B;
  int b_dtype;
  int64_t b_sk, b_sn;
  float* C;
  int64_t ldc;
  float alpha, beta;
};
cudaError_t launch_simt_gemm(const SimtGemm& g, cudaStream_t stream);

// Per-row LayerNorm statistics of U [T, d] fp32: mu, rstd (biased variance, eps).
cudaError_t launch_ln_stats(const float* U, int64_t T, int d, float eps, float* mu,
                            float* rstd, cudaStream_t stream);
// H = (U - mu) * rstd, fp32.
cudaError_t launch_ln_apply(const float* U, const float* mu, const float* rstd, int64_t T,
                            int d, float* H, cudaStream_t stream);
// dst (dtype) = src (fp32), n elements.
cudaError_t launch_cast(const float* src, void* dst, int dst_dtype, int64_t n,
                        cudaStream_t stream);

// One thread waits, with the given limit, on an mbarrier phase nothing completes (the
// timeout path of the kernels' bounded waits); l3_selftest.cu.
cudaError_t launch_wait_selftest(DevStatus* st, uint64_t limit_ns, cudaStream_t stream);

// ---- tensor-core GEMMs (l3_gemm_tc.cu), bf16 layers ------------------------------------------
// Partial LayerNorm statistics per row: tc_up_stat_tiles(d) tiles of (sum, M2).
int tc_up_stat_tiles(int d);
// fp32 scratch of the split-K form both GEMMs take when T gives too few output tiles to
// fill the GPU (0 when neither splits).
size_t tc_splitk_floats(int64_t T, int d, int d_v);
// U = bf16(A W_upᵀ) [T, d] and the partial statistics stats [tiles][T][2]; with colsum
// non-null, also colsum[n] = sum_{k < d} W_mix[n, k] (W_mix [d, 2d], 16-byte aligned).
cudaError_t launch_tc_up(const __nv_bfloat16* A, const __nv_bfloat16* W_up, int64_t T, int d,
                         int d_v, __nv_bfloat16* U, float* stats, float* slab,
                         size_t slab_floats, const __nv_bfloat16* W_mix, float* colsum,
                         DevStatus* st, cudaStream_t stream);
// y = rstd (U W_mix[:, :d]ᵀ - mu colsum) + x W_mix[:, d:]ᵀ, mu/rstd merged from stats.
cudaError_t launch_tc_mix(const __nv_bfloat16* U, const __nv_bfloat16* x,
                          const __nv_bfloat16* W_mix, int64_t T, int d, const float* stats,
                          const float* colsum, float eps, void* y, int y_dtype, float* mu_out,
                          float* rstd_out, float* slab, size_t slab_floats, DevStatus* st,
                          cudaStream_t stream);

// ---- backward (l3_backward.cu) -----------------------------------------------------------
// du = rstd * (dh - mean(dh) - h * mean(dh * h)), per row; dh has row stride ldh.
cudaError_t launch_ln_backward(const float* dh, int64_t ldh, const float* H,
                               const float* rstd, int64_t T, int d, float* du,
                               cudaStream_t stream);
struct AttendBwdArgs {
  const uint64_t* sorted_keys;
  int64_t T;
  const int32_t* offs;
  const void* K;
  const void* V;
  const void* x;
  int d, d_v, k_max;
  int dtype;
  const float* da;      // [T, d_v] batch order
  const float* dx_in;   // [T, ldx_in] direct term (dC[:, d:]), batch order
  int64_t ldx_in;
  float* dx;            // [T, d]
  float* p_buf;         // [T, k_max] sorted order
  float* ds_buf;        // [T, k_max] sorted order
};
cudaError_t launch_attend_bwd(const AttendBwdArgs& a, cudaStream_t stream);
struct SegReduceArgs {
  const uint64_t* sorted_keys;
  int64_t T;
  const int32_t* seg_start;
  const int32_t* n_seg;
  const int32_t* offs;
  const void* x;
  int dtype;
  const float* da;
  int d, d_v, k_max;
  const float* p_buf;
  const float* ds_buf;
  float* dK;
  float* dV;
};
cudaError_t launch_seg_reduce(const SegReduceArgs& a, cudaStream_t stream);

// ---- plain GEMMs of the backward on cuBLASLt (l3_blas.cu) ---------------------------------
// Column-major C[m x n] (ldc; fp32, or bf16 with c_bf16) = op(A)[m x k] op(B)[k x n]
// (+ C when accumulate), A and B bf16 (op = transpose when trans_*), fp32 accumulation.
struct LtGemm {
  int m, n, k;
  bool trans_a, trans_b;
  const void* A;
  int64_t lda;
  const void* B;
  int64_t ldb;
  void* C;
  int64_t ldc;
  bool c_bf16;
  bool accumulate;
};
constexpr size_t kLtWorkspace = size_t(32) << 20;  // cuBLASLt scratch carved from the workspace
cudaError_t lt_gemm(const LtGemm& g, void* ws, size_t ws_bytes, cudaStream_t stream);

// ---- token-stream counts (l3_count.cu) ---------------------------------------------------
// counts[t] (int64, zeroed here) = occurrences of id t in ids[0..n); ids outside [0, vocab)
// are not counted and set st->token_range.
cudaError_t launch_count_ids(const int32_t* ids, int64_t n, int64_t vocab, int64_t* counts,
                             DevStatus* st, cudaStream_t stream);

// ---- backward at batch scale with row gradients (l3_backward_rows.cu) --------------------
struct AttendBwdRowsArgs {
  const uint64_t* sorted_keys;
  int64_t T;
  const AttendGroup* groups;  // the routing plan's groups (every segment, ch-row chunks)
  const int32_t* hdr;
  const void* K;
  const void* V;
  int64_t v;
  int d, d_v, ch, k_max;
  const __nv_bfloat16* x_sorted;  // [T, d] sorted order
  const __nv_bfloat16* da16;      // [T, d_v] sorted order, bf16(da)
  const __nv_bfloat16* da16_lo;   // [T, d_v] sorted order, bf16(da - bf16(da))
  const float* ml;            // [T, 2] the forward's (max score, denominator)
  const float* delta;         // [T] a_i . da_i
  float* dx;                  // [T, d]: receives the attention term (batch order)
  float* p_buf;               // [T, k_max] by sorted position and row within the id
  float* ds_buf;              // [T, k_max]
  int n_cta;
  DevStatus* st;
};
// Rows per chunk of the backward's plan for a layer shape.
int attend_bwd_rows_per_chunk(int d, int d_v);
cudaError_t launch_attend_bwd_rows(const AttendBwdRowsArgs& a, cudaStream_t stream);
struct SegRowsArgs {
  const uint64_t* sorted_keys;
  const int32_t* seg_start;
  const int32_t* n_seg;
  const int32_t* offs;
  const int32_t* seg_row0;   // [S] first output row of each segment
  const int32_t* seg_unit0;  // [S + 1] first work unit of each segment
  const int64_t* seg_cost0;  // [S + 1] cost (k-steps) of the units before each segment
  const __nv_bfloat16* x_sorted;   // [T, d]
  const __nv_bfloat16* da_sorted;  // [T, d_v]
  const float* p_buf;
  const float* ds_buf;
  int k_max, d, d_v;
  int32_t* row_index;  // [max_rows]
  float* dK_rows;      // [max_rows, d]
  float* dV_rows;      // [max_rows, d_v]
  int64_t max_rows;
  DevStatus* st;
};
int seg_rows_col_blocks(int d, int d_v);
cudaError_t launch_seg_rows(const SegRowsArgs& a, cudaStream_t stream);
cudaError_t launch_row_plan(const uint64_t* keys, const int32_t* seg_start, const int32_t* n_seg,
                            const int32_t* offs, int d, int d_v, int32_t* seg_row0,
                            int32_t* seg_unit0, int64_t* seg_cost0, int32_t* n_rows,
                            int64_t max_rows, DevStatus* st, cudaStream_t stream);
// Row kernels of the backward: stage 0: LayerNorm of the fp32 U (h over U, h16, rstd);
// stage 1: du = LayerNorm backward of dh as bf16 hi + lo; stage 2: x and da in sorted
// order, da as bf16 hi + lo, delta = a . da; stage 3: a as bf16 hi + lo.
struct BwdSmallArgs {
  int stage;
  int64_t T;
  int d, d_v;
  float eps;
  float* U32;
  __nv_bfloat16* h16;
  float* rstd_out;
  const float* dh;
  __nv_bfloat16* du;
  __nv_bfloat16* du_lo;
  const uint64_t* keys;
  const __nv_bfloat16* x;
  const float* a;
  const float* da;
  __nv_bfloat16* x_sorted;
  __nv_bfloat16* da16;
  __nv_bfloat16* da16_lo;
  float* delta;
  __nv_bfloat16* a_hi;
  __nv_bfloat16* a_lo;
};
cudaError_t launch_bwd_small(const BwdSmallArgs& a, cudaStream_t stream);

// ---- small-batch GEMMs (l3_gemm_small.cu) --------------------------------------------------
// Batches of at most 64 tokens: u = W_up a with the LayerNorm statistics (GEMM-up), then
// y = W_mix [LayerNorm(u); x] (GEMM-mix), weight rows streamed by 32-feature CTAs.
constexpr int kSmallMaxTiles = 128;                 // d / 32 <= 128 (d <= 4096)
constexpr int kSyncWords = kSmallMaxTiles;          // arrival counters (zeroed per forward)
struct SmallGemmArgs {
  int64_t T;
  int d, d_v;
  float eps;
  const __nv_bfloat16* a;      // [T, d_v]
  const __nv_bfloat16* W_up;   // [d, d_v]
  const __nv_bfloat16* W_mix;  // [d, 2d]
  const __nv_bfloat16* x;      // [T, d]
  __nv_bfloat16* U;            // [T, d] bf16(u)
  float* tile_stats;           // [d / 32][64][2] (sum, M2) per 32-feature tile and token
  float* mu_out;               // optional (saved state)
  float* rstd_out;
  float* slab;                 // [d / 32][2][32][64] the mix halves' accumulators
  float* colsum;               // [d] row sums of W_mix[:, :d]
  uint32_t* counters;          // [d / 32], zero on entry; left at zero
  void* Y;                     // [T, d] y_dtype
  int y_dtype;
  DevStatus* st;
};
bool small_gemm_fits(int64_t T, int d, int d_v);
size_t small_gemm_floats(int d);
cudaError_t launch_small_up(const SmallGemmArgs& g, cudaStream_t stream);
cudaError_t launch_small_mix(const SmallGemmArgs& g, cudaStream_t stream);

// ---- staging of a batch's rows from host-resident tables (l3_stage.cu) ---------------------
struct StageArgs {
  const uint64_t* sorted_keys;
  const int32_t* seg_start;
  const int32_t* n_seg;
  const int32_t* offs;      // the full layer's offsets (device)
  const int32_t* seg_row0;  // [S] staged row of each segment's first row
  const int32_t* n_rows;    // [1] staged rows U
  const void* K_host;       // device-accessible address of the (pinned, mapped) host tables
  const void* V_host;
  int64_t k_row_bytes, v_row_bytes;
  void* K_st;               // [max_rows, d] staged tables (device)
  void* V_st;
  int64_t max_rows;
  int32_t* offs_st;         // [T + 1]
  int32_t* ids_st;          // [T]
  int64_t T;
  DevStatus* st;
};
cudaError_t launch_stage_rows(const StageArgs& a, cudaStream_t stream);

// ---- layer check (l3_api.cu) ---------------------------------------------------------------
cudaError_t launch_check_offsets(const int32_t* offs, int64_t vocab, int64_t v, int k_max,
                                 DevStatus* st, cudaStream_t stream);

}  // namespace l3
