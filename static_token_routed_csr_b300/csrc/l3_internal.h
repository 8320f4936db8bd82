// Internal interfaces between the C-ABI layer (l3_api.cu) and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "l3_common.cuh"

namespace l3 {

void count_launch(int n = 1);

// ---- routing (l3_route.cu) ---------------------------------------------------------------
struct RouteOut {
  int32_t* perm;       // [T]
  int32_t* seg_start;  // [T+1]
  int32_t* seg_id;     // [T]
  int32_t* n_seg;      // [1]
};
size_t route_scratch_bytes(int64_t T);
cudaError_t launch_route(const int32_t* ids, int64_t T, int64_t vocab, void* scratch,
                         RouteOut out, DevStatus* st, cudaStream_t stream,
                         const uint64_t** sorted_keys);

// ---- gather-attend (l3_attend.cu) ----------------------------------------------------------
struct AttendArgs {
  const uint64_t* sorted_keys;  // [T] (id << 32 | batch index), ascending
  int64_t T;
  const int32_t* offs;
  const void* K;
  const void* V;
  const void* x;
  int d, d_v, k_max;
  int dtype;             // L3_F32 / L3_BF16
  float* a_f32;          // [T, d_v] nullable, batch order
  __nv_bfloat16* a_bf16; // [T, d_v] nullable, batch order
  float* ml;             // [T, 2] nullable: (max score, softmax denominator)
  float* part;           // split-row partials, attend_part_floats(...) floats
  int n_split;           // row splits per token (>= 1)
};
int attend_choose_split(int64_t T, int k_max);
size_t attend_part_floats(int64_t T, int n_split, int d_v);
cudaError_t launch_attend_fwd(const AttendArgs& a, cudaStream_t stream);

// ---- gather-attend on tensor cores (l3_attend_tc.cu), bf16 prefill batches -----------------
struct AttendTcArgs {
  const uint64_t* sorted_keys;
  const int32_t* seg_start;
  const int32_t* n_seg;
  int64_t T;
  const int32_t* offs;
  const void* K;
  const void* V;
  const void* x;
  int64_t v;
  int d, d_v;
  __nv_bfloat16* x_sorted;  // [T, d] scratch
  void* items;              // attend_tc_items_bytes(T) scratch
  int32_t* n_items;         // [1] scratch
  __nv_bfloat16* a_bf16;    // [T, d_v]
  float* a_f32;             // nullable
  float* ml;                // nullable
  DevStatus* st;
};
bool attend_tc_supported(int64_t T, int d, int d_v, int dtype);
size_t attend_tc_items_bytes(int64_t T);
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

// ---- tensor-core GEMMs (l3_gemm_tc.cu), bf16 layers ------------------------------------------
// Partial LayerNorm statistics per row: tc_up_stat_tiles(d) tiles of (sum, M2).
int tc_up_stat_tiles(int d);
// U = bf16(A W_upᵀ) [T, d] and the partial statistics stats [tiles][T][2].
cudaError_t launch_tc_up(const __nv_bfloat16* A, const __nv_bfloat16* W_up, int64_t T, int d,
                         int d_v, __nv_bfloat16* U, float* stats, DevStatus* st,
                         cudaStream_t stream);
// out[r] = sum_{c < ncols} W[r, c] (row stride ld), fp32.
cudaError_t launch_rowsum(const __nv_bfloat16* W, int64_t rows, int ld, int ncols, float* out,
                          cudaStream_t stream);
// y = rstd (U W_mix[:, :d]ᵀ - mu colsum) + x W_mix[:, d:]ᵀ, mu/rstd merged from stats.
cudaError_t launch_tc_mix(const __nv_bfloat16* U, const __nv_bfloat16* x,
                          const __nv_bfloat16* W_mix, int64_t T, int d, const float* stats,
                          const float* colsum, float eps, void* y, int y_dtype, float* mu_out,
                          float* rstd_out, DevStatus* st, cudaStream_t stream);

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

// ---- layer check (l3_api.cu) ---------------------------------------------------------------
cudaError_t launch_check_offsets(const int32_t* offs, int64_t vocab, int64_t v, int k_max,
                                 DevStatus* st, cudaStream_t stream);

}  // namespace l3
