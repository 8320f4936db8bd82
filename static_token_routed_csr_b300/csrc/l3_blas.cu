// Plain matrix products of the backward pass (the weight gradients and the products with
// the weight matrices), on cuBLASLt: bf16 operands, fp32 accumulation, fp32 or bf16 results.
// These are library GEMMs with no fused epilogue; the layer's fused products (GEMM-up with
// the LayerNorm statistics, GEMM-mix with the LayerNorm and the concatenation) are this
// library's own tensor-core kernels. cuBLASLt takes its scratch from the caller's
// workspace, so the library still allocates no device memory.
#include <cublasLt.h>

#include <mutex>

#include "l3_internal.h"

namespace l3 {

namespace {

cublasLtHandle_t lt_handle() {
  static cublasLtHandle_t h = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    if (cublasLtCreate(&h) != CUBLAS_STATUS_SUCCESS) h = nullptr;
  });
  return h;
}

struct LtDescs {
  cublasLtMatmulDesc_t op = nullptr;
  cublasLtMatrixLayout_t a = nullptr, b = nullptr, c = nullptr;
  cublasLtMatmulPreference_t pref = nullptr;
  ~LtDescs() {
    if (pref) cublasLtMatmulPreferenceDestroy(pref);
    if (c) cublasLtMatrixLayoutDestroy(c);
    if (b) cublasLtMatrixLayoutDestroy(b);
    if (a) cublasLtMatrixLayoutDestroy(a);
    if (op) cublasLtMatmulDescDestroy(op);
  }
};

}  // namespace

cudaError_t lt_gemm(const LtGemm& g, void* ws, size_t ws_bytes, cudaStream_t stream) {
  cublasLtHandle_t h = lt_handle();
  if (!h) return cudaErrorNotSupported;
  if (g.m <= 0 || g.n <= 0) return cudaSuccess;
  LtDescs d;
  const cublasOperation_t ta = g.trans_a ? CUBLAS_OP_T : CUBLAS_OP_N;
  const cublasOperation_t tb = g.trans_b ? CUBLAS_OP_T : CUBLAS_OP_N;
  const cudaDataType_t ct = g.c_bf16 ? CUDA_R_16BF : CUDA_R_32F;
  bool ok = cublasLtMatmulDescCreate(&d.op, CUBLAS_COMPUTE_32F, CUDA_R_32F) == CUBLAS_STATUS_SUCCESS;
  ok = ok && cublasLtMatmulDescSetAttribute(d.op, CUBLASLT_MATMUL_DESC_TRANSA, &ta, sizeof(ta)) ==
                 CUBLAS_STATUS_SUCCESS;
  ok = ok && cublasLtMatmulDescSetAttribute(d.op, CUBLASLT_MATMUL_DESC_TRANSB, &tb, sizeof(tb)) ==
                 CUBLAS_STATUS_SUCCESS;
  // column-major layouts: A is m x k (k x m stored when transposed), B is k x n
  ok = ok && cublasLtMatrixLayoutCreate(&d.a, CUDA_R_16BF, g.trans_a ? g.k : g.m,
                                        g.trans_a ? g.m : g.k, g.lda) == CUBLAS_STATUS_SUCCESS;
  ok = ok && cublasLtMatrixLayoutCreate(&d.b, CUDA_R_16BF, g.trans_b ? g.n : g.k,
                                        g.trans_b ? g.k : g.n, g.ldb) == CUBLAS_STATUS_SUCCESS;
  ok = ok && cublasLtMatrixLayoutCreate(&d.c, ct, g.m, g.n, g.ldc) == CUBLAS_STATUS_SUCCESS;
  ok = ok && cublasLtMatmulPreferenceCreate(&d.pref) == CUBLAS_STATUS_SUCCESS;
  ok = ok && cublasLtMatmulPreferenceSetAttribute(d.pref, CUBLASLT_MATMUL_PREF_MAX_WORKSPACE_BYTES,
                                                  &ws_bytes, sizeof(ws_bytes)) ==
                 CUBLAS_STATUS_SUCCESS;
  if (!ok) return cudaErrorUnknown;
  cublasLtMatmulHeuristicResult_t res{};
  int found = 0;
  if (cublasLtMatmulAlgoGetHeuristic(h, d.op, d.a, d.b, d.c, d.c, d.pref, 1, &res, &found) !=
          CUBLAS_STATUS_SUCCESS ||
      found < 1)
    return cudaErrorUnknown;
  const float alpha = 1.f, beta = g.accumulate ? 1.f : 0.f;
  const cublasStatus_t st = cublasLtMatmul(h, d.op, &alpha, g.A, d.a, g.B, d.b, &beta, g.C, d.c,
                                           g.C, d.c, &res.algo, ws, ws_bytes, stream);
  count_launch();
  return st == CUBLAS_STATUS_SUCCESS ? cudaSuccess : cudaErrorUnknown;
}

}  // namespace l3
