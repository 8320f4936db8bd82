// CUDA-core (SIMT) fp32 GEMM with arbitrary operand strides, and the row kernels of
// LayerNorm ("L³: Large Lookup Layers", gist.science explainer, Technical Summary,
// "Core Architecture": u = W_up a, then LayerNorm(u), then W_mix [h; x]).
//
// This path serves fp32 layers (whose 1e-5 relative parity rules out tensor-core tf32)
// and the small GEMMs of the backward pass. Operands may be fp32 or bf16; accumulation
// is fp32 in a fixed k order, so results are deterministic.
#include <math.h>

#include "l3_internal.h"

namespace l3 {

namespace {

constexpr int BM = 64, BN = 64, BK = 16;

template <typename TA, typename TB>
__global__ void __launch_bounds__(256) simt_gemm_kernel(SimtGemm g) {
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs[BK][BN + 4];
  const TA* __restrict__ A = static_cast<const TA*>(g.A);
  const TB* __restrict__ B = static_cast<const TB*>(g.B);
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  const int64_t m0 = int64_t(blockIdx.y) * BM, n0 = int64_t(blockIdx.x) * BN;
  float acc[4][4] = {};
  for (int64_t k0 = 0; k0 < g.K; k0 += BK) {
    // Consecutive threads follow whichever index has unit stride, so loads coalesce.
    const bool a_kfast = g.a_sk == 1, b_kfast = g.b_sk == 1;
    for (int e = threadIdx.x; e < BM * BK; e += 256) {
      const int mm = a_kfast ? e / BK : e % BM, ka = a_kfast ? e % BK : e / BM;
      const int64_t m = m0 + mm, k = k0 + ka;
      As[ka][mm] = (m < g.M && k < g.K) ? ld_as_float(A + m * g.a_sm + k * g.a_sk) : 0.f;
      const int nn = b_kfast ? e / BK : e % BN, kb = b_kfast ? e % BK : e / BN;
      const int64_t n = n0 + nn, kk2 = k0 + kb;
      Bs[kb][nn] = (n < g.N && kk2 < g.K) ? ld_as_float(B + kk2 * g.b_sk + n * g.b_sn) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float av[4], bv[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) av[r] = As[kk][ty * 4 + r];
#pragma unroll
      for (int c = 0; c < 4; ++c) bv[c] = Bs[kk][tx * 4 + c];
#pragma unroll
      for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[r][c] = fmaf(av[r], bv[c], acc[r][c]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int64_t m = m0 + ty * 4 + r;
    if (m >= g.M) continue;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int64_t n = n0 + tx * 4 + c;
      if (n >= g.N) continue;
      float* dst = g.C + m * g.ldc + n;
      const float v = g.alpha * acc[r][c];
      *dst = g.beta == 0.f ? v : v + g.beta * *dst;
    }
  }
}

__global__ void ln_stats_kernel(const float* __restrict__ U, int64_t T, int d, float eps,
                                float* mu, float* rstd) {
  const int lane = threadIdx.x & 31;
  const int64_t row = int64_t(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (row >= T) return;
  const float* u = U + row * d;
  float s = 0.f;
  for (int c = lane; c < d; c += 32) s += u[c];
  const float mean = warp_sum(s) / float(d);
  float q = 0.f;
  for (int c = lane; c < d; c += 32) {
    const float z = u[c] - mean;
    q = fmaf(z, z, q);
  }
  const float var = warp_sum(q) / float(d);
  if (lane == 0) {
    mu[row] = mean;
    rstd[row] = 1.f / sqrtf(var + eps);
  }
}

__global__ void ln_apply_kernel(const float* __restrict__ U, const float* __restrict__ mu,
                                const float* __restrict__ rstd, int64_t T, int d, float* H) {
  const int64_t n = T * d;
  for (int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; e < n;
       e += int64_t(gridDim.x) * blockDim.x) {
    const int64_t row = e / d;
    H[e] = (U[e] - mu[row]) * rstd[row];
  }
}

__global__ void cast_kernel(const float* __restrict__ src, void* dst, int dst_dtype, int64_t n) {
  for (int64_t e = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; e < n;
       e += int64_t(gridDim.x) * blockDim.x) {
    if (dst_dtype == L3_BF16)
      static_cast<__nv_bfloat16*>(dst)[e] = __float2bfloat16_rn(src[e]);
    else
      static_cast<float*>(dst)[e] = src[e];
  }
}

unsigned grid_for(int64_t n, int threads) {
  int64_t b = (n + threads - 1) / threads;
  if (b > 148 * 64) b = 148 * 64;
  return unsigned(b < 1 ? 1 : b);
}

}  // namespace

cudaError_t launch_simt_gemm(const SimtGemm& g, cudaStream_t stream) {
  if (g.M <= 0 || g.N <= 0) return cudaSuccess;
  dim3 grid(unsigned((g.N + BN - 1) / BN), unsigned((g.M + BM - 1) / BM));
  const bool a16 = g.a_dtype == L3_BF16, b16 = g.b_dtype == L3_BF16;
  if (a16 && b16)
    simt_gemm_kernel<__nv_bfloat16, __nv_bfloat16><<<grid, 256, 0, stream>>>(g);
  else if (a16)
    simt_gemm_kernel<__nv_bfloat16, float><<<grid, 256, 0, stream>>>(g);
  else if (b16)
    simt_gemm_kernel<float, __nv_bfloat16><<<grid, 256, 0, stream>>>(g);
  else
    simt_gemm_kernel<float, float><<<grid, 256, 0, stream>>>(g);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_ln_stats(const float* U, int64_t T, int d, float eps, float* mu,
                            float* rstd, cudaStream_t stream) {
  if (T <= 0) return cudaSuccess;
  ln_stats_kernel<<<unsigned((T + 7) / 8), 256, 0, stream>>>(U, T, d, eps, mu, rstd);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_ln_apply(const float* U, const float* mu, const float* rstd, int64_t T,
                            int d, float* H, cudaStream_t stream) {
  if (T <= 0) return cudaSuccess;
  ln_apply_kernel<<<grid_for(T * d, 256), 256, 0, stream>>>(U, mu, rstd, T, d, H);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_cast(const float* src, void* dst, int dst_dtype, int64_t n,
                        cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  cast_kernel<<<grid_for(n, 256), 256, 0, stream>>>(src, dst, dst_dtype, n);
  count_launch();
  return cudaGetLastError();
}

}  // namespace l3
