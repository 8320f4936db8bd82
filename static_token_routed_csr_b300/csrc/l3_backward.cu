// Backward of the L³ layer formula ("L³: Large Lookup Layers", gist.science explainer,
// Technical Summary, "Core Architecture"; the pages name fast training but give no
// gradient formulas: these are the chain rule of the forward).
//
//   LayerNorm (no affine):  du = rstd (dh - mean(dh) - h mean(dh h))
//   Softmax aggregation:    dp_j = V_j . da,  ds_j = p_j (dp_j - sum_k p_k dp_k),
//                           dx += sum_j ds_j K_j,  dK_j += ds_j x,  dV_j += p_j da
//
// dK and dV are written by a segmented reduction: tokens are sorted by id ("Systems-
// Friendly Design", batch sorting), each table row belongs to exactly one id, and a row's
// gradient is the sum over that id's tokens in batch order. No floating-point atomics,
// so the result is bitwise reproducible.
#include <math.h>

#include "l3_internal.h"

namespace l3 {

namespace {

constexpr int kWarps = 4;

__global__ void ln_backward_kernel(const float* __restrict__ dh, int64_t ldh,
                                   const float* __restrict__ H, const float* __restrict__ rstd,
                                   int64_t T, int d, float* du) {
  const int lane = threadIdx.x & 31;
  const int64_t row = int64_t(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (row >= T) return;
  const float* g = dh + row * ldh;
  const float* h = H + row * d;
  float s1 = 0.f, s2 = 0.f;
  for (int c = lane; c < d; c += 32) {
    s1 += g[c];
    s2 = fmaf(g[c], h[c], s2);
  }
  const float mg = warp_sum(s1) / float(d), mgh = warp_sum(s2) / float(d);
  const float r = rstd[row];
  for (int c = lane; c < d; c += 32) du[row * d + c] = r * (g[c] - mg - h[c] * mgh);
}

template <typename TE, int KCH, int VCH>
__global__ void __launch_bounds__(kWarps * 32) attend_bwd_kernel(AttendBwdArgs a) {
  using E = Elem<TE>;
  constexpr int P = E::kPer16B;
  const int lane = threadIdx.x & 31;
  const int64_t q = int64_t(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  if (q >= a.T) return;
  const uint64_t key = a.sorted_keys[q];
  const int t = int(key >> 32);
  const int64_t i = int64_t(uint32_t(key));
  const int64_t r0 = a.offs[t];
  const int n = int(a.offs[t + 1] - r0);
  const TE* __restrict__ K = static_cast<const TE*>(a.K);
  const TE* __restrict__ V = static_cast<const TE*>(a.V);
  const int nck = a.d / P, ncv = a.d_v / P;
  float* pb = a.p_buf + q * a.k_max;
  float* db = a.ds_buf + q * a.k_max;

  float xr[KCH][P], dar[VCH][P];
  {
    const TE* xrow = static_cast<const TE*>(a.x) + i * a.d;
#pragma unroll
    for (int k = 0; k < KCH; ++k) {
      const int c = lane + 32 * k;
#pragma unroll
      for (int e = 0; e < P; ++e) xr[k][e] = 0.f;
      if (c < nck) E::load16(xrow + c * P, xr[k]);
    }
#pragma unroll
    for (int k = 0; k < VCH; ++k) {
      const int c = lane + 32 * k;
#pragma unroll
      for (int e = 0; e < P; ++e) dar[k][e] = (c < ncv) ? a.da[i * a.d_v + c * P + e] : 0.f;
    }
  }
  // pass 1: scores s_j and dp_j = V_j . da
  float m = -INFINITY;
  for (int j = 0; j < n; ++j) {
    const int64_t row = r0 + j;
    float s = 0.f, dp = 0.f;
#pragma unroll
    for (int k = 0; k < KCH; ++k) {
      const int c = lane + 32 * k;
      if (c < nck) {
        float kv[P];
        E::load16(K + row * a.d + c * P, kv);
#pragma unroll
        for (int e = 0; e < P; ++e) s = fmaf(kv[e], xr[k][e], s);
      }
    }
#pragma unroll
    for (int k = 0; k < VCH; ++k) {
      const int c = lane + 32 * k;
      if (c < ncv) {
        float vv[P];
        E::load16(V + row * a.d_v + c * P, vv);
#pragma unroll
        for (int e = 0; e < P; ++e) dp = fmaf(vv[e], dar[k][e], dp);
      }
    }
    s = warp_sum(s);
    dp = warp_sum(dp);
    m = fmaxf(m, s);
    if (lane == 0) {
      pb[j] = s;
      db[j] = dp;
    }
  }
  __syncwarp();
  // pass 2: p_j = e^(s_j - m) / l, delta = sum p_j dp_j, ds_j = p_j (dp_j - delta)
  float le = 0.f;
  for (int j = lane; j < n; j += 32) le += expf(pb[j] - m);
  const float l = warp_sum(le);
  float dl = 0.f;
  for (int j = lane; j < n; j += 32) dl = fmaf(expf(pb[j] - m) / l, db[j], dl);
  const float delta = warp_sum(dl);
  __syncwarp();
  for (int j = lane; j < n; j += 32) {
    const float p = expf(pb[j] - m) / l;
    const float dp = db[j];
    pb[j] = p;
    db[j] = p * (dp - delta);
  }
  __syncwarp();
  // pass 3: dx = dx_direct + sum_j ds_j K_j
  float acc[KCH][P];
#pragma unroll
  for (int k = 0; k < KCH; ++k)
#pragma unroll
    for (int e = 0; e < P; ++e) acc[k][e] = 0.f;
  for (int j = 0; j < n; ++j) {
    const float ds = db[j];
    const int64_t row = r0 + j;
#pragma unroll
    for (int k = 0; k < KCH; ++k) {
      const int c = lane + 32 * k;
      if (c < nck) {
        float kv[P];
        E::load16(K + row * a.d + c * P, kv);
#pragma unroll
        for (int e = 0; e < P; ++e) acc[k][e] = fmaf(ds, kv[e], acc[k][e]);
      }
    }
  }
#pragma unroll
  for (int k = 0; k < KCH; ++k) {
    const int c = lane + 32 * k;
    if (c < nck)
#pragma unroll
      for (int e = 0; e < P; ++e) {
        const int64_t col = c * P + e;
        a.dx[i * a.d + col] = a.dx_in[i * a.ldx_in + col] + acc[k][e];
      }
  }
}

// One CTA per segment (grid = T, CTAs past n_seg exit); warps take the segment's rows.
template <typename TE>
__global__ void __launch_bounds__(kWarps * 32) seg_reduce_kernel(SegReduceArgs a) {
  const int s = blockIdx.x;
  if (s >= *a.n_seg) return;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int q0 = a.seg_start[s], q1 = a.seg_start[s + 1];
  const int t = int(a.sorted_keys[q0] >> 32);
  const int64_t r0 = a.offs[t];
  const int n = int(a.offs[t + 1] - r0);
  const TE* __restrict__ x = static_cast<const TE*>(a.x);
  for (int j = wid; j < n; j += kWarps) {
    const int64_t row = r0 + j;
    for (int c0 = 0; c0 < a.d; c0 += 128) {
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      for (int q = q0; q < q1; ++q) {
        const int64_t i = int64_t(uint32_t(a.sorted_keys[q]));
        const float w = a.ds_buf[int64_t(q) * a.k_max + j];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int c = c0 + lane * 4 + e;
          if (c < a.d) acc[e] = fmaf(w, ld_as_float(x + i * a.d + c), acc[e]);
        }
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int c = c0 + lane * 4 + e;
        if (c < a.d) a.dK[row * a.d + c] = acc[e];
      }
    }
    for (int c0 = 0; c0 < a.d_v; c0 += 128) {
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      for (int q = q0; q < q1; ++q) {
        const int64_t i = int64_t(uint32_t(a.sorted_keys[q]));
        const float w = a.p_buf[int64_t(q) * a.k_max + j];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int c = c0 + lane * 4 + e;
          if (c < a.d_v) acc[e] = fmaf(w, a.da[i * a.d_v + c], acc[e]);
        }
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int c = c0 + lane * 4 + e;
        if (c < a.d_v) a.dV[row * a.d_v + c] = acc[e];
      }
    }
  }
}

int chunks_per_lane(int n16) {
  int c = (n16 + 31) / 32;
  int p = 1;
  while (p < c) p <<= 1;
  return p;
}

template <typename TE, int KCH>
cudaError_t bwd_v(const AttendBwdArgs& a, int vch, dim3 g, cudaStream_t s) {
  switch (vch) {
    case 1: attend_bwd_kernel<TE, KCH, 1><<<g, kWarps * 32, 0, s>>>(a); break;
    case 2: attend_bwd_kernel<TE, KCH, 2><<<g, kWarps * 32, 0, s>>>(a); break;
    case 4: attend_bwd_kernel<TE, KCH, 4><<<g, kWarps * 32, 0, s>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaSuccess;
}

template <typename TE>
cudaError_t bwd_k(const AttendBwdArgs& a, int kch, int vch, dim3 g, cudaStream_t s) {
  switch (kch) {
    case 1: return bwd_v<TE, 1>(a, vch, g, s);
    case 2: return bwd_v<TE, 2>(a, vch, g, s);
    case 4: return bwd_v<TE, 4>(a, vch, g, s);
    case 8: return bwd_v<TE, 8>(a, vch, g, s);
    case 16: return bwd_v<TE, 16>(a, vch, g, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_ln_backward(const float* dh, int64_t ldh, const float* H,
                               const float* rstd, int64_t T, int d, float* du,
                               cudaStream_t stream) {
  if (T <= 0) return cudaSuccess;
  ln_backward_kernel<<<unsigned((T + 7) / 8), 256, 0, stream>>>(dh, ldh, H, rstd, T, d, du);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_attend_bwd(const AttendBwdArgs& a, cudaStream_t stream) {
  if (a.T <= 0) return cudaSuccess;
  const int P = a.dtype == L3_BF16 ? 8 : 4;
  const int kch = chunks_per_lane(a.d / P), vch = chunks_per_lane(a.d_v / P);
  dim3 g(unsigned((a.T + kWarps - 1) / kWarps));
  cudaError_t e = a.dtype == L3_BF16 ? bwd_k<__nv_bfloat16>(a, kch, vch, g, stream)
                                     : bwd_k<float>(a, kch, vch, g, stream);
  if (e != cudaSuccess) return e;
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_seg_reduce(const SegReduceArgs& a, cudaStream_t stream) {
  if (a.T <= 0) return cudaSuccess;
  if (a.dtype == L3_BF16)
    seg_reduce_kernel<__nv_bfloat16><<<unsigned(a.T), kWarps * 32, 0, stream>>>(a);
  else
    seg_reduce_kernel<float><<<unsigned(a.T), kWarps * 32, 0, stream>>>(a);
  count_launch();
  return cudaGetLastError();
}

}  // namespace l3
