// Gather-attend forward: for each token i with id t (rows R = offs[t] .. offs[t+1]-1),
//   s = K_R x_i,  p = softmax(s),  a_i = V_Rᵀ p
// ("L³: Large Lookup Layers", gist.science explainer, Technical Summary, "Core
// Architecture": context-dependent aggregation of the token's keys and values).
//
// One warp per (token, row split). The warp keeps x_i in registers (lane-interleaved
// 16-byte chunks), streams the token's K rows with 16-byte loads, reduces each dot
// product with shuffles, and runs a single-pass (online) softmax with fp32 accumulation
// of V_Rᵀ p. Tokens are visited in sorted order, so the warps of one segment of equal ids
// run together and share its rows in L2. When the batch is too small to fill the GPU
// (decode), each token's range is cut into n_split row splits whose partial
// (max, denominator, accumulator) triples a second kernel merges.
#include <math.h>

#include "l3_internal.h"

namespace l3 {

namespace {

constexpr int kWarps = 4;

template <typename TE, int KCH, int VCH>
__global__ void __launch_bounds__(kWarps * 32) attend_fwd_kernel(AttendArgs a) {
  using E = Elem<TE>;
  constexpr int P = E::kPer16B;
  constexpr int R = KCH >= 8 ? 1 : 8 / KCH;  // rows in flight per iteration
  const int lane = threadIdx.x & 31;
  const int64_t gw = int64_t(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  const int64_t q = gw / a.n_split;
  const int sp = int(gw % a.n_split);
  if (q >= a.T) return;

  const uint64_t key = a.sorted_keys[q];
  const int t = int(key >> 32);
  const int64_t i = int64_t(uint32_t(key));
  const int64_t r0 = a.offs[t], r1 = a.offs[t + 1];
  const int64_t per = (r1 - r0 + a.n_split - 1) / a.n_split;
  int64_t rs = r0 + per * sp;
  if (rs > r1) rs = r1;
  const int64_t re = rs + per < r1 ? rs + per : r1;

  const TE* __restrict__ K = static_cast<const TE*>(a.K);
  const TE* __restrict__ V = static_cast<const TE*>(a.V);
  const int nck = a.d / P, ncv = a.d_v / P;

  float xr[KCH][P];
  {
    const TE* xrow = static_cast<const TE*>(a.x) + i * a.d;
#pragma unroll
    for (int k = 0; k < KCH; ++k) {
      const int c = lane + 32 * k;
      if (c < nck) {
        E::load16(xrow + c * P, xr[k]);
      } else {
#pragma unroll
        for (int e = 0; e < P; ++e) xr[k][e] = 0.f;
      }
    }
  }

  float m = -INFINITY, l = 0.f;
  float acc[VCH][P];
#pragma unroll
  for (int k = 0; k < VCH; ++k)
#pragma unroll
    for (int e = 0; e < P; ++e) acc[k][e] = 0.f;

  for (int64_t r = rs; r < re; r += R) {
    float s[R];
#pragma unroll
    for (int u = 0; u < R; ++u) {
      s[u] = 0.f;
      const int64_t row = r + u;
      if (row < re) {
        float kv[KCH][P];
#pragma unroll
        for (int k = 0; k < KCH; ++k) {
          const int c = lane + 32 * k;
          if (c < nck) E::load16(K + row * a.d + c * P, kv[k]);
        }
#pragma unroll
        for (int k = 0; k < KCH; ++k) {
          const int c = lane + 32 * k;
          if (c < nck) {
#pragma unroll
            for (int e = 0; e < P; ++e) s[u] = fmaf(kv[k][e], xr[k][e], s[u]);
          }
        }
      }
    }
    float m_new = m;
#pragma unroll
    for (int u = 0; u < R; ++u) {
      s[u] = warp_sum(s[u]);
      if (r + u < re) m_new = fmaxf(m_new, s[u]);
    }
    const float scale = expf(m - m_new);
    l *= scale;
#pragma unroll
    for (int k = 0; k < VCH; ++k)
#pragma unroll
      for (int e = 0; e < P; ++e) acc[k][e] *= scale;
#pragma unroll
    for (int u = 0; u < R; ++u) {
      const int64_t row = r + u;
      if (row < re) {
        const float w = expf(s[u] - m_new);
        l += w;
#pragma unroll
        for (int k = 0; k < VCH; ++k) {
          const int c = lane + 32 * k;
          if (c < ncv) {
            float vv[P];
            E::load16(V + row * a.d_v + c * P, vv);
#pragma unroll
            for (int e = 0; e < P; ++e) acc[k][e] = fmaf(w, vv[e], acc[k][e]);
          }
        }
      }
    }
    m = m_new;
  }

  if (a.n_split > 1) {
    float* pp = a.part + (q * a.n_split + sp) * int64_t(a.d_v + 2);
    if (lane == 0) {
      pp[0] = m;
      pp[1] = l;
    }
#pragma unroll
    for (int k = 0; k < VCH; ++k) {
      const int c = lane + 32 * k;
      if (c < ncv)
#pragma unroll
        for (int e = 0; e < P; ++e) pp[2 + c * P + e] = acc[k][e];
    }
    return;
  }
  const float inv = 1.f / l;
#pragma unroll
  for (int k = 0; k < VCH; ++k) {
    const int c = lane + 32 * k;
    if (c < ncv) {
#pragma unroll
      for (int e = 0; e < P; ++e) {
        const float val = acc[k][e] * inv;
        if (a.a_f32) a.a_f32[i * a.d_v + c * P + e] = val;
        if (a.a_bf16) a.a_bf16[i * a.d_v + c * P + e] = __float2bfloat16_rn(val);
      }
    }
  }
  if (a.ml && lane == 0) {
    a.ml[2 * i] = m;
    a.ml[2 * i + 1] = l;
  }
}

// Merge the row splits of each token: m = max m_s, l = sum l_s e^(m_s - m),
// acc = sum acc_s e^(m_s - m), a = acc / l.
__global__ void __launch_bounds__(kWarps * 32) attend_combine_kernel(AttendArgs a) {
  const int lane = threadIdx.x & 31;
  const int64_t q = int64_t(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  if (q >= a.T) return;
  const int64_t i = int64_t(uint32_t(a.sorted_keys[q]));
  const int64_t stride = a.d_v + 2;
  const float* pp = a.part + q * a.n_split * stride;
  float m = -INFINITY;
  for (int s = 0; s < a.n_split; ++s) m = fmaxf(m, pp[s * stride]);
  float l = 0.f;
  for (int s = 0; s < a.n_split; ++s) l += pp[s * stride + 1] * expf(pp[s * stride] - m);
  const float inv = 1.f / l;
  for (int c = lane; c < a.d_v; c += 32) {
    float acc = 0.f;
    for (int s = 0; s < a.n_split; ++s) {
      const float ms = pp[s * stride];
      if (ms != -INFINITY) acc += pp[s * stride + 2 + c] * expf(ms - m);
    }
    const float val = acc * inv;
    if (a.a_f32) a.a_f32[i * a.d_v + c] = val;
    if (a.a_bf16) a.a_bf16[i * a.d_v + c] = __float2bfloat16_rn(val);
  }
  if (a.ml && lane == 0) {
    a.ml[2 * i] = m;
    a.ml[2 * i + 1] = l;
  }
}

template <typename TE, int KCH>
cudaError_t launch_v(const AttendArgs& a, int vch, dim3 grid, cudaStream_t s) {
  switch (vch) {
    case 1: attend_fwd_kernel<TE, KCH, 1><<<grid, kWarps * 32, 0, s>>>(a); break;
    case 2: attend_fwd_kernel<TE, KCH, 2><<<grid, kWarps * 32, 0, s>>>(a); break;
    case 4: attend_fwd_kernel<TE, KCH, 4><<<grid, kWarps * 32, 0, s>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaSuccess;
}

template <typename TE>
cudaError_t launch_k(const AttendArgs& a, int kch, int vch, dim3 grid, cudaStream_t s) {
  switch (kch) {
    case 1: return launch_v<TE, 1>(a, vch, grid, s);
    case 2: return launch_v<TE, 2>(a, vch, grid, s);
    case 4: return launch_v<TE, 4>(a, vch, grid, s);
    case 8: return launch_v<TE, 8>(a, vch, grid, s);
    case 16: return launch_v<TE, 16>(a, vch, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

int chunks_per_lane(int n16) {
  int c = (n16 + 31) / 32;
  int p = 1;
  while (p < c) p <<= 1;
  return p;
}

}  // namespace

int attend_choose_split(int64_t T, int k_max) {
  // Aim for about 16 warps per SM on 148 SMs; keep at least 16 rows per split.
  const int64_t want = 148 * 16;
  if (T <= 0 || T >= want) return 1;
  int64_t s = (want + T - 1) / T;
  const int64_t cap = k_max / 16 > 1 ? k_max / 16 : 1;
  if (s > cap) s = cap;
  return int(s < 1 ? 1 : s);
}

size_t attend_part_floats(int64_t T, int n_split, int d_v) {
  return n_split > 1 ? size_t(T) * size_t(n_split) * size_t(d_v + 2) : 0;
}

cudaError_t launch_attend_fwd(const AttendArgs& a, cudaStream_t stream) {
  if (a.T <= 0) return cudaSuccess;
  const int P = a.dtype == L3_BF16 ? 8 : 4;
  const int kch = chunks_per_lane(a.d / P), vch = chunks_per_lane(a.d_v / P);
  const int64_t warps = a.T * a.n_split;
  dim3 grid(unsigned((warps + kWarps - 1) / kWarps));
  cudaError_t e = a.dtype == L3_BF16 ? launch_k<__nv_bfloat16>(a, kch, vch, grid, stream)
                                     : launch_k<float>(a, kch, vch, grid, stream);
  if (e != cudaSuccess) return e;
  count_launch();
  if (a.n_split > 1) {
    attend_combine_kernel<<<unsigned((a.T + kWarps - 1) / kWarps), kWarps * 32, 0, stream>>>(a);
    count_launch();
  }
  return cudaGetLastError();
}

}  // namespace l3
