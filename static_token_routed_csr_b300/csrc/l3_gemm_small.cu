// The layer's two dense contractions for batches of at most 64 tokens, on warp-level
// tensor cores ("L³: Large Lookup Layers", gist.science explainer, Technical Summary,
// "Core Architecture": u = W_up a, h = LayerNorm(u), y = W_mix [h; x]).
//
// At this batch size the weight matrices dominate the bytes (W_up is d x d_v and W_mix is
// d x 2d, each read once) while the activations are a few hundred KB that stay in L2. So
// each CTA owns 32 output features and streams their weight rows through a ring of
// shared-memory stages (TMA, 256 columns a stage, 128-byte swizzle), with the activation
// columns of the same stage beside them; warp w multiplies the 32 rows by tokens
// 8w .. 8w + 7 (mma.sync m16n8k16, bf16 in, fp32 out).
//
//   small_up_kernel:  U = bf16(W_up aᵀ)ᵀ for the CTA's 32 features, and per token the
//     (sum, sum of squared deviations from the tile mean) of those 32 rounded values.
//   small_mix_kernel: two CTAs per 32 features, one per half of W_mix: acc0 = W1 Uᵀ (and
//     the row sums c = W1 1, taken from the staged rows) and acc1 = W2 xᵀ. The CTA of the
//     pair that finishes last merges the tiles' statistics of every token (Chan's pairwise
//     rule, fixed order) into mu and rstd and applies y = rstd (acc0 - mu c) + acc1, which
//     is W_mix [(U - mu) rstd; x] written out (LayerNorm is affine per token).
// Both kernels are programmatic dependents of the kernel before them. The arrival counters
// live in the workspace, are zeroed at the start of the forward and left at zero again by
// the CTA that counts last; merges run in a fixed order, so results do not depend on which
// CTA finishes last.
#include "l3_internal.h"
#include "l3_mma.cuh"

namespace l3 {

namespace {

using namespace wmma;

constexpr int kQThreads = 256;  // 8 warps
constexpr int kQF = 32;         // output features per CTA
constexpr int kQTok = 64;       // tokens at most
constexpr int kQKc = 256;       // columns per stage
constexpr int kQStages = 4;
constexpr int kQWBytes = kQF * kQKc * 2;    // a stage's weight rows: [4 col blocks][32][64]
constexpr int kQABytes = kQTok * kQKc * 2;  // its activation rows: [4 col blocks][64][64]
constexpr int kQStageBytes = kQWBytes + kQABytes;
constexpr int kQSmem = kQStages * kQStageBytes + 1024;  // + alignment of the ring

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

struct QSync {
  uint64_t full[kQStages];
  int abort;
};

// The K loop of both kernels over K = nch * 256 columns: each stage holds the 32 weight rows
// w_row0 .. (column blocks w_cb0 + 4 j ..) and the activation rows 0 .. 63 (column blocks
// a_cb0 + 4 j ..; rows past T arrive as zeros), both by TMA onto one mbarrier. Warp w takes
// k-steps w and w + 8 of every stage for all 32 features and all 64 tokens, so each staged
// element is read from shared memory once; acc[m][n][e] holds the warp's partial sums for
// features 16 m + g8 (+ 8 for e >= 2) and tokens 8 n + 2 t4 (+ 1 for odd e), and
// reduce_warps() adds the eight warps' parts in warp order. With want_csum, thread t also
// sums columns 32 (t % 8) .. + 31 of weight row t / 8 of every stage into the return value.
// The weights do not depend on the kernel before this one: the first stages' weight copies
// go out before `wait` (the programmatic-dependency wait when the activations come from
// that kernel), their activation copies after it. Every CTA reads the same activation rows;
// each starts at its own column block (rot) and wraps around, so that at any moment the
// CTAs ask L2 for different lines. A wait that runs out stops the loop (status code 0x800000
// in the device status) after the copies in flight have landed.
template <bool want_csum, typename Wait>
__device__ __forceinline__ float small_k_loop(const CUtensorMap* mw, int w_row0, int w_cb0,
                                              const CUtensorMap* ma, int a_cb0, int T, int nch,
                                              uint32_t ring, QSync* sy, DevStatus* st,
                                              float (&acc)[2][8][4], int rot, Wait wait) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  rot %= nch;
  auto cb = [&](int ch) { return 4 * (ch + rot < nch ? ch + rot : ch + rot - nch); };
  auto stage = [&](int ch) { return ring + uint32_t((ch % kQStages) * kQStageBytes); };
  if (tid == 0) {
    for (int s = 0; s < kQStages; ++s) tc::mbar_init(&sy->full[s], 1);
    sy->abort = 0;
    tc::fence_barrier_init();
    tc::tma_prefetch_desc(mw);
    tc::tma_prefetch_desc(ma);
  }
  __syncthreads();
  const int pre = nch < kQStages ? nch : kQStages;
  if (tid == 0)
    for (int c = 0; c < pre; ++c) {
      tc::mbar_arrive_expect_tx(&sy->full[c], uint32_t(kQStageBytes));
      tma_load_3d(mw, &sy->full[c], stage(c), 0, w_row0, w_cb0 + cb(c));
    }
  wait();
  if (tid == 0)
    for (int c = 0; c < pre; ++c)
      tma_load_3d(ma, &sy->full[c], stage(c) + uint32_t(kQWBytes), 0, 0, a_cb0 + cb(c));
  const int nt = (T + 7) / 8;  // token tiles with tokens
  volatile int* abort_flag = &sy->abort;
  float csum = 0.f;
  int ch = 0;
  for (; ch < nch; ++ch) {
    tc::mbar_wait(&sy->full[ch % kQStages], (ch / kQStages) & 1, abort_flag, st, 0x800000);
    __syncthreads();
    if (*abort_flag) break;
    const uint32_t sw = stage(ch), sa = sw + uint32_t(kQWBytes);
    if (want_csum) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 q = lds128(sw + sw128(kQF, tid >> 3, 32 * (tid & 7) + 8 * i));
        csum += ((bf_lo(q.x) + bf_hi(q.x)) + (bf_lo(q.y) + bf_hi(q.y))) +
                ((bf_lo(q.z) + bf_hi(q.z)) + (bf_lo(q.w) + bf_hi(q.w)));
      }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int ks = warp + 8 * h;
      uint32_t a[2][4];
#pragma unroll
      for (int m = 0; m < 2; ++m)
        ldsm_x4(sw + sw128(kQF, 16 * m + (lane & 15), 16 * ks + (lane >> 4) * 8), a[m][0],
                a[m][1], a[m][2], a[m][3]);
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        if (2 * p >= nt) break;
        // B of token tiles 2p, 2p + 1: lanes 0-7 tokens 16p.. at k, 8-15 the same at k + 8,
        // 16-31 tokens 16p + 8.. likewise
        uint32_t b[4];
        ldsm_x4(sa + sw128(kQTok, 16 * p + (lane & 7) + (lane >> 4) * 8, 16 * ks + ((lane >> 3) & 1) * 8),
                b[0], b[1], b[2], b[3]);
#pragma unroll
        for (int m = 0; m < 2; ++m) {
          mma16(acc[m][2 * p], a[m][0], a[m][1], a[m][2], a[m][3], b[0], b[1]);
          mma16(acc[m][2 * p + 1], a[m][0], a[m][1], a[m][2], a[m][3], b[2], b[3]);
        }
      }
    }
    __syncthreads();  // every warp is done with the stage
    if (tid == 0 && ch + kQStages < nch) {
      const int c = ch + kQStages;
      tc::mbar_arrive_expect_tx(&sy->full[ch % kQStages], uint32_t(kQStageBytes));
      tma_load_3d(mw, &sy->full[ch % kQStages], stage(c), 0, w_row0, w_cb0 + cb(c));
      tma_load_3d(ma, &sy->full[ch % kQStages], stage(c) + uint32_t(kQWBytes), 0, 0, a_cb0 + cb(c));
    }
  }
  if (ch < nch && tid == 0) {
    // stopped early: let the copies in flight land before the CTA's memory goes away
    volatile int no_abort = 0;
    const int last = nch < ch + kQStages ? nch : ch + kQStages;
    for (int c = ch; c < last; ++c)
      tc::mbar_wait(&sy->full[c % kQStages], (c / kQStages) & 1, &no_abort, st, 0x800000,
                    100000000ull);
  }
  return csum;
}

// Sum of the eight warps' partial tiles, in warp order, into D[feature][token] (row stride
// kQDld floats) in the ring's shared memory (free once the K loop is done).
constexpr int kQDld = kQTok + 4;
__device__ __forceinline__ void reduce_warps(const float (&acc)[2][8][4], float* part, float* D) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g8 = lane >> 2, t4 = lane & 3;
  float* mine = part + warp * (kQF * kQDld);
#pragma unroll
  for (int m = 0; m < 2; ++m)
#pragma unroll
    for (int n = 0; n < 8; ++n) {
      const int f = 16 * m + g8, t = 8 * n + 2 * t4;
      *reinterpret_cast<float2*>(mine + f * kQDld + t) = make_float2(acc[m][n][0], acc[m][n][1]);
      *reinterpret_cast<float2*>(mine + (f + 8) * kQDld + t) = make_float2(acc[m][n][2], acc[m][n][3]);
    }
  __syncthreads();
  for (int i = tid; i < kQF * kQTok; i += kQThreads) {
    const int f = i / kQTok, t = i % kQTok;
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) v += part[w * (kQF * kQDld) + f * kQDld + t];
    D[f * kQDld + t] = v;
  }
  __syncthreads();
}

__device__ __forceinline__ uint32_t ring_base(unsigned char* raw) {
  return (tc::smem_u32(raw) + 1023u) & ~1023u;
}

// One CTA per 32 features f0 = 32 blockIdx.x .. of u = W_up a.
__global__ void __launch_bounds__(kQThreads, 1)
    small_up_kernel(const __grid_constant__ CUtensorMap mw, const __grid_constant__ CUtensorMap ma,
                    const SmallGemmArgs g) {
  extern __shared__ __align__(1024) unsigned char q_smem[];
  __shared__ QSync sy;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g8 = lane >> 2, t4 = lane & 3;
  const int T = int(g.T), d = g.d, tile = blockIdx.x, f0 = kQF * tile;
  float acc[2][8][4] = {};
  small_k_loop<false>(&mw, f0, 0, &ma, 0, T, g.d_v / kQKc, ring_base(q_smem), &sy, g.st, acc,
                      tile, [] {
                        grid_dep_wait();  // a is complete
                        grid_dep_release();
                      });
  float* part = reinterpret_cast<float*>(q_smem + (ring_base(q_smem) - tc::smem_u32(q_smem)));
  float* D = part + 8 * kQF * kQDld;
  reduce_warps(acc, part, D);
  // U (rounded to bf16) and this tile's statistics: token tid / 4, features 8 (tid % 4) ..
  const int tok = tid >> 2, c = tid & 3;
  float r[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) r[j] = __bfloat162float(__float2bfloat16_rn(D[(8 * c + j) * kQDld + tok]));
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) s += r[j];
  s += __shfl_xor_sync(0xffffffffu, s, 1);
  s += __shfl_xor_sync(0xffffffffu, s, 2);
  const float mt = s * (1.f / float(kQF));
  float q = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) q = fmaf(r[j] - mt, r[j] - mt, q);
  q += __shfl_xor_sync(0xffffffffu, q, 1);
  q += __shfl_xor_sync(0xffffffffu, q, 2);
  if (tok < T) {
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) w[j] = pack_bf16(r[2 * j], r[2 * j + 1]);
    *reinterpret_cast<uint4*>(g.U + int64_t(tok) * d + f0 + 8 * c) = make_uint4(w[0], w[1], w[2], w[3]);
    if (c == 0)
      *reinterpret_cast<float2*>(g.tile_stats + (int64_t(tile) * kQTok + tok) * 2) = make_float2(s, q);
  }
  (void)warp;
  (void)g8;
  (void)t4;
}

// CTA pair (2 fb, 2 fb + 1) for features f0 = 32 fb ..: half 0 takes W_mix[:, :d] with U
// (and its row sums), half 1 W_mix[:, d:] with x; the pair's last CTA writes y.
__global__ void __launch_bounds__(kQThreads, 1)
    small_mix_kernel(const __grid_constant__ CUtensorMap mw, const __grid_constant__ CUtensorMap mu,
                     const __grid_constant__ CUtensorMap mx, const SmallGemmArgs g) {
  extern __shared__ __align__(1024) unsigned char q_smem[];
  __shared__ QSync sy;
  __shared__ int s_last;
  __shared__ float s_cs[kQF];
  __shared__ float s_mu[kQTok], s_rstd[kQTok];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g8 = lane >> 2, t4 = lane & 3;
  const int T = int(g.T), d = g.d, fb = blockIdx.x >> 1, half = blockIdx.x & 1;
  const int f0 = kQF * fb;
  float acc[2][8][4] = {};
  if (half == 0) {
    // U comes from GEMM-up: its rows are requested after the dependency wait
    float cs = small_k_loop<true>(&mw, f0, 0, &mu, 0, T, d / kQKc, ring_base(q_smem), &sy, g.st,
                                  acc, fb, [] {
                                    grid_dep_wait();
                                    grid_dep_release();
                                  });
    cs += __shfl_xor_sync(0xffffffffu, cs, 1);
    cs += __shfl_xor_sync(0xffffffffu, cs, 2);
    cs += __shfl_xor_sync(0xffffffffu, cs, 4);
    if ((tid & 7) == 0) s_cs[tid >> 3] = cs;
  } else {
    // x is an input of the layer: this half runs beside GEMM-up, without waiting for it
    grid_dep_release();
    small_k_loop<false>(&mw, f0, d / 64, &mx, 0, T, d / kQKc, ring_base(q_smem), &sy, g.st, acc,
                        fb, [] {});
  }
  // this half's sums (and row sums) to the pair's slab: [half][feature][token]
  float* part = reinterpret_cast<float*>(q_smem + (ring_base(q_smem) - tc::smem_u32(q_smem)));
  float* D = part + 8 * kQF * kQDld;
  reduce_warps(acc, part, D);
  float* sl = g.slab + (int64_t(fb) * 2 + half) * (kQF * kQTok);
  for (int i = tid; i < kQF * kQTok; i += kQThreads) sl[i] = D[(i / kQTok) * kQDld + i % kQTok];
  (void)warp;
  (void)g8;
  (void)t4;
  if (half == 0 && tid < kQF) g.colsum[f0 + tid] = s_cs[tid];
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(&g.counters[fb], 1u) == 1u ? 1 : 0;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  grid_dep_wait();  // (GEMM-up's statistics: complete once the other half arrived; a no-op wait)
  const int tok = tid >> 2, c = tid & 3;
  {
    // mu and rstd of token tid / 4 from GEMM-up's tile statistics: thread part c takes
    // tiles c, c + 4, ... (all loads at once), then sums across the 4 threads in a fixed
    // order (Chan's rule: M2 = sum_j M2_j + 32 (mean_j - mean)^2)
    const int nt = d / kQF;
    float2 v[kSmallMaxTiles / 4];
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < kSmallMaxTiles / 4; ++i) {
      const int j = c + 4 * i;
      v[i] = j < nt ? __ldcg(reinterpret_cast<const float2*>(g.tile_stats) + int64_t(j) * kQTok + tok)
                    : make_float2(0.f, 0.f);
      s += v[i].x;
    }
    s += __shfl_xor_sync(0xffffffffu, s, 1);
    s += __shfl_xor_sync(0xffffffffu, s, 2);
    const float mean = s / float(d);
    float m2 = 0.f;
#pragma unroll
    for (int i = 0; i < kSmallMaxTiles / 4; ++i) {
      const float dm = v[i].x * (1.f / float(kQF)) - mean;
      if (c + 4 * i < nt) m2 += v[i].y + float(kQF) * dm * dm;
    }
    m2 += __shfl_xor_sync(0xffffffffu, m2, 1);
    m2 += __shfl_xor_sync(0xffffffffu, m2, 2);
    const float rstd = 1.f / sqrtf(m2 / float(d) + g.eps);
    if (c == 0) {
      s_mu[tok] = mean;
      s_rstd[tok] = rstd;
      if (fb == 0 && g.mu_out && tok < T) {
        g.mu_out[tok] = mean;
        g.rstd_out[tok] = rstd;
      }
    }
  }
  __syncthreads();
  // y[token][f0 + 8 c .. + 8] for token tid / 4, c = tid % 4
  if (tok < T) {
    const float mean = s_mu[tok], rstd = s_rstd[tok];
    const float* s0 = g.slab + (int64_t(fb) * 2) * (kQF * kQTok);
    const float* s1 = s0 + kQF * kQTok;
    float y[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int f = 8 * c + j;
      y[j] = fmaf(rstd, __ldcg(s0 + f * kQTok + tok) - mean * __ldcg(g.colsum + f0 + f),
                  __ldcg(s1 + f * kQTok + tok));
    }
    if (g.y_dtype == L3_BF16) {
      uint32_t w[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) w[j] = pack_bf16(y[2 * j], y[2 * j + 1]);
      *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(g.Y) + int64_t(tok) * d + f0 + 8 * c) =
          make_uint4(w[0], w[1], w[2], w[3]);
    } else {
      float4* o = reinterpret_cast<float4*>(static_cast<float*>(g.Y) + int64_t(tok) * d + f0 + 8 * c);
      o[0] = make_float4(y[0], y[1], y[2], y[3]);
      o[1] = make_float4(y[4], y[5], y[6], y[7]);
    }
  }
  if (tid == 0) g.counters[fb] = 0u;
}

}  // namespace

bool small_gemm_fits(int64_t T, int d, int d_v) {
  return T >= 1 && T <= kQTok && d % kQKc == 0 && d_v % kQKc == 0 && d / kQF <= kSmallMaxTiles;
}

size_t small_gemm_floats(int d) {
  return size_t(d / kQF) * kQTok * 2 + size_t(d) * kQTok * 2 + size_t(d);
}

cudaError_t launch_small_up(const SmallGemmArgs& g, cudaStream_t stream) {
  if (!small_gemm_fits(g.T, g.d, g.d_v)) return cudaErrorInvalidValue;
  CUtensorMap mw, ma;
  if (!make_row_block_map(&mw, g.W_up, g.d, g.d_v, kQF, kQKc / 64) ||
      !make_row_block_map(&ma, g.a, g.T, g.d_v, kQTok, kQKc / 64))
    return cudaErrorInvalidValue;
  const cudaError_t a = ensure_smem_attr(small_up_kernel, kQSmem);
  if (a != cudaSuccess) return a;
  const cudaError_t e = launch_pdl(small_up_kernel, dim3(unsigned(g.d / kQF)), dim3(kQThreads),
                                   size_t(kQSmem), stream, mw, ma, g);
  count_launch();
  return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_small_mix(const SmallGemmArgs& g, cudaStream_t stream) {
  if (!small_gemm_fits(g.T, g.d, g.d_v)) return cudaErrorInvalidValue;
  CUtensorMap mw, mu, mx;
  if (!make_row_block_map(&mw, g.W_mix, g.d, 2 * int64_t(g.d), kQF, kQKc / 64) ||
      !make_row_block_map(&mu, g.U, g.T, g.d, kQTok, kQKc / 64) ||
      !make_row_block_map(&mx, g.x, g.T, g.d, kQTok, kQKc / 64))
    return cudaErrorInvalidValue;
  const cudaError_t a = ensure_smem_attr(small_mix_kernel, kQSmem);
  if (a != cudaSuccess) return a;
  const cudaError_t e = launch_pdl(small_mix_kernel, dim3(unsigned(2 * (g.d / kQF))),
                                   dim3(kQThreads), size_t(kQSmem), stream, mw, mu, mx, g);
  count_launch();
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace l3
