// Tensor-core (tcgen05 / TMEM) GEMMs of the layer's dense contractions, bf16 operands
// with fp32 accumulation ("L³: Large Lookup Layers", gist.science explainer, Technical
// Summary, "Core Architecture": u = W_up a, then W_mix [LayerNorm(u); x]).
//
//   up:  U = A W_upᵀ          (M = T, N = d, K = d_v). The epilogue rounds U to bf16,
//        stores it, and writes per-row partial LayerNorm statistics of its N tile:
//        (sum, sum of squared deviations from the tile mean) of the rounded values.
//   mix: Y = [h; x] W_mixᵀ with h = (U - mu) rstd, never materialised. Two TMEM
//        accumulators take the two halves of the K loop: acc0 = U W_mix[:, :d]ᵀ and
//        acc1 = x W_mix[:, d:]ᵀ. LayerNorm is affine per row, so
//        y = rstd (acc0 - mu c) + acc1 with c_n = sum_k W_mix[n, k] (k < d).
//        The epilogue merges the up GEMM's partial statistics (Chan's pairwise rule) into
//        mu and rstd for its rows.
//
// One persistent CTA per SM, 6 warps: warp 0 issues TMA loads (128-byte swizzled K-major
// tiles, BK = 64) into a ring of shared-memory stages; one thread of warp 1 issues
// tcgen05.mma (M = 128, N = BN, K = 16 per instruction) into a double-buffered TMEM
// accumulator; warps 2..5 drain TMEM (tcgen05.ld) and run the epilogue while the next
// tile accumulates. Every mbarrier wait is bounded: a wait that runs out sets a status
// word, the CTA drains its copies and MMAs in flight, frees TMEM and returns.
#include <cudaTypedefs.h>

#include <mutex>

#include "l3_internal.h"
#include "l3_tc.cuh"

namespace l3 {

namespace {

constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;

struct TcParams {
  int M, N;
  int kb1, kb2;  // k-blocks read from A1, then from A2 (mix only)
  int mode;      // 0 up, 1 mix
  __nv_bfloat16* U;
  float* stats;  // up: [n_tiles][M][2]
  const float* stats_in;
  int stat_tiles, stat_bn;
  const float* colsum;
  float eps;
  void* Y;
  int y_dtype;
  float* mu_out;
  float* rstd_out;
  DevStatus* st;
};

__device__ __forceinline__ float round_bf16(float v) {
  return __bfloat162float(__float2bfloat16_rn(v));
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(a));
  const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(b));
  return lo | (hi << 16);
}

template <int BN, int NACC, int STAGES>
__global__ void __launch_bounds__(kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap mapA1,
                   const __grid_constant__ CUtensorMap mapA2,
                   const __grid_constant__ CUtensorMap mapB, const TcParams p) {
  static_assert(2 * NACC * BN <= int(kTmemCols), "TMEM budget");
  constexpr int A_BYTES = kBM * kBK * 2;
  constexpr int B_BYTES = BN * kBK * 2;
  constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + STAGES * STAGE_BYTES);
  uint64_t* empty = full + STAGES;
  uint64_t* tfull = empty + STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m_tiles = (p.M + kBM - 1) / kBM;
  const int n_tiles = (p.N + BN - 1) / BN;
  const int tiles = m_tiles * n_tiles;
  const int kbt = p.kb1 + p.kb2;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&tfull[b], 1);
      tc::mbar_init(&tempty[b], 4);
    }
    tc::mbar_init(drain, 1);
    *abort_flag = 0;
    tc::fence_barrier_init();
    tc::fence_proxy_async();
  }
  if (warp == 1) tc::tmem_alloc(tmem_slot, kTmemCols);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      tc::tma_prefetch_desc(&mapA1);
      tc::tma_prefetch_desc(&mapA2);
      tc::tma_prefetch_desc(&mapB);
      uint32_t it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < tiles; tile += gridDim.x) {
        const int m_blk = tile / n_tiles, n_blk = tile % n_tiles;
        for (int kb = 0; kb < kbt; ++kb) {
          const uint32_t s = it % STAGES, ph = (it / STAGES) & 1;
          if (!tc::mbar_wait(&empty[s], ph ^ 1, abort_flag, p.st, 0x1)) {
            ok = false;
            break;
          }
          tc::mbar_arrive_expect_tx(&full[s], STAGE_BYTES);
          unsigned char* a_dst = smem + s * STAGE_BYTES;
          if (kb < p.kb1)
            tc::tma_load_2d(&mapA1, &full[s], a_dst, kb * kBK, m_blk * kBM);
          else
            tc::tma_load_2d(&mapA2, &full[s], a_dst, (kb - p.kb1) * kBK, m_blk * kBM);
          tc::tma_load_2d(&mapB, &full[s], a_dst + A_BYTES, kb * kBK, n_blk * BN);
          ++it;
        }
      }
      if (!ok) {
        // Let the copies already issued land before the CTA's shared memory goes away.
        const uint32_t first = it > uint32_t(STAGES) ? it - STAGES : 0;
        volatile int no_abort = 0;
        for (uint32_t j = first; j < it; ++j)
          tc::mbar_wait(&full[j % STAGES], (j / STAGES) & 1, &no_abort, p.st, 0x10,
                        100000000ull);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_bf16_f32(kBM, BN);
      uint32_t it = 0, lt = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < tiles; tile += gridDim.x, ++lt) {
        const uint32_t b = lt & 1, tph = (lt >> 1) & 1;
        if (!tc::mbar_wait(&tempty[b], tph ^ 1, abort_flag, p.st, 0x2)) {
          ok = false;
          break;
        }
        tc::tc_fence_after();
        for (int kb = 0; kb < kbt; ++kb) {
          const uint32_t s = it % STAGES, ph = (it / STAGES) & 1;
          if (!tc::mbar_wait(&full[s], ph, abort_flag, p.st, 0x4)) {
            ok = false;
            break;
          }
          tc::tc_fence_after();
          const int acc = (NACC == 2 && kb >= p.kb1) ? 1 : 0;
          const bool first = kb == 0 || (NACC == 2 && kb == p.kb1);
          const uint32_t d_tmem = tmem + uint32_t((int(b) * NACC + acc) * BN);
          const uint32_t a_addr = tc::smem_u32(smem + s * STAGE_BYTES);
          const uint32_t b_addr = a_addr + A_BYTES;
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)
            tc::mma_bf16(d_tmem, tc::desc_kmajor_sw128(a_addr + 32 * k),
                         tc::desc_kmajor_sw128(b_addr + 32 * k), idesc,
                         (first && k == 0) ? 0u : 1u);
          tc::mma_commit(&empty[s]);
          ++it;
        }
        if (!ok) break;
        tc::mma_commit(&tfull[b]);
      }
      // All MMAs issued by this thread must finish before TMEM is released.
      tc::mma_commit(drain);
      volatile int no_abort = 0;
      tc::mbar_wait(drain, 0, &no_abort, p.st, 0x20, 100000000ull);
    }
  } else {
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const uint32_t lane_base = tmem + (uint32_t(q * 32) << 16);
    uint32_t lt = 0;
    for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x, ++lt) {
      const int m_blk = tile / n_tiles, n_blk = tile % n_tiles;
      const uint32_t b = lt & 1, tph = (lt >> 1) & 1;
      if (!tc::mbar_wait(&tfull[b], tph, abort_flag, p.st, 0x8)) break;
      tc::tc_fence_after();
      const int m = m_blk * kBM + q * 32 + lane;
      const bool row_ok = m < p.M;
      const int n0 = n_blk * BN;
      const int ncols = p.N - n0 < BN ? p.N - n0 : BN;
      const uint32_t acc0 = lane_base + uint32_t(int(b) * NACC * BN);
      if (p.mode == 0) {
        // One pass over the tile row, 64 columns per TMEM load: round to bf16, store, and
        // fold each 64-column block's (mean, squared deviations) into the row's running
        // pair by the pairwise rule.
        float mean = 0.f, m2 = 0.f;
        int cnt = 0;
        for (int c = 0; c < BN / 64; ++c) {
          if (c * 64 >= ncols) break;
          float v[64];
          tc::tmem_ld64(acc0 + c * 64, v);
          float bs = 0.f;
#pragma unroll
          for (int j = 0; j < 64; ++j) {
            v[j] = round_bf16(v[j]);
            bs += v[j];
          }
          const float bmean = bs * (1.f / 64.f);
          float bm2 = 0.f;
#pragma unroll
          for (int j = 0; j < 64; ++j) bm2 = fmaf(v[j] - bmean, v[j] - bmean, bm2);
          const float delta = bmean - mean;
          const float wb = 64.f / float(cnt + 64);
          mean = fmaf(delta, wb, mean);
          m2 += bm2 + delta * delta * float(cnt) * wb;
          cnt += 64;
          if (row_ok) {
            uint4* dst = reinterpret_cast<uint4*>(p.U + int64_t(m) * p.N + n0 + c * 64);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              dst[j] = make_uint4(pack_bf16(v[8 * j], v[8 * j + 1]), pack_bf16(v[8 * j + 2], v[8 * j + 3]),
                                  pack_bf16(v[8 * j + 4], v[8 * j + 5]),
                                  pack_bf16(v[8 * j + 6], v[8 * j + 7]));
          }
        }
        if (row_ok) {
          float* st = p.stats + (int64_t(n_blk) * p.M + m) * 2;
          st[0] = mean * float(cnt);
          st[1] = m2;
        }
      } else {
        // Merge the partial statistics of the row (fixed order: deterministic).
        float mean = 0.f, rstd = 0.f;
        {
          const int mm = row_ok ? m : 0;
          float tot = 0.f;
          for (int j = 0; j < p.stat_tiles; ++j) tot += p.stats_in[(int64_t(j) * p.M + mm) * 2];
          mean = tot / float(p.N);
          float m2 = 0.f;
          for (int j = 0; j < p.stat_tiles; ++j) {
            const float* st = p.stats_in + (int64_t(j) * p.M + mm) * 2;
            const int cnt = p.N - j * p.stat_bn < p.stat_bn ? p.N - j * p.stat_bn : p.stat_bn;
            const float dm = st[0] / float(cnt) - mean;
            m2 += st[1] + float(cnt) * dm * dm;
          }
          rstd = 1.f / sqrtf(m2 / float(p.N) + p.eps);
        }
        if (row_ok && n_blk == 0 && p.mu_out) {
          p.mu_out[m] = mean;
          p.rstd_out[m] = rstd;
        }
        for (int c = 0; c < BN / 32; ++c) {
          if (c * 32 >= ncols) break;
          float v0[32], v1[32];
          tc::tmem_ld32(acc0 + c * 32, v0);
          tc::tmem_ld32(acc0 + BN + c * 32, v1);
          const float* cs = p.colsum + n0 + c * 32;
#pragma unroll
          for (int j = 0; j < 32; ++j) v0[j] = fmaf(rstd, v0[j] - mean * __ldg(cs + j), v1[j]);
          if (row_ok) {
            if (p.y_dtype == L3_BF16) {
              uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.Y) +
                                                    int64_t(m) * p.N + n0 + c * 32);
#pragma unroll
              for (int j = 0; j < 4; ++j)
                dst[j] = make_uint4(pack_bf16(v0[8 * j], v0[8 * j + 1]),
                                    pack_bf16(v0[8 * j + 2], v0[8 * j + 3]),
                                    pack_bf16(v0[8 * j + 4], v0[8 * j + 5]),
                                    pack_bf16(v0[8 * j + 6], v0[8 * j + 7]));
            } else {
              float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.Y) +
                                                      int64_t(m) * p.N + n0 + c * 32);
#pragma unroll
              for (int j = 0; j < 8; ++j)
                dst[j] = make_float4(v0[4 * j], v0[4 * j + 1], v0[4 * j + 2], v0[4 * j + 3]);
            }
          }
        }
      }
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&tempty[b]);
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tc::tmem_dealloc(tmem, kTmemCols);
  }
}

// sum_k W[n, k] for k < ncols of rows with stride ld (bf16), fp32.
__global__ void rowsum_kernel(const __nv_bfloat16* __restrict__ W, int64_t rows, int ld,
                              int ncols, float* out) {
  const int lane = threadIdx.x & 31;
  const int64_t r = int64_t(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (r >= rows) return;
  float s = 0.f;
  if ((reinterpret_cast<uintptr_t>(W) & 15) == 0 && ld % 8 == 0 && ncols % 8 == 0) {
    // 8 columns per 16-byte load, the row's loads all in flight together
    const uint4* row = reinterpret_cast<const uint4*>(W + r * ld);
#pragma unroll 4
    for (int c = lane; c < ncols / 8; c += 32) {
      const uint4 q = __ldg(row + c);
      const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
        s += __bfloat162float(__ushort_as_bfloat16(uint16_t(w[i] & 0xffffu))) +
             __bfloat162float(__ushort_as_bfloat16(uint16_t(w[i] >> 16)));
    }
  } else {
    for (int c = lane; c < ncols; c += 32) s += __bfloat162float(W[r * ld + c]);
  }
  s = warp_sum(s);
  if (lane == 0) out[r] = s;
}

// ---- host side ----------------------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Row-major bf16 matrix [rows, cols]; box of box_rows x 64 elements, 128-byte swizzle.
bool make_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cuuint64_t(cols), cuuint64_t(rows)};
  cuuint64_t strides[1] = {cuuint64_t(cols) * 2};
  cuuint32_t box[2] = {cuuint32_t(kBK), cuuint32_t(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int num_sms() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

template <int BN, int NACC, int STAGES>
cudaError_t launch_tc(const CUtensorMap& a1, const CUtensorMap& a2, const CUtensorMap& b,
                      const TcParams& p, cudaStream_t stream) {
  constexpr int kSmem = STAGES * (kBM + BN) * kBK * 2 + 1024 + 256;
  auto kern = tc_gemm_kernel<BN, NACC, STAGES>;
  static std::once_flag once;
  static cudaError_t attr = cudaSuccess;
  std::call_once(once, [&] {
    attr = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  });
  if (attr != cudaSuccess) return attr;
  const int tiles = ((p.M + kBM - 1) / kBM) * ((p.N + BN - 1) / BN);
  const int grid = tiles < num_sms() ? tiles : num_sms();
  kern<<<grid, kThreads, kSmem, stream>>>(a1, a2, b, p);
  count_launch();
  return cudaGetLastError();
}

constexpr int kUpBN = 256, kMixBN = 128;

}  // namespace

int tc_up_stat_tiles(int d) { return (d + kUpBN - 1) / kUpBN; }

cudaError_t launch_tc_up(const __nv_bfloat16* A, const __nv_bfloat16* W_up, int64_t T, int d,
                         int d_v, __nv_bfloat16* U, float* stats, DevStatus* st,
                         cudaStream_t stream) {
  if (T <= 0) return cudaSuccess;
  CUtensorMap ma, mb;
  if (!make_map(&ma, A, T, d_v, kBM) || !make_map(&mb, W_up, d, d_v, kUpBN))
    return cudaErrorInvalidValue;
  TcParams p{};
  p.M = int(T);
  p.N = d;
  p.kb1 = d_v / kBK;
  p.kb2 = 0;
  p.mode = 0;
  p.U = U;
  p.stats = stats;
  p.st = st;
  return launch_tc<kUpBN, 1, 4>(ma, ma, mb, p, stream);
}

cudaError_t launch_rowsum(const __nv_bfloat16* W, int64_t rows, int ld, int ncols, float* out,
                          cudaStream_t stream) {
  rowsum_kernel<<<unsigned((rows + 7) / 8), 256, 0, stream>>>(W, rows, ld, ncols, out);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_tc_mix(const __nv_bfloat16* U, const __nv_bfloat16* x,
                          const __nv_bfloat16* W_mix, int64_t T, int d, const float* stats,
                          const float* colsum, float eps, void* y, int y_dtype, float* mu_out,
                          float* rstd_out, DevStatus* st, cudaStream_t stream) {
  if (T <= 0) return cudaSuccess;
  CUtensorMap mu, mx, mw;
  if (!make_map(&mu, U, T, d, kBM) || !make_map(&mx, x, T, d, kBM) ||
      !make_map(&mw, W_mix, d, 2 * int64_t(d), kMixBN))
    return cudaErrorInvalidValue;
  TcParams p{};
  p.M = int(T);
  p.N = d;
  p.kb1 = d / kBK;
  p.kb2 = d / kBK;
  p.mode = 1;
  p.stats_in = stats;
  p.stat_tiles = tc_up_stat_tiles(d);
  p.stat_bn = kUpBN;
  p.colsum = colsum;
  p.eps = eps;
  p.Y = y;
  p.y_dtype = y_dtype;
  p.mu_out = mu_out;
  p.rstd_out = rstd_out;
  p.st = st;
  return launch_tc<kMixBN, 2, 6>(mu, mx, mw, p, stream);
}

}  // namespace l3
