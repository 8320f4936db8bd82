// Tensor-core (tcgen05 / TMEM) GEMMs of the layer's dense contractions, bf16 operands
// with fp32 accumulation ("L³: Large Lookup Layers", gist.science explainer, Technical
// Summary, "Core Architecture": u = W_up a, then W_mix [LayerNorm(u); x]).
//
//   up:  U = A W_upᵀ          (M = T, N = d, K = d_v). The epilogue rounds U to bf16,
//        stores it, and writes per-row partial LayerNorm statistics of each 128 columns:
//        (sum, sum of squared deviations from their mean) of the rounded values.
//   mix: Y = [h; x] W_mixᵀ with h = (U - mu) rstd, never materialised. Two TMEM
//        accumulators take the two halves of the K loop: acc0 = U W_mix[:, :d]ᵀ and
//        acc1 = x W_mix[:, d:]ᵀ. LayerNorm is affine per row, so
//        y = rstd (acc0 - mu c) + acc1 with c_n = sum_k W_mix[n, k] (k < d).
//        The epilogue merges the up GEMM's partial statistics (Chan's pairwise rule) into
//        mu and rstd for its rows.
//
// One persistent CTA per SM, 10 warps: warp 0 issues TMA loads (128-byte swizzled K-major
// tiles, BK = 64) into a ring of shared-memory stages; one thread of warp 1 issues
// tcgen05.mma (M = 128, N = BN, K = 16 per instruction) into a TMEM accumulator (double-
// buffered where two fit in the 512 columns); warps 2..9 drain TMEM (tcgen05.ld) and run the
// epilogue while the next tile accumulates, two warps per 32-lane quarter, one per half of
// the columns (the split and transposed forms use warps 2..5 only). The plain forms store
// their outputs through shared memory with TMA tensor stores, and with four or more waves of
// tiles run as CTA pairs (one cta_group::2 MMA of M = 256 per pair). Every mbarrier wait is
// bounded: a wait that runs out sets a status word, the CTA drains its copies and MMAs in
// flight, frees TMEM and returns.
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "l3_internal.h"
#include "l3_tc.cuh"

namespace l3 {

namespace {

constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr int kThreads = 320;
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
  // split-K (few output tiles): unit u = tile u % tiles, K part u / tiles of `splits`; the
  // epilogue then stores raw fp32 accumulators to slab[(split * NACC + acc) * M + row][N]
  // and a finishing kernel applies the mode's epilogue to their sum
  int splits;
  float* slab;
  // optional side job of the epilogue warps before their first tile (GEMM-up): the row sums
  // cs_out[r] = sum_{c < cs_cols} cs_W[r, c] of a bf16 matrix (row stride cs_ld)
  const __nv_bfloat16* cs_W;
  int cs_rows, cs_ld, cs_cols;
  float* cs_out;
  DevStatus* st;
};

// Sum of the bf16 row `row` (ncols columns, a multiple of 8, 16-byte aligned) by one warp.
__device__ __forceinline__ float warp_row_sum(const __nv_bfloat16* row, int ncols, int lane) {
  const uint4* r4 = reinterpret_cast<const uint4*>(row);
  float s = 0.f;
#pragma unroll 4
  for (int c = lane; c < ncols / 8; c += 32) {
    const uint4 q = __ldg(r4 + c);
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
      s += __bfloat162float(__ushort_as_bfloat16(uint16_t(w[i] & 0xffffu))) +
           __bfloat162float(__ushort_as_bfloat16(uint16_t(w[i] >> 16)));
  }
  return warp_sum(s);
}

__device__ __forceinline__ float round_bf16(float v) {
  return __bfloat162float(__float2bfloat16_rn(v));
}

// Two floats rounded (to nearest even) to a bf16 pair, `a` in the low half, by one paired
// conversion (the scalar conversions run at a fraction of the paired one's rate).
__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  uint32_t r;
  memcpy(&r, &h, sizeof(r));
  return r;
}

// The two values of a bf16 pair, as floats.
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Shared staging of the swapped GEMM-up epilogue: 128 rows (features) x up to 64 columns
// (tokens), row stride 65 floats (conflict-free both ways).
constexpr int kSwapLd = 65;
constexpr int kSwapStageBytes = kBM * kSwapLd * 4;

// Longest K loop (in 64-wide blocks) whose next tile's A rows are prefetched into L2.
constexpr int kPrefetchKb = 16;

// Output box of the plain forms' TMA stores: 32 rows x 128 bytes.
constexpr int kBoxRows = 32;
constexpr int kBoxBytes = kBoxRows * 128;

// Columns of one partial LayerNorm statistic of GEMM-up: each plain-form epilogue warp
// covers one such half of a 256-column tile.
constexpr int kStatBN = 128;

// Dynamic shared memory: the stage ring, 1024 bytes of alignment slack, then either the
// barriers (256 bytes) and the transposed epilogue's staging, or the barriers padded to
// 1024 bytes and the eight epilogue warps' output boxes.
template <int BN, int STAGES, bool SPLIT, bool SWAP, bool PAIR>
constexpr int tc_smem_bytes() {
  return STAGES * (kBM + (PAIR ? BN / 2 : BN)) * kBK * 2 + 1024 +
         (SPLIT || SWAP ? 256 + (SWAP && !SPLIT ? kSwapStageBytes : 0) : 1024 + 8 * kBoxBytes);
}

// NACC * BN TMEM columns per accumulator set; two sets (the epilogue of one tile overlaps
// the next tile's MMAs) when they fit in the 512 columns, else one.
// SWAP (batches of at most 64 tokens): the weight matrix is the 128-row operand A (rows =
// output features, K contiguous, from mapA1 at every k-block) and the tokens are the N = 64
// columns, from mapB for k-blocks below kb1 and mapB2 above; the epilogue writes the
// transposed outputs.
//
// PAIR (plain forms): clusters of two CTAs share each tcgen05 MMA (M = 256: each CTA holds
// its own 128 rows of A and half of the tile's BN rows of B; each receives its 128 rows of
// the accumulator in its own TMEM). A CTA then reads a third less from L2 per output and
// its shared memory carries a third less per MMA. The even CTA issues the MMAs; both CTAs'
// TMA loads complete on its full barriers, its commits arrive on both CTAs' barriers, and
// both CTAs' epilogue warps release the accumulator on its tempty barriers.
template <int BN, int NACC, int STAGES, bool SPLIT, bool SWAP = false, bool PAIR = false>
__global__ void __launch_bounds__(kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap mapA1,
                   const __grid_constant__ CUtensorMap mapA2,
                   const __grid_constant__ CUtensorMap mapB,
                   const __grid_constant__ CUtensorMap mapB2,
                   const __grid_constant__ CUtensorMap mapY, const TcParams p) {
  static_assert(NACC * BN <= int(kTmemCols), "TMEM budget");
  // epilogue warps: eight in the plain forms (two per TMEM lane quarter, each taking half of
  // the tile's columns), four in the split and transposed forms
  constexpr int kEpiWarps = SPLIT || SWAP ? 4 : 8;
  static_assert(SPLIT || SWAP || BN % 128 == 0, "plain forms split BN into two halves");
  constexpr uint32_t NBUF = 2 * NACC * BN <= int(kTmemCols) ? 2 : 1;
  // One set of two accumulators (GEMM-mix, BN = 256): the epilogue frees acc0 (tempty[0])
  // as soon as it holds its columns in registers, and acc1 (tempty[1]) at the end; the next
  // tile's MMAs wait for each only when they first write it, so acc0's K half overlaps the
  // rest of the epilogue.
  constexpr bool kSplitFree = NACC == 2 && NBUF == 1;
  static_assert(!PAIR || (!SPLIT && !SWAP), "CTA pairs take the plain forms");
  constexpr int A_BYTES = kBM * kBK * 2;
  constexpr int B_BYTES = (PAIR ? BN / 2 : BN) * kBK * 2;
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
  const uint32_t rank = PAIR ? tc::cluster_rank() : 0u;  // CTA of the pair
  const int cta0 = PAIR ? int(blockIdx.x >> 1) : int(blockIdx.x);  // first unit
  const int ncta = PAIR ? int(gridDim.x >> 1) : int(gridDim.x);    // unit stride
  const int m_tiles = (p.M + kBM - 1) / kBM;
  const int n_tiles = (p.N + BN - 1) / BN;
  const int tiles = (PAIR ? (m_tiles + 1) / 2 : m_tiles) * n_tiles;
  const int splits = SPLIT ? p.splits : 1;
  const int units = tiles * splits;
  const int kbt = p.kb1 + p.kb2;
  // unit -> output tile and K range [k_lo, k_hi)
  auto unit_of = [&](int u, int& m_blk, int& n_blk, int& k_lo, int& k_hi) {
    const int tile = u % tiles, part = u / tiles;
    m_blk = PAIR ? (tile / n_tiles) * 2 + int(rank) : tile / n_tiles;
    n_blk = tile % n_tiles;
    k_lo = SPLIT ? int(int64_t(part) * kbt / splits) : 0;
    k_hi = SPLIT ? int(int64_t(part + 1) * kbt / splits) : kbt;
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&tfull[b], 1);
      tc::mbar_init(&tempty[b], kEpiWarps * (PAIR ? 2 : 1));
    }
    tc::mbar_init(drain, 1);
    *abort_flag = 0;
    tc::fence_barrier_init();
    tc::fence_proxy_async();
  }
  if (warp == 1) {
    if (PAIR)
      tc::tmem_alloc_pair(tmem_slot, kTmemCols);
    else
      tc::tmem_alloc(tmem_slot, kTmemCols);
  }
  tc::tc_fence_before();
  __syncthreads();
  if (PAIR) tc::cluster_sync();  // both CTAs' barriers exist before either signals the other
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  grid_dep_wait();  // the previous kernels' outputs (A or U, the statistics) are complete
  grid_dep_release();

  if (warp == 0) {
    if (lane == 0) {
      tc::tma_prefetch_desc(&mapA1);
      tc::tma_prefetch_desc(&mapA2);
      tc::tma_prefetch_desc(&mapB);
      if (SWAP) tc::tma_prefetch_desc(&mapB2);
      uint32_t it = 0;
      bool ok = true;
      for (int u = cta0; ok && u < units; u += ncta) {
        int m_blk, n_blk, k_lo, k_hi;
        unit_of(u, m_blk, n_blk, k_lo, k_hi);
        if (!SWAP && !SPLIT && kbt <= kPrefetchKb && u + ncta < units) {
          // short K loops (GEMM-up): the next tile's rows of A, which the ring reaches only
          // a few stages before its MMAs, go to L2 now
          int m2, n2, k2lo, k2hi;
          unit_of(u + ncta, m2, n2, k2lo, k2hi);
          if (m2 != m_blk)
            for (int kb = k2lo; kb < k2hi; ++kb)
              tc::tma_prefetch_l2_2d(kb < p.kb1 ? &mapA1 : &mapA2,
                                     (kb < p.kb1 ? kb : kb - p.kb1) * kBK, m2 * kBM);
        }
        for (int kb = k_lo; kb < k_hi; ++kb) {
          const uint32_t s = it % STAGES, ph = (it / STAGES) & 1;
          if (!tc::mbar_wait(&empty[s], ph ^ 1, abort_flag, p.st, 0x1)) {
            ok = false;
            break;
          }
          unsigned char* a_dst = smem + s * STAGE_BYTES;
          if constexpr (PAIR) {
            // both CTAs' halves complete on the even CTA's barrier
            if (rank == 0) tc::mbar_arrive_expect_tx(&full[s], 2 * STAGE_BYTES);
            const uint32_t fb = tc::map_to_rank(&full[s], 0);
            if (kb < p.kb1)
              tc::tma_load_2d_pair(&mapA1, fb, a_dst, kb * kBK, m_blk * kBM);
            else
              tc::tma_load_2d_pair(&mapA2, fb, a_dst, (kb - p.kb1) * kBK, m_blk * kBM);
            tc::tma_load_2d_pair(&mapB, fb, a_dst + A_BYTES, kb * kBK,
                                 n_blk * BN + int(rank) * (BN / 2));
            ++it;
            continue;
          }
          tc::mbar_arrive_expect_tx(&full[s], STAGE_BYTES);
          if (SWAP) {
            tc::tma_load_2d(&mapA1, &full[s], a_dst, kb * kBK, m_blk * kBM);
            if (kb < p.kb1)
              tc::tma_load_2d(&mapB, &full[s], a_dst + A_BYTES, kb * kBK, n_blk * BN);
            else
              tc::tma_load_2d(&mapB2, &full[s], a_dst + A_BYTES, (kb - p.kb1) * kBK, n_blk * BN);
          } else {
            if (kb < p.kb1)
              tc::tma_load_2d(&mapA1, &full[s], a_dst, kb * kBK, m_blk * kBM);
            else
              tc::tma_load_2d(&mapA2, &full[s], a_dst, (kb - p.kb1) * kBK, m_blk * kBM);
            tc::tma_load_2d(&mapB, &full[s], a_dst + A_BYTES, kb * kBK, n_blk * BN);
          }
          ++it;
        }
      }
      if (!ok) {
        // Let the copies already issued land before the CTA's shared memory goes away (the
        // odd CTA of a pair cannot watch the even CTA's barriers: it waits 200 us).
        const uint32_t first = it > uint32_t(STAGES) ? it - STAGES : 0;
        volatile int no_abort = 0;
        if (PAIR && rank != 0) {
          for (int i = 0; i < 200; ++i) __nanosleep(1000);
        } else {
          for (uint32_t j = first; j < it; ++j)
            tc::mbar_wait(&full[j % STAGES], (j / STAGES) & 1, &no_abort, p.st, 0x10,
                          100000000ull);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      constexpr uint32_t idesc = tc::idesc_bf16_f32(PAIR ? 2 * kBM : kBM, BN);
      uint32_t it = 0, lt = 0;
      bool ok = true;
      for (int u = cta0; ok && u < units; u += ncta, ++lt) {
        int m_blk, n_blk, k_lo, k_hi;
        unit_of(u, m_blk, n_blk, k_lo, k_hi);
        const uint32_t b = lt % NBUF, tph = (lt / NBUF) & 1;
        if (!kSplitFree) {
          if (!tc::mbar_wait(&tempty[b], tph ^ 1, abort_flag, p.st, 0x2)) {
            ok = false;
            break;
          }
          tc::tc_fence_after();
        }
        for (int kb = k_lo; kb < k_hi; ++kb) {
          if (kSplitFree && (kb == k_lo || kb == p.kb1)) {
            // first MMA into this accumulator of the tile: the previous tile's epilogue
            // has read it
            if (!tc::mbar_wait(&tempty[kb < p.kb1 ? 0 : 1], tph ^ 1, abort_flag, p.st, 0x2)) {
              ok = false;
              break;
            }
            tc::tc_fence_after();
          }
          const uint32_t s = it % STAGES, ph = (it / STAGES) & 1;
          if (!tc::mbar_wait(&full[s], ph, abort_flag, p.st, 0x4)) {
            ok = false;
            break;
          }
          tc::tc_fence_after();
          const int acc = (NACC == 2 && kb >= p.kb1) ? 1 : 0;
          const bool first = kb == k_lo || (NACC == 2 && kb == p.kb1);
          const uint32_t d_tmem = tmem + uint32_t((int(b) * NACC + acc) * BN);
          const uint32_t a_addr = tc::smem_u32(smem + s * STAGE_BYTES);
          const uint32_t b_addr = a_addr + A_BYTES;
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            if (PAIR)
              tc::mma_bf16_pair(d_tmem, tc::desc_kmajor_sw128(a_addr + 32 * k),
                                tc::desc_kmajor_sw128(b_addr + 32 * k), idesc,
                                (first && k == 0) ? 0u : 1u);
            else
              tc::mma_bf16(d_tmem, tc::desc_kmajor_sw128(a_addr + 32 * k),
                           tc::desc_kmajor_sw128(b_addr + 32 * k), idesc,
                           (first && k == 0) ? 0u : 1u);
          }
          if (PAIR)
            tc::mma_commit_pair(&empty[s], 0x3);
          else
            tc::mma_commit(&empty[s]);
          ++it;
        }
        if (!ok) break;
        if (PAIR)
          tc::mma_commit_pair(&tfull[b], 0x3);
        else
          tc::mma_commit(&tfull[b]);
      }
      // All MMAs issued by this thread must finish before TMEM is released.
      if (PAIR)
        tc::mma_commit_pair(drain, 0x3);
      else
        tc::mma_commit(drain);
      volatile int no_abort = 0;
      tc::mbar_wait(drain, 0, &no_abort, p.st, 0x20, 100000000ull);
    } else if (PAIR && lane == 0) {
      // the odd CTA: the even CTA's MMAs into this CTA's TMEM are done before it is freed
      volatile int no_abort = 0;
      tc::mbar_wait(drain, 0, &no_abort, p.st, 0x20, 100000000ull);
    }
  } else if (warp < 2 + kEpiWarps) {
    const int q = warp & 3;         // TMEM lane quarter this warp may access
    const int h = (warp - 2) >> 2;  // plain forms: the half of the tile's columns it takes
    const uint32_t lane_base = tmem + (uint32_t(q * 32) << 16);
    if (p.cs_W) {  // while the first accumulator fills
      for (int64_t r = int64_t(blockIdx.x) * kEpiWarps + (warp - 2); r < p.cs_rows;
           r += int64_t(gridDim.x) * kEpiWarps) {
        const float sum = warp_row_sum(p.cs_W + r * p.cs_ld, p.cs_cols, lane);
        if (lane == 0) p.cs_out[r] = sum;
      }
    }
    // Output staging of the plain forms: one box of 32 rows x 128 bytes per warp, written
    // in the 128-byte swizzle pattern (conflict-free: the 8 lanes of a store phase hit 8
    // distinct 16-byte columns) and stored by TMA from lane 0 as whole lines.
    unsigned char* box = smem + STAGES * STAGE_BYTES + 1024 + (warp - 2) * kBoxBytes;
    auto stage_box = [&]() {
      if (lane == 0) tc::bulk_wait_read<0>();  // the box's previous store has read it
      __syncwarp();
    };
    auto store_box = [&](int x, int y) {
      tc::fence_proxy_async();  // this thread's shared-memory writes, to the async proxy
      __syncwarp();
      if (lane == 0 && y < p.M) {  // a warp whose 32 rows all lie past the end stores nothing
        tc::tma_store_2d(&mapY, box, x, y);
        tc::bulk_commit();
      }
    };
    // release of an accumulator: on this CTA's tempty barrier, or on the even CTA's
    auto release = [&](int i) {
      if (lane == 0) {
        if (PAIR)
          tc::mbar_arrive_cluster(tc::map_to_rank(&tempty[i], 0));
        else
          tc::mbar_arrive(&tempty[i]);
      }
    };
    uint32_t lt = 0;
    for (int u = cta0; u < units; u += ncta, ++lt) {
      int m_blk, n_blk, k_lo, k_hi;
      unit_of(u, m_blk, n_blk, k_lo, k_hi);
      const uint32_t b = lt % NBUF, tph = (lt / NBUF) & 1;
      const int m = m_blk * kBM + q * 32 + lane;
      const bool row_ok = m < p.M;
      // GEMM-mix: merge the row's partial statistics from GEMM-up (fixed order:
      // deterministic) while the tile's MMAs still run
      float row_mean = 0.f, row_rstd = 0.f;
      if (!SPLIT && !SWAP && p.mode == 1) {
        const int mm = row_ok ? m : 0;
        float tot = 0.f;
        for (int j = 0; j < p.stat_tiles; ++j) tot += p.stats_in[(int64_t(j) * p.M + mm) * 2];
        row_mean = tot / float(p.N);
        float m2 = 0.f;
        for (int j = 0; j < p.stat_tiles; ++j) {
          const float* st = p.stats_in + (int64_t(j) * p.M + mm) * 2;
          const int cnt = p.N - j * p.stat_bn < p.stat_bn ? p.N - j * p.stat_bn : p.stat_bn;
          const float dm = st[0] / float(cnt) - row_mean;
          m2 += st[1] + float(cnt) * dm * dm;
        }
        row_rstd = 1.f / sqrtf(m2 / float(p.N) + p.eps);
      }
      if (!tc::mbar_wait(&tfull[b], tph, abort_flag, p.st, 0x8)) break;
      tc::tc_fence_after();
      const int n0 = n_blk * BN;
      const int ncols = p.N - n0 < BN ? p.N - n0 : BN;
      const uint32_t acc0 = lane_base + uint32_t(int(b) * NACC * BN);
      if (SWAP && SPLIT) {
        // split-K part, transposed problem: row m is an output feature, columns are tokens;
        // raw accumulators to slab[(part NACC + acc) N + n][M], token-major, so that the
        // lanes of a warp (consecutive features) store consecutive floats
        const int part = u / tiles;
#pragma unroll
        for (int acc = 0; acc < NACC; ++acc) {
          const bool has = NACC == 1 || (acc == 0 ? k_lo < p.kb1 : k_hi > p.kb1);
          float* dst = p.slab + (int64_t(part) * NACC + acc) * p.N * p.M + m;
          for (int c = 0; c < BN / 32; ++c) {
            if (c * 32 >= ncols) break;
            float v[32];
            if (has) {
              tc::tmem_ld32(acc0 + uint32_t(acc * BN + c * 32), v);
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] = 0.f;
            }
            if (row_ok)
#pragma unroll
              for (int j = 0; j < 32; ++j)
                if (c * 32 + j < ncols) dst[int64_t(n0 + c * 32 + j) * p.M] = v[j];
          }
        }
      } else if (SWAP) {
        // GEMM-up, transposed: row m is feature m, columns the tokens. U[token][m] = bf16,
        // then per token the (sum, squared deviations) of this tile's 128 rounded features,
        // through a shared staging tile (threads e < ncols take token e).
        float* su = reinterpret_cast<float*>(smem + STAGES * STAGE_BYTES + 256);
        const int e = q * 32 + lane;  // epilogue thread id = row of the tile
        for (int c = 0; c < BN / 32; ++c) {
          if (c * 32 >= ncols) break;
          float v[32];
          tc::tmem_ld32(acc0 + uint32_t(c * 32), v);
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float r = round_bf16(v[j]);
            su[e * kSwapLd + c * 32 + j] = row_ok ? r : 0.f;
            if (row_ok && c * 32 + j < ncols)
              p.U[int64_t(n0 + c * 32 + j) * p.M + m] = __float2bfloat16_rn(r);
          }
        }
        asm volatile("bar.sync 2, 128;" ::: "memory");
        if (e < ncols) {
          const int rows = p.M - m_blk * kBM < kBM ? p.M - m_blk * kBM : kBM;
          float sum = 0.f;
          for (int f = 0; f < rows; ++f) sum += su[f * kSwapLd + e];
          const float mean = sum / float(rows);
          float m2 = 0.f;
          for (int f = 0; f < rows; ++f) {
            const float dd = su[f * kSwapLd + e] - mean;
            m2 = fmaf(dd, dd, m2);
          }
          float* st = p.stats + (int64_t(m_blk) * p.N + n0 + e) * 2;
          st[0] = sum;
          st[1] = m2;
        }
        asm volatile("bar.sync 2, 128;" ::: "memory");
      } else if (SPLIT) {
        // split-K part: raw accumulators (zeros for an accumulator this K range missed)
        const int part = u / tiles;
#pragma unroll
        for (int acc = 0; acc < NACC; ++acc) {
          const bool has = NACC == 1 || (acc == 0 ? k_lo < p.kb1 : k_hi > p.kb1);
          float* dst = p.slab + ((int64_t(part) * NACC + acc) * p.M + m) * p.N + n0;
          for (int c = 0; c < BN / 32; ++c) {
            if (c * 32 >= ncols) break;
            float v[32];
            if (has) {
              tc::tmem_ld32(acc0 + uint32_t(acc * BN + c * 32), v);
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j) v[j] = 0.f;
            }
            if (row_ok) {
              float4* d4 = reinterpret_cast<float4*>(dst + c * 32);
#pragma unroll
              for (int j = 0; j < 8; ++j)
                d4[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
            }
          }
        }
      } else if (p.mode == 0) {
        // This warp's half of the tile row (kStatBN columns), 64 columns per TMEM load:
        // round to bf16, store, and fold each 64-column block's (mean, squared deviations)
        // into the half's running pair by the pairwise rule; the half's (sum, squared
        // deviations) are the row's statistics of that kStatBN-column tile.
        float mean = 0.f, m2 = 0.f;
        int cnt = 0;
        for (int cc = 0; cc < BN / 128; ++cc) {
          const int c = h * (BN / 128) + cc;
          if (c * 64 >= ncols) break;
          float v[64];
          tc::tmem_ld64(acc0 + c * 64, v);
          uint32_t w[32];  // the rounded values as stored; v takes them back as floats
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            w[j] = pack_bf16(v[2 * j], v[2 * j + 1]);
            v[2 * j] = bf16_lo(w[j]);
            v[2 * j + 1] = bf16_hi(w[j]);
          }
          float ps[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int j = 0; j < 64; ++j) ps[j & 3] += v[j];
          const float bmean = ((ps[0] + ps[1]) + (ps[2] + ps[3])) * (1.f / 64.f);
          float pm[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int j = 0; j < 64; ++j) pm[j & 3] = fmaf(v[j] - bmean, v[j] - bmean, pm[j & 3]);
          const float bm2 = (pm[0] + pm[1]) + (pm[2] + pm[3]);
          const float delta = bmean - mean;
          const float wb = 64.f / float(cnt + 64);
          mean = fmaf(delta, wb, mean);
          m2 += bm2 + delta * delta * float(cnt) * wb;
          cnt += 64;
          // the warp's 32 rows x 64 columns as one 128-byte swizzled box, stored by TMA
          stage_box();
#pragma unroll
          for (int j = 0; j < 8; ++j)
            *reinterpret_cast<uint4*>(box + lane * 128 + ((j ^ (lane & 7)) << 4)) =
                make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
          store_box(n0 + c * 64, m - lane);
        }
        if (row_ok && cnt > 0) {
          float* st = p.stats + (int64_t(n_blk * (BN / kStatBN) + h) * p.M + m) * 2;
          st[0] = mean * float(cnt);
          st[1] = m2;
        }
      } else {
        // row_mean and row_rstd: merged above, before the wait
        if (row_ok && n_blk == 0 && h == 0 && p.mu_out) {
          p.mu_out[m] = row_mean;
          p.rstd_out[m] = row_rstd;
        }
        // kSplitFree: this warp's half of acc0 into registers as acc0 - mu c, then acc0 is
        // released
        float a0[kSplitFree ? BN / 2 : 1];
        if constexpr (kSplitFree) {
#pragma unroll
          for (int i = 0; i < BN / 64; ++i) {
            float t[32];
            tc::tmem_ld32(acc0 + uint32_t(h * (BN / 2) + i * 32), t);
            const float* cs = p.colsum + n0 + h * (BN / 2) + i * 32;
#pragma unroll
            for (int j = 0; j < 32; ++j) a0[i * 32 + j] = t[j] - row_mean * __ldg(cs + j);
          }
          tc::tc_fence_before();
          __syncwarp();
          release(0);
        }
#pragma unroll
        for (int cc = 0; cc < BN / 64; ++cc) {
          const int c = h * (BN / 64) + cc;  // this warp's half of the columns
          if (c * 32 >= ncols) break;
          float v0[32], v1[32];
          tc::tmem_ld32(acc0 + BN + c * 32, v1);
          if constexpr (kSplitFree) {
#pragma unroll
            for (int j = 0; j < 32; ++j) v0[j] = fmaf(row_rstd, a0[cc * 32 + j], v1[j]);
          } else {
            tc::tmem_ld32(acc0 + c * 32, v0);
            const float* cs = p.colsum + n0 + c * 32;
#pragma unroll
            for (int j = 0; j < 32; ++j) v0[j] = fmaf(row_rstd, v0[j] - row_mean * __ldg(cs + j), v1[j]);
          }
          if (p.y_dtype == L3_BF16) {
            // two 32-column steps fill one 64-column box (N is a multiple of 64)
            if ((c & 1) == 0) stage_box();
#pragma unroll
            for (int j = 0; j < 4; ++j)
              *reinterpret_cast<uint4*>(box + lane * 128 +
                                        ((((c & 1) * 4 + j) ^ (lane & 7)) << 4)) =
                  make_uint4(pack_bf16(v0[8 * j], v0[8 * j + 1]),
                             pack_bf16(v0[8 * j + 2], v0[8 * j + 3]),
                             pack_bf16(v0[8 * j + 4], v0[8 * j + 5]),
                             pack_bf16(v0[8 * j + 6], v0[8 * j + 7]));
            if ((c & 1) == 1) store_box(n0 + (c - 1) * 32, m - lane);
          } else {
            stage_box();
#pragma unroll
            for (int j = 0; j < 8; ++j)
              *reinterpret_cast<float4*>(box + lane * 128 + ((j ^ (lane & 7)) << 4)) =
                  make_float4(v0[4 * j], v0[4 * j + 1], v0[4 * j + 2], v0[4 * j + 3]);
            store_box(n0 + c * 32, m - lane);
          }
        }
      }
      tc::tc_fence_before();
      __syncwarp();
      release(kSplitFree ? 1 : int(b));
    }
    if (lane == 0) tc::bulk_wait_all();  // the outputs are written before the CTA exits
  }
  tc::tc_fence_before();
  __syncthreads();
  if (PAIR) tc::cluster_sync();  // neither CTA frees TMEM or exits while the other works
  tc::tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    if (PAIR)
      tc::tmem_dealloc_pair(tmem, kTmemCols);
    else
      tc::tmem_dealloc(tmem, kTmemCols);
  }
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

int num_sms() { return device_sm_count(); }

// Row-major output matrix [rows, cols] of 2- or 4-byte elements for the epilogue's TMA
// stores: box of 32 rows x 128 bytes, 128-byte swizzle.
bool make_out_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, bool f32) {
  auto fn = encode_fn();
  if (!fn) return false;
  const int esz = f32 ? 4 : 2;
  cuuint64_t dims[2] = {cuuint64_t(cols), cuuint64_t(rows)};
  cuuint64_t strides[1] = {cuuint64_t(cols) * esz};
  cuuint32_t box[2] = {cuuint32_t(128 / esz), cuuint32_t(kBoxRows)};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
            const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// `y` is the output map of the plain forms (U for GEMM-up, Y for GEMM-mix); the split and
// transposed forms store with ordinary instructions and ignore it.
// Persistent launch of a CTA-pair kernel: one pair per two SMs that can hold a cluster of
// two (looked up once), at most one per unit; programmatic dependent launch as launch_pdl.
template <typename K, typename... Args>
cudaError_t launch_pairs(K* kern, int units, int smem, cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg{};
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = size_t(smem);
  cfg.stream = stream;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  // co-resident pairs, per kernel instantiation and device (a race only repeats the query)
  constexpr int kDevs = 64;
  static int max_pairs_of[kDevs];
  int dev = 0;
  const cudaError_t ed = cudaGetDevice(&dev);
  if (ed != cudaSuccess) return ed;
  if (dev < 0 || dev >= kDevs) return cudaErrorInvalidDevice;
  int max_pairs = __atomic_load_n(&max_pairs_of[dev], __ATOMIC_RELAXED);
  if (max_pairs == 0) {
    cfg.gridDim = dim3(2 * (num_sms() / 2));
    cfg.numAttrs = 1;
    int n = 0;
    const cudaError_t q = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
    if (q != cudaSuccess) return q;
    if (n < 1) return cudaErrorInvalidConfiguration;
    __atomic_store_n(&max_pairs_of[dev], n, __ATOMIC_RELAXED);
    max_pairs = n;
  }
  const int pairs = units < max_pairs ? units : max_pairs;
  cfg.gridDim = dim3(2 * pairs);
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

template <int BN, int NACC, int STAGES, bool SPLIT, bool SWAP = false, bool PAIR = false>
cudaError_t launch_tc(const CUtensorMap& a1, const CUtensorMap& a2, const CUtensorMap& b,
                      const CUtensorMap& b2, const CUtensorMap& y, const TcParams& p,
                      cudaStream_t stream) {
  constexpr int kSmem = tc_smem_bytes<BN, STAGES, SPLIT, SWAP, PAIR>();
  static_assert(kSmem <= 232448, "dynamic shared memory per block");
  auto kern = tc_gemm_kernel<BN, NACC, STAGES, SPLIT, SWAP, PAIR>;
  const cudaError_t attr = ensure_smem_attr(kern, kSmem);
  if (attr != cudaSuccess) return attr;
  if constexpr (PAIR) {
    const int pair_units = ((p.M + 2 * kBM - 1) / (2 * kBM)) * ((p.N + BN - 1) / BN);
    const cudaError_t e = launch_pairs(kern, pair_units, kSmem, stream, a1, a2, b, b2, y, p);
    count_launch();
    return e != cudaSuccess ? e : cudaGetLastError();
  }
  const int units = ((p.M + kBM - 1) / kBM) * ((p.N + BN - 1) / BN) * (SPLIT ? p.splits : 1);
  // a side job (row sums) is spread over every SM even when there are fewer tiles
  const int grid = units < num_sms() && !p.cs_W ? units : num_sms();
  const cudaError_t e = launch_pdl(kern, dim3(grid), dim3(kThreads), size_t(kSmem), stream, a1,
                                   a2, b, b2, y, p);
  count_launch();
  return e != cudaSuccess ? e : cudaGetLastError();
}

constexpr int kUpBN = 256, kMixBN = 256;
constexpr int kMixSplitBN = 128;  // GEMM-mix tile width when K is split (decode-sized T)

// K parts of a GEMM with too few output tiles to fill the GPU (a decode batch): enough to
// give every SM a unit, at most one per 64-wide k-block and 16 in all.
int splitk_parts(int64_t M, int N, int BN, int kbt) {
  const int64_t tiles = ((M + kBM - 1) / kBM) * ((N + BN - 1) / BN);
  if (tiles < 1 || tiles * 2 > num_sms()) return 1;
  int s = int(num_sms() / tiles);
  if (s > kbt) s = kbt;
  if (s > 16) s = 16;
  return s < 1 ? 1 : s;
}

// Split-K finish of GEMM-up: U = bf16(sum of the parts), and per 128 columns the row's
// (sum, squared deviations from their mean) of the rounded values, as the fused epilogue
// writes them. One warp per (row, 256-column tile), 8 columns per lane.
__global__ void splitk_up_finish_kernel(const float* __restrict__ slab, int parts, int M, int N,
                                        __nv_bfloat16* __restrict__ U, float* __restrict__ stats) {
  grid_dep_wait();
  grid_dep_release();
  const int lane = threadIdx.x & 31;
  const int64_t w = int64_t(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5);
  const int n_tiles = (N + kUpBN - 1) / kUpBN;
  if (w >= int64_t(M) * n_tiles) return;
  const int m = int(w / n_tiles), tile = int(w % n_tiles);
  const int n0 = tile * kUpBN, ncols = N - n0 < kUpBN ? N - n0 : kUpBN;
  const int c0 = n0 + 8 * lane;
  const bool on = 8 * lane < ncols;
  float v[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) v[j] = 0.f;
  if (on)
#pragma unroll 4
    for (int s = 0; s < parts; ++s) {
      const float4* src = reinterpret_cast<const float4*>(slab + (int64_t(s) * M + m) * N + c0);
      const float4 a = __ldcg(src), b = __ldcg(src + 1);
      v[0] += a.x; v[1] += a.y; v[2] += a.z; v[3] += a.w;
      v[4] += b.x; v[5] += b.y; v[6] += b.z; v[7] += b.w;
    }
  // statistics per kStatBN = 128 columns: lanes 0..15 and 16..31 reduce separately
  const int half = lane >> 4;
  const int hcols = ncols - half * kStatBN < kStatBN ? ncols - half * kStatBN : kStatBN;
  float sum = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    v[j] = round_bf16(v[j]);
    sum += on ? v[j] : 0.f;
  }
  for (int o = 8; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  const float mean = hcols > 0 ? sum / float(hcols) : 0.f;
  float m2 = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) m2 += on ? (v[j] - mean) * (v[j] - mean) : 0.f;
  for (int o = 8; o > 0; o >>= 1) m2 += __shfl_xor_sync(0xffffffffu, m2, o);
  if (on)
    *reinterpret_cast<uint4*>(U + int64_t(m) * N + c0) =
        make_uint4(pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]), pack_bf16(v[4], v[5]),
                   pack_bf16(v[6], v[7]));
  if ((lane & 15) == 0 && hcols > 0) {
    const int64_t j = int64_t(tile) * (kUpBN / kStatBN) + half;
    stats[(j * M + m) * 2] = sum;
    stats[(j * M + m) * 2 + 1] = m2;
  }
}

// Split-K finish of GEMM-mix: y = rstd (sum acc0 - mu colsum) + sum acc1 with the row's
// mu / rstd merged from the up GEMM's partial statistics (the fused epilogue's rule).
// One warp per (row, 256 columns), 8 columns per lane.
__global__ void splitk_mix_finish_kernel(const float* __restrict__ slab, int parts, int M, int N,
                                         const float* __restrict__ stats_in, int stat_tiles,
                                         int stat_bn, const float* __restrict__ colsum, float eps,
                                         void* Y, int y_dtype, float* mu_out, float* rstd_out) {
  grid_dep_wait();
  grid_dep_release();
  const int lane = threadIdx.x & 31;
  const int64_t w = int64_t(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5);
  const int n_chunks = (N + 255) / 256;
  if (w >= int64_t(M) * n_chunks) return;
  const int m = int(w / n_chunks), chunk = int(w % n_chunks);
  float tot = 0.f;
#pragma unroll 4
  for (int j = 0; j < stat_tiles; ++j) tot += stats_in[(int64_t(j) * M + m) * 2];
  const float mean = tot / float(N);
  float m2 = 0.f;
#pragma unroll 4
  for (int j = 0; j < stat_tiles; ++j) {
    const float* st = stats_in + (int64_t(j) * M + m) * 2;
    const int cnt = N - j * stat_bn < stat_bn ? N - j * stat_bn : stat_bn;
    const float dm = st[0] / float(cnt) - mean;
    m2 += st[1] + float(cnt) * dm * dm;
  }
  const float rstd = 1.f / sqrtf(m2 / float(N) + eps);
  if (chunk == 0 && lane == 0 && mu_out) {
    mu_out[m] = mean;
    rstd_out[m] = rstd;
  }
  const int c0 = chunk * 256 + 8 * lane;
  if (c0 >= N) return;
  float v0[8], v1[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) v0[j] = v1[j] = 0.f;
#pragma unroll 4
  for (int s = 0; s < parts; ++s) {
    const float4* a = reinterpret_cast<const float4*>(slab + ((int64_t(s) * 2) * M + m) * N + c0);
    const float4* b = reinterpret_cast<const float4*>(slab + ((int64_t(s) * 2 + 1) * M + m) * N + c0);
    const float4 a0 = __ldcg(a), a1 = __ldcg(a + 1), b0 = __ldcg(b), b1 = __ldcg(b + 1);
    v0[0] += a0.x; v0[1] += a0.y; v0[2] += a0.z; v0[3] += a0.w;
    v0[4] += a1.x; v0[5] += a1.y; v0[6] += a1.z; v0[7] += a1.w;
    v1[0] += b0.x; v1[1] += b0.y; v1[2] += b0.z; v1[3] += b0.w;
    v1[4] += b1.x; v1[5] += b1.y; v1[6] += b1.z; v1[7] += b1.w;
  }
  float y[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) y[j] = fmaf(rstd, v0[j] - mean * __ldg(colsum + c0 + j), v1[j]);
  if (y_dtype == L3_BF16) {
    *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(Y) + int64_t(m) * N + c0) =
        make_uint4(pack_bf16(y[0], y[1]), pack_bf16(y[2], y[3]), pack_bf16(y[4], y[5]),
                   pack_bf16(y[6], y[7]));
  } else {
    float4* d = reinterpret_cast<float4*>(static_cast<float*>(Y) + int64_t(m) * N + c0);
    d[0] = make_float4(y[0], y[1], y[2], y[3]);
    d[1] = make_float4(y[4], y[5], y[6], y[7]);
  }
}

// Split-K finish of the transposed GEMM-mix (batches of at most 64 tokens): slab holds
// [part][acc][token][feature]; y[token][feature] = rstd (sum acc0 - mu colsum) + sum acc1
// with the token's mu / rstd merged from the transposed GEMM-up's per-128-feature
// statistics. A CTA takes one token; each thread eight consecutive features.
constexpr int kSwapTok = 64;
__global__ void __launch_bounds__(256) splitk_mix_swap_finish_kernel(
    const float* __restrict__ slab, int parts, int M, int N, const float* __restrict__ stats_in,
    int stat_tiles, int stat_bn, const float* __restrict__ colsum, float eps, void* Y,
    int y_dtype, float* mu_out, float* rstd_out) {
  grid_dep_wait();
  grid_dep_release();
  __shared__ float s_mr[2];
  const int n = blockIdx.x, tid = threadIdx.x;
  if (tid < 32) {
    float tot = 0.f;
    for (int j = tid; j < stat_tiles; j += 32) tot += stats_in[(int64_t(j) * N + n) * 2];
    tot = warp_sum(tot);
    const float mean = tot / float(M);
    float m2 = 0.f;
    for (int j = tid; j < stat_tiles; j += 32) {
      const float* st = stats_in + (int64_t(j) * N + n) * 2;
      const int cnt = M - j * stat_bn < stat_bn ? M - j * stat_bn : stat_bn;
      const float dm = st[0] / float(cnt) - mean;
      m2 += st[1] + float(cnt) * dm * dm;
    }
    m2 = warp_sum(m2);
    if (tid == 0) {
      const float rstd = 1.f / sqrtf(m2 / float(M) + eps);
      s_mr[0] = mean;
      s_mr[1] = rstd;
      if (mu_out) {
        mu_out[n] = mean;
        rstd_out[n] = rstd;
      }
    }
  }
  __syncthreads();
  const int f = 8 * tid;
  if (f >= M) return;
  const float mean = s_mr[0], rstd = s_mr[1];
  float v0[8], v1[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) v0[j] = v1[j] = 0.f;
#pragma unroll 4
  for (int s = 0; s < parts; ++s) {
    const float4* a = reinterpret_cast<const float4*>(slab + ((int64_t(s) * 2) * N + n) * M + f);
    const float4* b =
        reinterpret_cast<const float4*>(slab + ((int64_t(s) * 2 + 1) * N + n) * M + f);
    const float4 a0 = __ldcg(a), a1 = __ldcg(a + 1), b0 = __ldcg(b), b1 = __ldcg(b + 1);
    v0[0] += a0.x; v0[1] += a0.y; v0[2] += a0.z; v0[3] += a0.w;
    v0[4] += a1.x; v0[5] += a1.y; v0[6] += a1.z; v0[7] += a1.w;
    v1[0] += b0.x; v1[1] += b0.y; v1[2] += b0.z; v1[3] += b0.w;
    v1[4] += b1.x; v1[5] += b1.y; v1[6] += b1.z; v1[7] += b1.w;
  }
  float y[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) y[j] = fmaf(rstd, v0[j] - mean * __ldg(colsum + f + j), v1[j]);
  if (y_dtype == L3_BF16) {
    *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(Y) + int64_t(n) * M + f) =
        make_uint4(pack_bf16(y[0], y[1]), pack_bf16(y[2], y[3]), pack_bf16(y[4], y[5]),
                   pack_bf16(y[6], y[7]));
  } else {
    float4* d = reinterpret_cast<float4*>(static_cast<float*>(Y) + int64_t(n) * M + f);
    d[0] = make_float4(y[0], y[1], y[2], y[3]);
    d[1] = make_float4(y[4], y[5], y[6], y[7]);
  }
}

}  // namespace

// Batches of at most this many tokens take the transposed GEMMs (weights as the 128-row
// MMA operand, the tokens as its N = 64 columns): GEMM-up needs no split, GEMM-mix splits
// K over enough parts to fill the SMs.
constexpr int64_t kSwapMaxT = kSwapTok;
constexpr int kSwapBN = kSwapTok;
int swap_mix_parts(int d) {
  const int tiles = (d + kBM - 1) / kBM;
  int s = num_sms() / tiles;
  const int kbt = 2 * d / kBK;
  if (s > kbt) s = kbt;
  if (s > 16) s = 16;
  return s < 1 ? 1 : s;
}

// GEMM-mix splits K when its wide tiles would leave most SMs idle; it then takes narrower
// tiles (more units) and at least two parts.
int mix_parts(int64_t T, int d) {
  const int kbt = 2 * d / kBK;
  if (splitk_parts(T, d, kMixBN, kbt) == 1) return 1;
  const int s = splitk_parts(T, d, kMixSplitBN, kbt);
  return s > 1 ? s : 2;
}

size_t tc_splitk_floats(int64_t T, int d, int d_v) {
  if (T <= kSwapMaxT) return size_t(swap_mix_parts(d)) * 2 * size_t(T) * size_t(d);
  const size_t up = size_t(splitk_parts(T, d, kUpBN, d_v / kBK));
  const size_t mix = size_t(mix_parts(T, d));
  const size_t a = up > 1 ? up * size_t(T) * size_t(d) : 0;
  const size_t b = mix > 1 ? 2 * mix * size_t(T) * size_t(d) : 0;
  return a > b ? a : b;
}

// Statistics tiles of GEMM-up: 256-column tiles, or 128-feature tiles in the transposed form
// (the buffer is sized for the larger count).
int tc_up_stat_tiles(int d) { return (d + kBM - 1) / kBM; }

// The plain forms run as CTA pairs when the GEMM has at least four waves of 128 x 256
// tiles (the pairs' higher MMA rate then outweighs their coarser last wave and the pair
// coupling; measured: 65536 tokens faster as pairs, 8192 tokens faster as single CTAs).
bool use_pairs(int64_t M, int N) {
  const int64_t tiles = ((M + kBM - 1) / kBM) * ((N + 255) / 256);
  return tiles >= 4 * int64_t(num_sms());
}

cudaError_t launch_tc_up(const __nv_bfloat16* A, const __nv_bfloat16* W_up, int64_t T, int d,
                         int d_v, __nv_bfloat16* U, float* stats, float* slab,
                         size_t slab_floats, const __nv_bfloat16* W_mix, float* colsum,
                         DevStatus* st, cudaStream_t stream) {
  if (T <= 0) return cudaSuccess;
  if (T <= kSwapMaxT) {
    // transposed: D[features x tokens] = W_up A^T, U[token][feature] and per-token
    // statistics of each 128-feature tile
    CUtensorMap mw, ma;
    if (!make_map(&mw, W_up, d, d_v, kBM) || !make_map(&ma, A, T, d_v, kSwapBN))
      return cudaErrorInvalidValue;
    TcParams p{};
    p.M = d;
    p.N = int(T);
    p.kb1 = d_v / kBK;
    p.kb2 = 0;
    p.mode = 0;
    p.U = U;
    p.stats = stats;
    p.st = st;
    p.splits = 1;
    if (colsum) {
      if ((reinterpret_cast<uintptr_t>(W_mix) & 15) != 0) return cudaErrorInvalidValue;
      p.cs_W = W_mix;
      p.cs_rows = d;
      p.cs_ld = 2 * d;
      p.cs_cols = d;
      p.cs_out = colsum;
    }
    return launch_tc<kSwapBN, 1, 6, false, true>(mw, mw, ma, ma, ma, p, stream);
  }
  const int splits = splitk_parts(T, d, kUpBN, d_v / kBK);
  const bool split = splits > 1 && slab && size_t(splits) * size_t(T) * size_t(d) <= slab_floats;
  const bool pairs = !split && use_pairs(T, d);
  CUtensorMap ma, mb;
  // the CTA-pair form loads half of a tile's W_up rows per CTA
  if (!make_map(&ma, A, T, d_v, kBM) || !make_map(&mb, W_up, d, d_v, pairs ? kUpBN / 2 : kUpBN))
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
  if (colsum) {
    // the mix GEMM's column sums of W_mix[:, :d], in the epilogue warps' idle start
    if ((reinterpret_cast<uintptr_t>(W_mix) & 15) != 0) return cudaErrorInvalidValue;
    p.cs_W = W_mix;
    p.cs_rows = d;
    p.cs_ld = 2 * d;
    p.cs_cols = d;
    p.cs_out = colsum;
  }
  p.splits = split ? splits : 1;  // no room for the parts: one K range per tile
  if (p.splits == 1) {
    CUtensorMap mu;
    if (!make_out_map(&mu, U, T, d, false)) return cudaErrorInvalidValue;
    if (pairs) return launch_tc<kUpBN, 1, 6, false, false, true>(ma, ma, mb, mb, mu, p, stream);
    return launch_tc<kUpBN, 1, 4, false>(ma, ma, mb, mb, mu, p, stream);
  }
  p.slab = slab;
  const cudaError_t e = launch_tc<kUpBN, 1, 4, true>(ma, ma, mb, mb, mb, p, stream);
  if (e != cudaSuccess) return e;
  const int64_t warps = T * ((d + kUpBN - 1) / kUpBN);
  const cudaError_t e2 = launch_pdl(splitk_up_finish_kernel, dim3(unsigned((warps + 7) / 8)),
                                    dim3(256), 0, stream, slab, p.splits, int(T), d, U, stats);
  count_launch();
  return e2 != cudaSuccess ? e2 : cudaGetLastError();
}

cudaError_t launch_tc_mix(const __nv_bfloat16* U, const __nv_bfloat16* x,
                          const __nv_bfloat16* W_mix, int64_t T, int d, const float* stats,
                          const float* colsum, float eps, void* y, int y_dtype, float* mu_out,
                          float* rstd_out, float* slab, size_t slab_floats, DevStatus* st,
                          cudaStream_t stream) {
  if (T <= 0) return cudaSuccess;
  if (T <= kSwapMaxT) {
    // transposed: D[features x tokens] = W_mix [U x]^T over K = 2d in parts, then the finish
    const int parts = swap_mix_parts(d);
    if (!slab || 2 * size_t(parts) * size_t(T) * size_t(d) > slab_floats)
      return cudaErrorInvalidValue;
    CUtensorMap mw, mu, mx;
    if (!make_map(&mw, W_mix, d, 2 * int64_t(d), kBM) || !make_map(&mu, U, T, d, kSwapBN) ||
        !make_map(&mx, x, T, d, kSwapBN))
      return cudaErrorInvalidValue;
    TcParams p{};
    p.M = d;
    p.N = int(T);
    p.kb1 = d / kBK;
    p.kb2 = d / kBK;
    p.mode = 1;
    p.st = st;
    p.splits = parts;
    p.slab = slab;
    cudaError_t e = launch_tc<kSwapBN, 2, 6, true, true>(mw, mw, mu, mx, mx, p, stream);
    if (e != cudaSuccess) return e;
    e = launch_pdl(splitk_mix_swap_finish_kernel, dim3(unsigned(T)), dim3(256), 0,
                   stream, slab, parts, d, int(T), stats, tc_up_stat_tiles(d), int(kBM), colsum,
                   eps, y, y_dtype, mu_out, rstd_out);
    count_launch();
    return e != cudaSuccess ? e : cudaGetLastError();
  }
  const int parts = mix_parts(T, d);
  CUtensorMap mu, mx, mw;
  const bool pairs = parts == 1 && use_pairs(T, d);
  // the CTA-pair form loads half of a tile's W_mix rows per CTA
  if (!make_map(&mu, U, T, d, kBM) || !make_map(&mx, x, T, d, kBM) ||
      !make_map(&mw, W_mix, d, 2 * int64_t(d),
                parts > 1 ? kMixSplitBN : (pairs ? kMixBN / 2 : kMixBN)))
    return cudaErrorInvalidValue;
  TcParams p{};
  p.M = int(T);
  p.N = d;
  p.kb1 = d / kBK;
  p.kb2 = d / kBK;
  p.mode = 1;
  p.stats_in = stats;
  p.stat_tiles = (d + kStatBN - 1) / kStatBN;
  p.stat_bn = kStatBN;
  p.colsum = colsum;
  p.eps = eps;
  p.Y = y;
  p.y_dtype = y_dtype;
  p.mu_out = mu_out;
  p.rstd_out = rstd_out;
  p.st = st;
  p.splits = parts;
  if (p.splits > 1 && (!slab || 2 * size_t(p.splits) * size_t(T) * size_t(d) > slab_floats))
    return cudaErrorInvalidValue;  // the workspace is sized for the parts
  if (p.splits == 1) {
    CUtensorMap my;
    if (!make_out_map(&my, y, T, d, y_dtype != L3_BF16)) return cudaErrorInvalidValue;
    if (pairs) return launch_tc<kMixBN, 2, 6, false, false, true>(mu, mx, mw, mw, my, p, stream);
    return launch_tc<kMixBN, 2, 4, false>(mu, mx, mw, mw, my, p, stream);
  }
  p.slab = slab;
  const cudaError_t e = launch_tc<kMixSplitBN, 2, 6, true>(mu, mx, mw, mw, mw, p, stream);
  if (e != cudaSuccess) return e;
  const int64_t warps = T * ((d + 255) / 256);
  const cudaError_t e2 = launch_pdl(
      splitk_mix_finish_kernel, dim3(unsigned((warps + 7) / 8)), dim3(256), 0, stream, slab,
      p.splits, int(T), d, stats, p.stat_tiles, p.stat_bn, colsum, eps, y, y_dtype, mu_out,
      rstd_out);
  count_launch();
  return e2 != cudaSuccess ? e2 : cudaGetLastError();
}

}  // namespace l3
