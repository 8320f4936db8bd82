// Gather-attend forward on tcgen05 tensor cores for the long segments of equal token ids
// ("L³: Large Lookup Layers", gist.science explainer, Technical Summary: "Core
// Architecture" for the aggregation a = V_tᵀ softmax(K_t x); "Systems-Friendly Design",
// batch sorting, for grouping the tokens of one id so that its rows are read once).
//
// A work item is one id t with up to 64 of its tokens (longer segments are cut into
// 64-token chunks). With n = n_t rows and the item's tokens X (sorted order, N = 16..64
// columns):
//   phase 1   Sᵀ = K_t Xᵀ           M = 128 table rows per chunk (TMEM lanes), N tokens,
//                                    K = d in 64-wide blocks; up to 4 row chunks.
//   softmax   per token: m = max_rows s, e = exp(s - m) (rows >= n give 0), l = sum e;
//             Pᵀ = bf16(e) is written to shared memory as the phase-2 B operand.
//   phase 2   Aᵀ = V_tᵀ Pᵀ           M = 128 value columns per chunk, N tokens, K = rows
//                                    in 16-row steps (both operands MN-major).
//   epilogue  a = Aᵀ / l, scattered to batch order (bf16 for the GEMM, fp32 if asked).
// K_t rows arrive by TMA in 128-row boxes and V_t rows in 64-row boxes (rows past an item's
// range are read and masked): few large copies per stage, since each TMA instruction costs
// tens of nanoseconds to issue. The item's x rows come straight from x, 64 columns of four
// tokens per 4-row TMA gather (the producer warp looks up the tokens' batch indices).
// Phase 1 walks the 64-wide K blocks outermost: an x block is copied once into its own
// small ring and serves all row chunks of the item (released after the last chunk's MMAs),
// so the K ring holds only K boxes and more bytes are in flight.
// One persistent CTA per SM, 11 warps: the K / V producer, the MMA issuer, 8 softmax/epilogue
// warps (two per TMEM lane quarter, each taking 32 of the item's 64 token columns) and the
// x producer, whose 4-row gathers (16 per x box) would otherwise delay the K stream. All waits
// are bounded; the softmax warps synchronise on an mbarrier (bounded) rather than a named
// barrier, so no thread can be left waiting.
#include <cstring>
#include <cudaTypedefs.h>

#include <mutex>

#include "l3_internal.h"
#include "l3_tc.cuh"

namespace l3 {

namespace {

constexpr int kThreads = 352;
constexpr int kSoftWarps = 8;  // warps 2 .. 9
constexpr int kNT = 64;            // tokens per item
constexpr int kStages = 8;         // K / V ring (16 KB stages)
constexpr int kXSlots = 2;         // x boxes (8 KB), one per K block in flight
constexpr int kKTile = 128 * 128;  // 128 rows x 64 bf16
constexpr int kXTile = kNT * 128;  // 64 tokens x 64 bf16
constexpr int kStageBytes = kKTile;
constexpr int kPBytes = 512 * 128;  // Pᵀ: up to 512 rows x 64 tokens bf16
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kSCol = 0;    // Sᵀ chunk rc at columns 64 rc
constexpr uint32_t kACol = 256;  // Aᵀ chunk dc at columns 256 + 64 dc
constexpr int kSmemBytes =
    kStages * kStageBytes + kXSlots * kXTile + kPBytes + 8 * kNT * 4 + 256 + 1024;

static_assert(kNT == kTcNT, "item size of the plan");
using Item = AttendItem;

struct TcAttendParams {
  const Item* items;
  const int32_t* n_items;
  const uint64_t* sorted_keys;
  const int32_t* offs;
  int d, d_v;
  __nv_bfloat16* a_bf16;  // [T, d_v] batch order
  float* a_f32;           // nullable
  float* ml;              // nullable [T, 2]
  DevStatus* st;
};

// MN-major operand in the 128-byte swizzle: 64 elements (128 B) contiguous along M/N, K
// rows 128 B apart in 8-row groups of 1024 B; further 64-element M/N blocks lbo bytes on.
__device__ __forceinline__ uint64_t desc_mnmajor_sw128(uint32_t addr, uint32_t lbo_bytes) {
  uint64_t d = 0;
  d |= uint64_t((addr >> 4) & 0x3FFFu);
  d |= uint64_t((lbo_bytes >> 4) & 0x3FFFu) << 16;  // stride between 64-element MN blocks
  d |= uint64_t(1024 >> 4) << 32;                   // stride between 8-row K groups
  d |= uint64_t(1) << 46;
  d |= uint64_t(2) << 61;
  return d;
}

__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int a_mn, int b_mn) {
  return tc::idesc_bf16_f32(M, N) | (uint32_t(a_mn) << 15) | (uint32_t(b_mn) << 16);
}

// Wait that ends only when the phase completes or this thread's own time limit runs out
// (then it raises the CTA's abort flag): used where all 128 softmax threads must take
// the same path, so no thread leaves a phase the others complete.
__device__ __forceinline__ bool wait_own(uint64_t* bar, uint32_t parity, volatile int* abort,
                                         DevStatus* st, int code) {
  volatile int never = 0;
  if (tc::mbar_wait(bar, parity, &never, st, code)) return true;
  *abort = 1;
  return false;
}

// Barrier of the softmax warps on an mbarrier (one arrival per warp), bounded.
__device__ __forceinline__ bool group_sync(uint64_t* bar, uint32_t& phase, volatile int* abort,
                                           DevStatus* st) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) tc::mbar_arrive(bar);
  const bool ok = wait_own(bar, phase, abort, st, 0x4000);
  phase ^= 1;
  return ok;
}

// Butterfly reduce-scatter over 32 lanes of a 32-vector: afterwards v[0] holds the
// reduction for entry `lane`.
template <bool kMax>
__device__ __forceinline__ void reduce_scatter32(float (&v)[32], int lane) {
#pragma unroll
  for (int step = 0; step < 5; ++step) {
    const int o = 16 >> step;
    const int half = 16 >> step;
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float lo = v[i], hi = v[i + half];
      const float send = up ? lo : hi;
      const float keep = up ? hi : lo;
      const float got = __shfl_xor_sync(0xffffffffu, send, o);
      v[i] = kMax ? fmaxf(keep, got) : keep + got;
    }
  }
}

// 4-row gather of a 2-D tensor (box one row high, 64 columns): rows r0..r3 at column x land
// as consecutive 128-byte rows of dst in the map's swizzle, completing 512 bytes on bar.
// dst must lie in a 1024-byte aligned tile (the swizzle follows the shared address).
__device__ __forceinline__ void tma_gather4(const CUtensorMap* map, uint64_t* bar, void* dst,
                                            int32_t x, int32_t r0, int32_t r1, int32_t r2,
                                            int32_t r3) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(tc::smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(tc::smem_u32(bar)), "r"(x), "r"(r0), "r"(r1),
      "r"(r2), "r"(r3)
      : "memory");
}

// mapX views x in one-row boxes (for the 4-row gathers).
__global__ void __launch_bounds__(kThreads, 1)
    attend_tc_kernel(const __grid_constant__ CUtensorMap mapK,
                     const __grid_constant__ CUtensorMap mapX,
                     const __grid_constant__ CUtensorMap mapV, const TcAttendParams p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* stages = smem;
  unsigned char* xbuf = smem + kStages * kStageBytes;
  unsigned char* pbuf = xbuf + kXSlots * kXTile;
  float* red = reinterpret_cast<float*>(pbuf + kPBytes);    // [4][64]
  float* fin_m = red + 4 * kNT;                              // [64]
  float* fin_l = fin_m + kNT;                                // [64]
  int32_t* orig = reinterpret_cast<int32_t*>(fin_l + kNT);  // [64]
  int32_t* xrow = orig + kNT;                                // [64] producer: x row per token
  uint64_t* full = reinterpret_cast<uint64_t*>(xrow + kNT);
  uint64_t* empty = full + kStages;
  uint64_t* xfull = empty + kStages;
  uint64_t* xempty = xfull + kXSlots;
  uint64_t* s_full = xempty + kXSlots;
  uint64_t* s_free = s_full + 1;
  uint64_t* a_full = s_free + 1;
  uint64_t* a_free = a_full + 1;
  uint64_t* drain = a_free + 1;
  uint64_t* grp = drain + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(grp + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // Stage buffers start zeroed so that rows a partial TMA box leaves untouched are finite.
  for (int i = threadIdx.x; i < (kStages * kStageBytes + kXSlots * kXTile) / 16; i += kThreads)
    reinterpret_cast<uint4*>(stages)[i] = make_uint4(0, 0, 0, 0);
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < kXSlots; ++s) {
      tc::mbar_init(&xfull[s], 1);
      tc::mbar_init(&xempty[s], 1);
    }
    tc::mbar_init(s_full, 1);
    tc::mbar_init(s_free, kSoftWarps);
    tc::mbar_init(a_full, 1);
    tc::mbar_init(a_free, kSoftWarps);
    tc::mbar_init(drain, 1);
    tc::mbar_init(grp, kSoftWarps);
    *abort_flag = 0;
    tc::fence_barrier_init();
  }
  tc::fence_proxy_async();
  if (warp == 1) tc::tmem_alloc(tmem_slot, kTmemCols);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  grid_dep_wait();  // the previous kernels' outputs (plan, gathered x) are complete
  grid_dep_release();

  const int n_items = *p.n_items;
  const int KB = p.d / 64;
  const int DC = p.d_v / 128;

  if (warp == 0) {
    if (lane == 0) {
      tc::tma_prefetch_desc(&mapK);
      tc::tma_prefetch_desc(&mapX);
      tc::tma_prefetch_desc(&mapV);
      uint32_t it = 0;
      bool ok = true;
      for (int i = blockIdx.x; ok && i < n_items; i += gridDim.x) {
        const Item item = p.items[i];
        const int r0 = p.offs[item.t];
        const int n = p.offs[item.t + 1] - r0;
        const int RC = (n + 127) / 128;
        for (int kb = 0; ok && kb < KB; ++kb) {
          for (int rc = 0; rc < RC; ++rc) {
            const uint32_t s = it % kStages, ph = (it / kStages) & 1;
            if (!tc::mbar_wait(&empty[s], ph ^ 1, abort_flag, p.st, 0x100)) {
              ok = false;
              break;
            }
            unsigned char* st = stages + s * kStageBytes;
            // one 128-row box of K (rows past the item's range are read and masked): few,
            // large copies keep the TMA unit's issue rate off the critical path
            tc::mbar_arrive_expect_tx(&full[s], uint32_t(kKTile));
            tc::tma_load_2d(&mapK, &full[s], st, kb * 64, r0 + 128 * rc);
            ++it;
          }
        }
        const int NB = (n + 63) / 64;
        for (int b = 0; ok && b < NB; ++b) {
          for (int dc = 0; dc < DC; ++dc) {
            const uint32_t s = it % kStages, ph = (it / kStages) & 1;
            if (!tc::mbar_wait(&empty[s], ph ^ 1, abort_flag, p.st, 0x100)) {
              ok = false;
              break;
            }
            unsigned char* st = stages + s * kStageBytes;
            tc::mbar_arrive_expect_tx(&full[s], 2u * 8192u);
            for (int h = 0; h < 2; ++h)
              tc::tma_load_2d(&mapV, &full[s], st + h * 8192, dc * 128 + h * 64, r0 + 64 * b);
            ++it;
          }
        }
      }
      if (!ok) {
        // Let the copies already issued land before the CTA's shared memory goes away.
        const uint32_t first = it > uint32_t(kStages) ? it - kStages : 0;
        volatile int no_abort = 0;
        for (uint32_t j = first; j < it; ++j)
          tc::mbar_wait(&full[j % kStages], (j / kStages) & 1, &no_abort, p.st, 0x1000,
                        100000000ull);
      }
    }
  } else if (warp == 2 + kSoftWarps) {
    // x producer: per item, the tokens' batch indices (slots past nt repeat the first: read,
    // then masked as the softmax masks token columns past nt), then per 64-wide K block one x
    // box of 16 four-row gathers
    uint32_t xt = 0;
    bool ok = true;
    for (int i = blockIdx.x; ok && i < n_items; i += gridDim.x) {
      const Item item = p.items[i];
      for (int j = lane; j < kNT; j += 32)
        xrow[j] = int32_t(uint32_t(p.sorted_keys[item.q0 + (j < item.nt ? j : 0)]));
      __syncwarp();
      if (lane == 0) {
        for (int kb = 0; kb < KB; ++kb, ++xt) {
          const uint32_t xs = xt % kXSlots, xph = (xt / kXSlots) & 1;
          if (!tc::mbar_wait(&xempty[xs], xph ^ 1, abort_flag, p.st, 0x100)) {
            ok = false;
            break;
          }
          tc::mbar_arrive_expect_tx(&xfull[xs], uint32_t(kXTile));
          unsigned char* xd = xbuf + xs * kXTile;
#pragma unroll 4
          for (int g = 0; g < kNT / 4; ++g)
            tma_gather4(&mapX, &xfull[xs], xd + g * 512, kb * 64, xrow[4 * g],
                        xrow[4 * g + 1], xrow[4 * g + 2], xrow[4 * g + 3]);
        }
      }
      // lane 0's verdict for the whole warp; xrow is rewritten only after its copies issued
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      __syncwarp();
    }
    if (lane == 0 && !ok) {
      volatile int no_abort = 0;
      for (uint32_t j = xt > uint32_t(kXSlots) ? xt - kXSlots : 0; j < xt; ++j)
        tc::mbar_wait(&xfull[j % kXSlots], (j / kXSlots) & 1, &no_abort, p.st, 0x1000,
                      100000000ull);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      uint32_t it = 0, xt = 0, item_no = 0;
      bool ok = true;
      for (int i = blockIdx.x; ok && i < n_items; i += gridDim.x, ++item_no) {
        const Item item = p.items[i];
        const int r0 = p.offs[item.t];
        const int n = p.offs[item.t + 1] - r0;
        const int Nt = (item.nt + 15) & ~15;
        const int RC = (n + 127) / 128;
        const uint32_t id1 = idesc_bf16(128, Nt, 0, 0);
        const uint32_t id2 = idesc_bf16(128, Nt, 1, 1);
        // phase 1: Sᵀ = K_t Xᵀ
        for (int kb = 0; ok && kb < KB; ++kb, ++xt) {
          const uint32_t xs = xt % kXSlots;
          if (!tc::mbar_wait(&xfull[xs], (xt / kXSlots) & 1, abort_flag, p.st, 0x200)) {
            ok = false;
            break;
          }
          const uint32_t b_addr = tc::smem_u32(xbuf + xs * kXTile);
          for (int rc = 0; rc < RC; ++rc) {
            const uint32_t s = it % kStages, ph = (it / kStages) & 1;
            if (!tc::mbar_wait(&full[s], ph, abort_flag, p.st, 0x200)) {
              ok = false;
              break;
            }
            tc::tc_fence_after();
            const uint32_t a_addr = tc::smem_u32(stages + s * kStageBytes);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              tc::mma_bf16(tmem + kSCol + 64 * rc, tc::desc_kmajor_sw128(a_addr + 32 * k),
                           tc::desc_kmajor_sw128(b_addr + 32 * k), id1,
                           (kb > 0 || k > 0) ? 1u : 0u);
            tc::mma_commit(&empty[s]);
            ++it;
          }
          if (!ok) break;
          tc::mma_commit(&xempty[xs]);  // after every chunk's MMAs have read the x box
        }
        if (!ok) break;
        tc::mma_commit(s_full);
        // phase 2 needs Pᵀ (softmax done) and a free Aᵀ (previous epilogue done)
        if (!tc::mbar_wait(s_free, item_no & 1, abort_flag, p.st, 0x400)) break;
        if (!tc::mbar_wait(a_free, (item_no & 1) ^ 1, abort_flag, p.st, 0x400)) break;
        tc::tc_fence_after();
        const int NB = (n + 63) / 64;
        const uint32_t p_addr = tc::smem_u32(pbuf);
        for (int b = 0; ok && b < NB; ++b) {
          for (int dc = 0; dc < DC; ++dc) {
            const uint32_t s = it % kStages, ph = (it / kStages) & 1;
            if (!tc::mbar_wait(&full[s], ph, abort_flag, p.st, 0x200)) {
              ok = false;
              break;
            }
            tc::tc_fence_after();
            const uint32_t v_addr = tc::smem_u32(stages + s * kStageBytes);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              tc::mma_bf16(tmem + kACol + 64 * dc, desc_mnmajor_sw128(v_addr + 2048 * k, 8192),
                           desc_mnmajor_sw128(p_addr + 8192 * b + 2048 * k, 8192), id2,
                           (b > 0 || k > 0) ? 1u : 0u);
            tc::mma_commit(&empty[s]);
            ++it;
          }
        }
        if (!ok) break;
        tc::mma_commit(a_full);
      }
      // All MMAs issued by this thread must finish before TMEM is released.
      tc::mma_commit(drain);
      volatile int no_abort = 0;
      tc::mbar_wait(drain, 0, &no_abort, p.st, 0x2000, 100000000ull);
    }
  } else if (warp < 2 + kSoftWarps) {
    // softmax / epilogue warp (q, h): TMEM lane quarter q (hardware rule: warp % 4), token
    // columns [32 h, 32 h + 32) of the item
    const int q = warp & 3;
    const int h = (warp - 2) >> 2;
    const int L = q * 32 + lane;  // TMEM lane: table row in a chunk / value column in a chunk
    const uint32_t lane_base = tmem + (uint32_t(q * 32) << 16);
    const int j0 = 32 * h;        // first token column of this warp
    uint32_t item_no = 0, gph = 0;
    for (int i = blockIdx.x; i < n_items; i += gridDim.x, ++item_no) {
      const Item item = p.items[i];
      const int r0 = p.offs[item.t];
      const int n = p.offs[item.t + 1] - r0;
      const int nt = item.nt;
      const int RC = (n + 127) / 128;
      const bool cols = j0 < nt;  // this warp has tokens of the item
      if (!wait_own(s_full, item_no & 1, abort_flag, p.st, 0x800)) break;
      tc::tc_fence_after();
      if (h == 0 && L < nt) orig[L] = int32_t(uint32_t(p.sorted_keys[item.q0 + L]));
      // pass 1: per-token max over the rows
      float v[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = -INFINITY;
      if (cols) {
        for (int rc = 0; rc < RC; ++rc) {
          float sv[32];
          tc::tmem_ld32(lane_base + kSCol + 64 * rc + j0, sv);
          if (128 * rc + L < n)
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = fmaxf(v[j], sv[j]);
        }
      }
      reduce_scatter32<true>(v, lane);
      red[q * kNT + j0 + lane] = v[0];
      if (!group_sync(grp, gph, abort_flag, p.st)) break;
      if (q == 0) {
        const int j = j0 + lane;
        fin_m[j] = fmaxf(fmaxf(red[j], red[kNT + j]), fmaxf(red[2 * kNT + j], red[3 * kNT + j]));
      }
      if (!group_sync(grp, gph, abort_flag, p.st)) break;
      // pass 2: e = exp(s - m) as bf16 into Pᵀ, and its sum
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = 0.f;
      const int rows_written = ((n + 63) / 64) * 64;
      // e = 2^(s log2(e) - m log2(e)): one multiply-add and one exp2 per weight (the weights
      // are rounded to bf16 next, far coarser than exp2f's error)
      constexpr float kLog2e = 1.4426950408889634f;
      float mj[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) mj[j] = -fin_m[j0 + j] * kLog2e;
      for (int rc = 0; rc < RC; ++rc) {
        const int row = 128 * rc + L;
        const bool valid = row < n;
        uint32_t packed[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) packed[j] = 0;
        if (cols) {
          float sv[32];
          tc::tmem_ld32(lane_base + kSCol + 64 * rc + j0, sv);
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            const int t0 = j0 + j, t1 = t0 + 1;
            const float e0 = (valid && t0 < nt) ? exp2f(fmaf(sv[j], kLog2e, mj[j])) : 0.f;
            const float e1 = (valid && t1 < nt) ? exp2f(fmaf(sv[j + 1], kLog2e, mj[j + 1])) : 0.f;
            // one paired conversion (the scalar ones run at a fraction of its rate)
            const __nv_bfloat162 b01 = __floats2bfloat162_rn(e0, e1);
            uint32_t w;
            memcpy(&w, &b01, sizeof(w));
            v[j] += __uint_as_float(w << 16);
            v[j + 1] += __uint_as_float(w & 0xffff0000u);
            packed[j / 2] = w;
          }
        }
        if (row < rows_written) {
          // this warp's half of a Pᵀ row: tokens j0 .. j0 + 31 = 16-byte chunks 4 h .. 4 h + 3
          // of the row's 128 bytes, 128-byte swizzle within 8-row groups
          unsigned char* prow = pbuf + row * 128;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int c16 = 4 * h + c;
            *reinterpret_cast<uint4*>(prow + ((c16 ^ (row & 7)) << 4)) =
                make_uint4(packed[4 * c], packed[4 * c + 1], packed[4 * c + 2], packed[4 * c + 3]);
          }
        }
      }
      tc::fence_proxy_async();
      reduce_scatter32<false>(v, lane);
      red[q * kNT + j0 + lane] = v[0];
      if (!group_sync(grp, gph, abort_flag, p.st)) break;
      if (q == 0) {
        const int j = j0 + lane;
        fin_l[j] = (red[j] + red[kNT + j]) + (red[2 * kNT + j] + red[3 * kNT + j]);
      }
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(s_free);
      if (!group_sync(grp, gph, abort_flag, p.st)) break;  // fin_l visible to all warps
      // epilogue: a = Aᵀ / l, batch order
      if (!wait_own(a_full, item_no & 1, abort_flag, p.st, 0x800)) break;
      tc::tc_fence_after();
      if (cols) {
        float inv[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) inv[j] = 1.f / fin_l[j0 + j];
        for (int dc = 0; dc < DC; ++dc) {
          const int col = 128 * dc + L;
          float acc[32];
          tc::tmem_ld32(lane_base + kACol + 64 * dc + j0, acc);
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int tok = j0 + j;
            if (tok < nt) {
              const float a = acc[j] * inv[j];
              const int64_t o = int64_t(orig[tok]) * p.d_v + col;
              p.a_bf16[o] = __float2bfloat16_rn(a);
              if (p.a_f32) p.a_f32[o] = a;
            }
          }
        }
      }
      if (p.ml && h == 0 && L < nt) {
        p.ml[2 * int64_t(orig[L])] = fin_m[L];
        p.ml[2 * int64_t(orig[L]) + 1] = fin_l[L];
      }
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(a_free);
      if (!group_sync(grp, gph, abort_flag, p.st)) break;  // orig/fin_* are rewritten next
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

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// bf16 [rows, cols] row-major; box box_rows rows x 64 columns, 128-byte swizzle.
bool make_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cuuint64_t(cols), cuuint64_t(rows)};
  cuuint64_t strides[1] = {cuuint64_t(cols) * 2};
  cuuint32_t box[2] = {64, cuuint32_t(box_rows)};
  cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() { return device_sm_count(); }

}  // namespace

int attend_tc_threshold(int64_t T, int d, int d_v, int dtype) {
  // Segments of fewer tokens have too little arithmetic per table byte for tensor cores:
  // the split-row CUDA-core kernel streams them at memory speed.
  const bool ok = dtype == L3_BF16 && T >= 1024 && d % 64 == 0 && d_v % 128 == 0 && d_v <= 512;
  return ok ? 8 : 0;
}

cudaError_t launch_attend_tc(const AttendTcArgs& a, cudaStream_t stream) {
  if (a.T <= 0 || a.max_items <= 0) return cudaSuccess;
  CUtensorMap mk, mx, mv;
  // x in one-row boxes for the kernel's 4-row gathers (x is 16-byte aligned)
  if (!make_map(&mk, a.K, a.v, a.d, 128) || !make_map(&mx, a.x, a.T, a.d, 1) ||
      !make_map(&mv, a.V, a.v, a.d_v, 64))
    return cudaErrorInvalidValue;
  const Item* items = a.items;
  TcAttendParams p{};
  p.items = items;
  p.n_items = a.hdr + kPlanItems;
  p.sorted_keys = a.sorted_keys;
  p.offs = a.offs;
  p.d = a.d;
  p.d_v = a.d_v;
  p.a_bf16 = a.a_bf16;
  p.a_f32 = a.a_f32;
  p.ml = a.ml;
  p.st = a.st;
  const cudaError_t attr = ensure_smem_attr(attend_tc_kernel, kSmemBytes);
  if (attr != cudaSuccess) return attr;
  const cudaError_t e = launch_pdl(attend_tc_kernel, dim3(sm_count()), dim3(kThreads),
                                   size_t(kSmemBytes), stream, mk, mx, mv, p);
  count_launch();
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace l3
