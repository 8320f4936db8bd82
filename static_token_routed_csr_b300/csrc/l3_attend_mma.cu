// Gather-attend forward of bf16 layers for the short segments of equal ids (all segments of
// a small batch), rows split across the GPU, products on warp-level tensor cores:
//   for each token i with id t (rows R = offs[t] .. offs[t+1]-1):
//   s = K_R x_i,  p = softmax(s),  a_i = V_Rᵀ p
// ("L³: Large Lookup Layers", gist.science explainer, Technical Summary, "Core
// Architecture"; "Systems-Friendly Design": the batch sorted by id, so a group of up to 8
// tokens of one id shares every row it reads).
//
// Work list: the routing pass's plan (groups of <= 8 tokens, each group's rows in chunks of
// `ch` = 8 or 16 rows), cut into one contiguous chunk range per persistent CTA (one per SM)
// so that the ranges cost about the same: the plan weighs each chunk and, on top, each
// group start, since a group's x loads and output writes take about as long as a chunk.
// A consumer step takes two consecutive chunks of a group (16 or 32 rows) when it can.
//
// Data movement: a chunk's K rows and V rows are each one TMA copy. The tables are viewed
// as 3-D tensors [column block of 64][row][64 columns] with the 128-byte swizzle, so a copy
// lands the chunk as ch-row by 128-byte atoms whose 16-byte pieces are XOR-permuted by row:
// the matrix loads below read them without shared-memory bank conflicts. A producer warp
// keeps a ring of up to 6 stages in flight: it waits for a stage to be free, writes the
// stage's group description (token indices included, read from the plan 32 groups at a
// time), arms a metadata barrier, then issues the two copies; metadata/full/empty
// mbarriers per stage, all waits bounded. The consumers never walk the plan themselves.
//
// Per chunk (8 consumer warps, synchronised by a named barrier the producer is not in):
//   scores  Sᵀ[rows][tokens] = K_chunk Xᵀ with mma.sync m16n8k16 (bf16 in, fp32 out): the
//           chunk's rows are M, the group's 8 token slots are N, and d is dealt to the
//           warps in 16-wide steps. Each warp loads its steps' Xᵀ fragments from x into
//           registers once per group, so per chunk only K is read from shared memory. bf16
//           products are exact in fp32: this is fp32 accumulation of the bf16 inputs.
//   softmax online update of the running max m and denominator l per token, and the
//           chunk's weights e = exp(s - m) (fp32).
//   values  accᵀ[d_v][tokens] = accᵀ * e^(m_old - m) + V_chunkᵀ Pᵀ, mma.sync with the
//           value columns as M and the weights as N. The weights enter as two bf16 terms
//           (hi = bf16(e), lo = bf16(e - hi)), which keeps them to about 2^-17 relative
//           error; the accumulator stays in registers for the whole group.
// A group that ends inside the CTA's range is finished there; otherwise its partial
// (m, l, acc) is merged by the CTA that completes the group's chunk count
// (see l3_attend_split.cuh).
#include <cudaTypedefs.h>

#include <mutex>

#include "l3_attend_split.cuh"
#include "l3_mma.cuh"

namespace l3 {

namespace {

using namespace split;
using namespace wmma;

constexpr int kWarps = kThreads / 32;       // consumer warps (scores, softmax, values)
constexpr int kCtaThreads = kThreads + 32;  // + one producer warp (TMA copies)
constexpr int kMaxStages = 6;
constexpr int kMaxMTiles = 4;   // 16-column value tiles per warp (d_v <= 512)
constexpr int kMaxKSteps = 16;  // 16-wide k-steps per warp (d <= 2048)
constexpr int kRedLd = 36;      // row stride of red (32 rows + 4)
constexpr int kEld = 40;        // row stride of e_buf (32 rows + 8, pairs 8-byte aligned)

// Group of a stage's chunk, written by the producer before it arms the stage's full
// barrier: the consumers take a new group's description and token indices from here.
struct StageMeta {
  int32_t g, q0, mt, n, c0, c1, pad0, pad1;
  int32_t tok[kMT];  // batch index of each of the group's tokens
};

struct Misc {
  StageMeta meta[kMaxStages];
  uint64_t meta_full[kMaxStages];  // the stage's StageMeta is written (before its copies land)
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  // Token-major, rows padded so that the softmax threads (one row each) read a token's row
  // partials from distinct banks, and the MMA lanes store theirs without conflicts.
  float red[kWarps][kMT][kRedLd];  // per-warp score partials (up to 32 rows per step)
  float e_buf[kMT][kEld];          // the step's weights e = exp(s - m) per token and row
  float m_run[2][kMT];
  float l_run[2][kMT];
  float scale[kMT];
  MergeSmem merge;
  int abort;
};

struct MmaShape {
  int ch;           // rows per chunk: 8 or 16
  int stages;
  int k_bytes;      // K block of a stage: ch rows x d
  int stage_bytes;  // K block, then the V block (ch rows x d_v)
  int smem;
};

MmaShape mma_shape(int d, int d_v) {
  MmaShape s{};
  s.ch = 16 * 2 * (d + d_v) <= 49152 ? 16 : 8;
  s.k_bytes = s.ch * 2 * d;
  s.stage_bytes = int(align_up(size_t(s.ch) * 2 * (d + d_v), 1024));
  const int fixed = 1024 + int(align_up(sizeof(Misc), 128));
  s.stages = (kSmemLimit - fixed) / s.stage_bytes;
  if (s.stages > kMaxStages) s.stages = kMaxStages;
  s.smem = fixed + s.stages * s.stage_bytes;
  return s;
}


// t[j] for j < 8 held in registers (a select chain, no local memory).
__device__ __forceinline__ int pick8(const int32_t (&t)[kMT], int j) {
  int v = t[0];
#pragma unroll
  for (int i = 1; i < kMT; ++i) v = j == i ? t[i] : v;
  return v;
}

// Barrier of the kThreads consumer threads (named barrier 1; the producer warp is not in it).
__device__ __forceinline__ void cbar() { asm volatile("bar.sync 1, %0;" ::"n"(kThreads) : "memory"); }

// CH: rows per chunk (8 or 16); a step takes up to two chunks of a group, RS = 2 CH rows
// (MS = RS / 16 tiles of 16 rows). KSW / MTW: k-steps / value tiles per warp when the
// shape fixes them at compile time (0: taken from d, d_v at run time, loops guarded).
template <int CH, int KSW, int MTW>
__global__ void __launch_bounds__(kCtaThreads, 1)
    attend_mma_kernel(const __grid_constant__ CUtensorMap mapK,
                      const __grid_constant__ CUtensorMap mapV, const AttendArgs a,
                      const MmaShape sh) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* ring = base;
  Misc* ms = reinterpret_cast<Misc*>(base + sh.stages * sh.stage_bytes);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g8 = lane >> 2, t4 = lane & 3;  // mma fragment coordinates
  const int b = blockIdx.x;
  if (tid == 0) {
    tc::tma_prefetch_desc(&mapK);
    tc::tma_prefetch_desc(&mapV);
  }
  grid_dep_wait();  // the routing kernel's plan is complete
  grid_dep_release();
  // The CTA's head (one 80-byte read by every thread): its chunk range and the group that
  // holds its first chunk, so that the copies and the first group's x loads start at once.
  const CtaHead hd = a.cta_head[b];
  const int total_chunks = a.hdr[kPlanChunks];
  const int64_t cb = hd.cb, ce = hd.ce;
  if (cb >= ce) return;
  if (hd.mt < 1 || hd.mt > kMT || hd.q0 < 0 || int64_t(hd.q0) + hd.mt > a.T || cb < hd.c0 ||
      cb >= hd.c1 || ce > total_chunks) {
    // an inconsistent plan (never expected): nothing is read or written
    if (tid == 0) atomicOr(&a.st->timeout, 0x1000000);
    return;
  }
  const int nk = int(ce - cb);
  const int d = a.d, dv = a.d_v, S = sh.stages;
  const __nv_bfloat16* __restrict__ Xg = static_cast<const __nv_bfloat16*>(a.x);
  const AttendGroup* __restrict__ groups = a.groups;
  const uint32_t ring_s = tc::smem_u32(ring);

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      tc::mbar_init(&ms->meta_full[s], 1);
      tc::mbar_init(&ms->full[s], 1);
      tc::mbar_init(&ms->empty[s], 1);
    }
    ms->abort = 0;
    tc::fence_barrier_init();
  }
  __syncthreads();

  volatile int* abort_flag = &ms->abort;

  // Producer (warp kWarps): lane 0 issues two TMA copies per chunk once the consumers have
  // released the stage; when it moves on to a new group, the whole warp prefetches that
  // group's x rows into L2, several chunks before the consumers load them. The group being
  // fetched is kept in registers.
  if (warp == kWarps) {
    // The plan's group list is read 32 groups at a time (lane l holds group w0 + l) and the
    // current group's fields are taken from the window by shuffles.
    const uint32_t tx = uint32_t(CH) * 2u * uint32_t(d + dv);
    // The range's first group comes from the head: the copies of its first chunks go out
    // at once; the group list is read meanwhile.
    int pg = hd.g;
    int g_q0 = hd.q0, g_mt = hd.mt, g_n = hd.n, g_row0 = hd.row0, g_c0 = hd.c0;
    int64_t p_next = hd.c1;
    const int r_first = hd.row;
    int ptok = pick8(hd.tok, lane & 7);  // lane j < 8: token j
    int early = int(p_next - cb);
    early = early < S ? early : S;
    early = early < nk ? early : nk;
    if (lane == 0) {
      for (int e = 0; e < early; ++e) {
        const uint32_t st = ring_s + uint32_t(e * sh.stage_bytes);
        tc::mbar_arrive_expect_tx(&ms->full[e], tx);
        tma_load_3d(&mapK, &ms->full[e], st, 0, r_first + e * CH, 0);
        tma_load_3d(&mapV, &ms->full[e], st + uint32_t(sh.k_bytes), 0, r_first + e * CH, 0);
      }
    }
    // The plan's group list is read 32 groups at a time (lane l holds group w0 + l) and the
    // fields of later groups are taken from the window by shuffles.
    const int n_groups = a.hdr[kPlanGroups];
    int w0 = pg;
    AttendGroup wg{};
    auto load_window = [&]() {
      if (w0 + lane <= n_groups) wg = groups[w0 + lane];
    };
    load_window();  // first used when the producer moves past the first group
    auto take = [&]() {  // fields of group pg; pg and pg + 1 lie in the window
      const int src = pg - w0;
      g_q0 = __shfl_sync(0xffffffffu, wg.q0, src);
      g_mt = __shfl_sync(0xffffffffu, wg.mt, src);
      g_n = __shfl_sync(0xffffffffu, wg.n, src);
      g_row0 = __shfl_sync(0xffffffffu, wg.row0, src);
      g_c0 = __shfl_sync(0xffffffffu, wg.c0, src);
      p_next = __shfl_sync(0xffffffffu, wg.c0, src + 1);
#pragma unroll
      for (int j = 0; j < kMT; ++j) {
        const int v = __shfl_sync(0xffffffffu, wg.tok[j], src);
        if (lane == j) ptok = v;
      }
    };
    auto prefetch_x = [&]() {
      for (int j = 0; j < g_mt; ++j) {
        const char* row = reinterpret_cast<const char*>(
            Xg + int64_t(__shfl_sync(0xffffffffu, ptok, j)) * d);
        for (int off = lane * 128; off < 2 * d; off += 32 * 128)
          asm volatile("prefetch.global.L2 [%0];" ::"l"(row + off));
      }
    };
    prefetch_x();
    int issued = 0;
    for (; issued < nk; ++issued) {
      const int s = issued % S;
      int ok = 1;
      // The first S stages start free. They are not waited for: the consumers take the first
      // group from the head and may already have released some of the early copies' stages,
      // which would put empty[s] one phase past the one a first-round wait expects.
      if (lane == 0 && issued >= S)
        ok = tc::mbar_wait_watch(&ms->empty[s], ((issued / S) & 1) ^ 1, abort_flag, a.st,
                                 0x40000)
                 ? 1
                 : 0;
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
      const int64_t c = cb + issued;
      bool fresh = false;
      while (p_next <= c && pg < n_groups) {
        ++pg;
        if (pg + 1 - w0 > 31) {
          w0 = pg;
          load_window();
        }
        take();
        fresh = true;
      }
      if (p_next <= c) {  // no group holds chunk c: an inconsistent plan (never expected)
        if (lane == 0) atomicOr(&a.st->timeout, 0x1000000);
        break;
      }
      // the stage's group description (the consumers read it once meta_full is armed)
      StageMeta* m = &ms->meta[s];
      if (lane < kMT) m->tok[lane] = ptok;
      if (lane == 0) {
        m->g = pg;
        m->q0 = g_q0;
        m->mt = g_mt;
        m->n = g_n;
        m->c0 = g_c0;
        m->c1 = int32_t(p_next);
      }
      __syncwarp();
      if (lane == 0) {
        tc::mbar_arrive(&ms->meta_full[s]);
        if (issued >= early) {  // (the first `early` chunks' copies are in flight)
          const int r0 = g_row0 + int(c - g_c0) * CH;
          const uint32_t st = ring_s + uint32_t(s * sh.stage_bytes);
          tc::mbar_arrive_expect_tx(&ms->full[s], tx);
          tma_load_3d(&mapK, &ms->full[s], st, 0, r0, 0);
          tma_load_3d(&mapV, &ms->full[s], st + uint32_t(sh.k_bytes), 0, r0, 0);
        }
      }
      if (fresh) prefetch_x();
    }
    if (issued < nk && lane == 0) {
      // Stopped early: let the copies in flight land before the CTA's memory goes away.
      volatile int no_abort = 0;
      for (int j = issued - S > 0 ? issued - S : 0; j < issued; ++j)
        tc::mbar_wait(&ms->full[j % S], (j / S) & 1, &no_abort, a.st, 0x20000, 100000000ull);
    }
    return;
  }

  const int n_mt = dv / 16;   // value tiles
  const int nks = d / 16;     // k-steps; warp w takes w, w + 8, ...
  constexpr int KS = KSW ? KSW : kMaxKSteps;
  constexpr int MT = MTW ? MTW : kMaxMTiles;
  constexpr int RS = 2 * CH;  // rows per step
  constexpr int MS = RS / 16;
  float acc[MT][4];
  uint32_t bx[KS][2];  // Xᵀ fragments of this warp's k-steps
  // current group: index, first sorted position, tokens, rows, chunk range [gc0, c_next)
  int cg = -1, q0 = 0, mt = 0, gn = 0;
  int64_t gc0 = 0, c_next = -1;
  // batch indices of this lane's two token slots (2 t4, 2 t4 + 1) and of token tid
  int64_t i0 = 0, i1 = 0, itid = 0;
  bool ok = true;

  auto finish = [&](int par) {
    const int64_t c0 = gc0, c1 = c_next;
    const bool whole = c0 >= cb && c1 <= ce;
    const bool second = c0 > cb;
    const int n0 = 2 * t4, n1 = 2 * t4 + 1;  // this lane's token slots
    const float inv0 = n0 < mt ? 1.f / ms->l_run[par][n0] : 0.f;
    const float inv1 = n1 < mt ? 1.f / ms->l_run[par][n1] : 0.f;
#pragma unroll
    for (int mi = 0; mi < MT; ++mi) {
      const int mtile = warp + kWarps * mi;
      if (!MTW && mtile >= n_mt) break;
      const int col0 = 16 * mtile + g8, col1 = col0 + 8;
      if (whole) {
        if (n0 < mt) {
          write_a(a, i0, col0, acc[mi][0] * inv0);
          write_a(a, i0, col1, acc[mi][2] * inv0);
        }
        if (n1 < mt) {
          write_a(a, i1, col0, acc[mi][1] * inv1);
          write_a(a, i1, col1, acc[mi][3] * inv1);
        }
      } else {
        if (n0 < mt) {
          float* pe = part_entry(a, b, second, n0);
          pe[2 + col0] = acc[mi][0];
          pe[2 + col1] = acc[mi][2];
        }
        if (n1 < mt) {
          float* pe = part_entry(a, b, second, n1);
          pe[2 + col0] = acc[mi][1];
          pe[2 + col1] = acc[mi][3];
        }
      }
    }
    if (whole) {
      if (a.ml && tid < mt) {
        a.ml[2 * itid] = ms->m_run[par][tid];
        a.ml[2 * itid + 1] = ms->l_run[par][tid];
      }
      return;
    }
    if (tid < mt) {
      float* pe = part_entry(a, b, second, tid);
      pe[0] = ms->m_run[par][tid];
      pe[1] = ms->l_run[par][tid];
    }
    // the CTA that completes the group's chunk count merges the partials
    arrive_and_merge(a, cg, c0, c1, cb, ce, q0, mt, &ms->merge, tid, kThreads, [] { cbar(); });
  };

  // A consumer step takes one chunk, or two consecutive chunks of the same group (stages k
  // and k+1): RS = 2 CH rows, row R of the step is row R % CH of chunk R / CH.
  // Xᵀ fragments of this warp's k-steps for the group of stage meta m, straight from x
  // (tokens past mt zero): b0 = x[token g8][16 s + 2 t4 .. +1], b1 = x[token g8][16 s + 8 + ..]
  auto load_x = [&](int tok_g8, int m_mt) {  // tok_g8: batch index of the group's token g8
    const unsigned int* xrow = nullptr;
    if (g8 < m_mt && tok_g8 >= 0 && tok_g8 < a.T)
      xrow = reinterpret_cast<const unsigned int*>(Xg + int64_t(tok_g8) * d);
#pragma unroll
    for (int i = 0; i < KS; ++i) {
      const int s16 = warp + kWarps * i;
      bx[i][0] = bx[i][1] = 0u;
      if ((KSW || s16 < nks) && xrow) {
        bx[i][0] = __ldg(xrow + 8 * s16 + t4);
        bx[i][1] = __ldg(xrow + 8 * s16 + 4 + t4);
      }
    }
  };
  uint32_t u = 0;  // steps done: (m, l) of the current group live in m_run/l_run[u & 1]
  {  // the range's first group, from the head (the consumers never wait for its metadata)
    cg = hd.g;
    q0 = hd.q0;
    mt = hd.mt;
    gn = hd.n;
    gc0 = hd.c0;
    c_next = hd.c1;
    i0 = 2 * t4 < mt ? int64_t(pick8(hd.tok, 2 * t4)) : 0;
    i1 = 2 * t4 + 1 < mt ? int64_t(pick8(hd.tok, 2 * t4 + 1)) : 0;
    itid = tid < mt ? int64_t(pick8(hd.tok, tid & 7)) : 0;
    load_x(pick8(hd.tok, g8), mt);
#pragma unroll
    for (int mi = 0; mi < MT; ++mi) acc[mi][0] = acc[mi][1] = acc[mi][2] = acc[mi][3] = 0.f;
    if (tid < kMT) {
      ms->m_run[0][tid] = -INFINITY;
      ms->l_run[0][tid] = 0.f;
    }
  }
  for (int k = 0; k < nk;) {
    const int64_t c = cb + k;
    if (c >= c_next) {  // the chunk opens the next group
      if (cg >= 0) {
        finish(u & 1);
        cbar();
      }
      // the group's description travels with its first stage in this CTA (published before
      // the stage's copies are issued, so x is fetched while they are in flight)
      const bool got =
          tc::mbar_wait(&ms->meta_full[k % S], (k / S) & 1, abort_flag, a.st, 0x10000);
      const StageMeta* m = &ms->meta[k % S];
      if (got) {
        cg = m->g;
        q0 = m->q0;
        mt = m->mt;
        gn = m->n;
        gc0 = m->c0;
        c_next = m->c1;
      } else {  // stopping: the barrier check below ends the loop
        mt = 0;
        gn = 0;
        gc0 = c;
        c_next = c + 1;
      }
      i0 = 2 * t4 < mt ? int64_t(m->tok[2 * t4]) : 0;
      i1 = 2 * t4 + 1 < mt ? int64_t(m->tok[2 * t4 + 1]) : 0;
      itid = tid < mt ? int64_t(m->tok[tid]) : 0;
      load_x(m->tok[g8], mt);
#pragma unroll
      for (int mi = 0; mi < MT; ++mi) acc[mi][0] = acc[mi][1] = acc[mi][2] = acc[mi][3] = 0.f;
      if (tid < kMT) {
        ms->m_run[u & 1][tid] = -INFINITY;
        ms->l_run[u & 1][tid] = 0.f;
      }
    }
    const int j0 = int(c - gc0);
    const int nr0 = gn - j0 * CH < CH ? gn - j0 * CH : CH;
    const bool pair = k + 1 < nk && c + 1 < c_next;
    const int nr1 = pair ? (gn - (j0 + 1) * CH < CH ? gn - (j0 + 1) * CH : CH) : 0;

    tc::mbar_wait(&ms->full[k % S], (k / S) & 1, abort_flag, a.st, 0x10000);
    if (pair) tc::mbar_wait(&ms->full[(k + 1) % S], ((k + 1) / S) & 1, abort_flag, a.st, 0x10000);
    cbar();
    if (*abort_flag) {  // some consumer's wait ran out (it set the flag before the barrier)
      ok = false;
      break;
    }
    const uint32_t st0 = ring_s + uint32_t((k % S) * sh.stage_bytes);
    const uint32_t st1 = pair ? ring_s + uint32_t(((k + 1) % S) * sh.stage_bytes) : st0;
    // stage and row of step row R (a lone chunk's second half repeats the first, masked)
    auto stage_of = [&](int R) { return R < CH ? st0 : st1; };

    // scores: Sᵀ = K Xᵀ, one 16-row tile per MS
    {
      float sc[MS][4][4];
#pragma unroll
      for (int t = 0; t < MS; ++t)
#pragma unroll
        for (int u4 = 0; u4 < 4; ++u4) sc[t][u4][0] = sc[t][u4][1] = sc[t][u4][2] = sc[t][u4][3] = 0.f;
      // A: matrix q from lanes 8q..8q+7 (q = 0: rows 0-7, k 0-7; 1: rows 8-15, k 0-7;
      // 2: rows 0-7, k 8-15; 3: rows 8-15, k 8-15) of tile t (step rows 16 t ..)
      const int lrow = (lane & 7) + ((lane >> 3) & 1) * 8;
      const int akof = (lane >> 4) * 8;
      uint32_t abase[MS];
      int arow[MS];
#pragma unroll
      for (int t = 0; t < MS; ++t) {
        const int R = 16 * t + lrow;
        abase[t] = stage_of(R);
        arow[t] = R % CH;
      }
#pragma unroll
      for (int i = 0; i < KS; ++i) {
        const int s16 = warp + kWarps * i;
        if (KSW || s16 < nks) {
#pragma unroll
          for (int t = 0; t < MS; ++t) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4(abase[t] + sw128(CH, arow[t], s16 * 16 + akof), a0, a1, a2, a3);
            mma16(sc[t][i & 3], a0, a1, a2, a3, bx[i][0], bx[i][1]);
          }
        }
      }
#pragma unroll
      for (int t = 0; t < MS; ++t) {
        float r4[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
          r4[i] = (sc[t][0][i] + sc[t][1][i]) + (sc[t][2][i] + sc[t][3][i]);
        ms->red[warp][2 * t4][16 * t + g8] = r4[0];
        ms->red[warp][2 * t4 + 1][16 * t + g8] = r4[1];
        ms->red[warp][2 * t4][16 * t + g8 + 8] = r4[2];
        ms->red[warp][2 * t4 + 1][16 * t + g8 + 8] = r4[3];
      }
    }
    cbar();
    // softmax update: thread (token j = tid / RS, row r = tid % RS) sums the warps' partial
    // score; the RS lanes of a token reduce max and sum by shuffles.
    const uint32_t par = u & 1;
    if (tid < RS * kMT) {
      const int j = tid / RS, r = tid % RS;
      const bool rv = r < CH ? r < nr0 : r - CH < nr1;
      float sv = 0.f;
#pragma unroll
      for (int w = 0; w < kWarps; ++w) sv += ms->red[w][j][r];
      const float mo = ms->m_run[par][j];
      float mx = rv ? sv : -INFINITY;
#pragma unroll
      for (int o = RS / 2; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      const float mn = fmaxf(mo, mx);
      const float e = (rv && j < mt) ? expf(sv - mn) : 0.f;
      float sum = e;
#pragma unroll
      for (int o = RS / 2; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      ms->e_buf[j][r] = e;
      if (r == 0) {
        if (j < mt) {
          const float scl = expf(mo - mn);
          ms->scale[j] = scl;
          ms->m_run[par ^ 1][j] = mn;
          ms->l_run[par ^ 1][j] = fmaf(ms->l_run[par][j], scl, sum);
        } else {
          ms->scale[j] = 0.f;
        }
      }
    }
    cbar();
    // values: accᵀ = accᵀ * scale + Vᵀ Pᵀ over the step's RS rows (P as bf16 hi + lo), one
    // 16-row k-step per tile t
    {
      const float sc0 = ms->scale[2 * t4], sc1 = ms->scale[2 * t4 + 1];
      uint32_t bh[MS][2], bl[MS][2];
#pragma unroll
      for (int t = 0; t < MS; ++t) {
        const float2 e0 = *reinterpret_cast<const float2*>(&ms->e_buf[g8][16 * t + 2 * t4]);
        const float2 e1 = *reinterpret_cast<const float2*>(&ms->e_buf[g8][16 * t + 2 * t4 + 8]);
        split_pair(e0.x, e0.y, bh[t][0], bl[t][0]);
        split_pair(e1.x, e1.y, bh[t][1], bl[t][1]);
      }
      // Vᵀ tile (16 value columns x 16 rows) by transposing loads: lanes 0-7 rows 0-7 at
      // column 0, lanes 8-15 rows 0-7 at column 8, lanes 16-31 rows 8-15
      const int vl = (lane & 7) + (lane >> 4) * 8;
      const int vcol = ((lane >> 3) & 1) * 8;
      uint32_t vb[MS];
      int vrow[MS];
#pragma unroll
      for (int t = 0; t < MS; ++t) {
        const int R = 16 * t + vl;
        vb[t] = stage_of(R) + uint32_t(sh.k_bytes);
        vrow[t] = R % CH;
      }
#pragma unroll
      for (int mi = 0; mi < MT; ++mi) {
        const int mtile = warp + kWarps * mi;
        if (MTW || mtile < n_mt) {
          acc[mi][0] *= sc0;
          acc[mi][1] *= sc1;
          acc[mi][2] *= sc0;
          acc[mi][3] *= sc1;
        }
      }
#pragma unroll
      for (int t = 0; t < MS; ++t) {
        uint32_t va[MT][4];
#pragma unroll
        for (int mi = 0; mi < MT; ++mi) {
          const int mtile = warp + kWarps * mi;
          if (MTW || mtile < n_mt)
            ldsm_x4_t(vb[t] + sw128(CH, vrow[t], 16 * mtile + vcol), va[mi][0], va[mi][1],
                      va[mi][2], va[mi][3]);
        }
        // all hi products, then all lo products: dependent pairs are MT mmas apart
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t b0 = h ? bl[t][0] : bh[t][0], b1 = h ? bl[t][1] : bh[t][1];
#pragma unroll
          for (int mi = 0; mi < MT; ++mi)
            if (MTW || warp + kWarps * mi < n_mt)
              mma16(acc[mi], va[mi][0], va[mi][1], va[mi][2], va[mi][3], b0, b1);
        }
      }
    }
    cbar();  // the stages and the score buffers are free again
    if (tid == 0) {
      tc::mbar_arrive(&ms->empty[k % S]);
      if (pair) tc::mbar_arrive(&ms->empty[(k + 1) % S]);
    }
    k += pair ? 2 : 1;
    ++u;
  }

  if (ok && cg >= 0) finish(u & 1);
}

template <int CH, int KSW, int MTW>
cudaError_t launch_ch(const AttendArgs& a, const MmaShape& sh, cudaStream_t stream) {
  CUtensorMap mk, mv;
  if (!make_row_block_map(&mk, a.K, a.v, a.d, CH) || !make_row_block_map(&mv, a.V, a.v, a.d_v, CH))
    return cudaErrorInvalidValue;
  const cudaError_t attr = ensure_smem_attr(attend_mma_kernel<CH, KSW, MTW>, kSmemLimit);
  if (attr != cudaSuccess) return attr;
  if (a.n_cta < 1 || a.n_cta > kMaxCtas) return cudaErrorInvalidValue;
  const cudaError_t e = launch_pdl(attend_mma_kernel<CH, KSW, MTW>, dim3(a.n_cta),
                                   dim3(kCtaThreads), size_t(sh.smem), stream, mk, mv, a, sh);
  count_launch();
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

namespace wmma {
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// bf16 table [rows, cols] viewed as [cols / 64][rows][64]; box: `box_cblocks` column blocks
// (all when 0) of `box_rows` rows, 128-byte swizzle.
bool make_row_block_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols,
                        int box_rows, int box_cblocks) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {64, cuuint64_t(rows), cuuint64_t(cols / 64)};
  cuuint64_t strides[2] = {cuuint64_t(cols) * 2, 128};
  cuuint32_t box[3] = {64, cuuint32_t(box_rows),
                       cuuint32_t(box_cblocks > 0 ? box_cblocks : cols / 64)};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace wmma

int attend_mma_rows_per_chunk(int d, int d_v) { return mma_shape(d, d_v).ch; }

int attend_mma_ctas(int, int) { return sm_count() < kMaxCtas ? sm_count() : kMaxCtas; }

cudaError_t launch_attend_mma(const AttendArgs& a, cudaStream_t stream) {
  const MmaShape sh = mma_shape(a.d, a.d_v);
  if (sh.stages < 2 || sh.smem > kSmemLimit || sh.ch != a.ch ||
      a.d_v > 16 * kWarps * kMaxMTiles || a.d > 16 * kWarps * kMaxKSteps || a.d % 64 != 0 ||
      a.d_v % 64 != 0)
    return cudaErrorInvalidValue;
  // the two table shapes of the benchmark presets get fully unrolled loops
  if (sh.ch == 8 && a.d == 2048 && a.d_v == 512) return launch_ch<8, 16, 4>(a, sh, stream);
  if (sh.ch == 16 && a.d == 1024 && a.d_v == 256) return launch_ch<16, 8, 2>(a, sh, stream);
  return sh.ch == 16 ? launch_ch<16, 0, 0>(a, sh, stream) : launch_ch<8, 0, 0>(a, sh, stream);
}

}  // namespace l3
