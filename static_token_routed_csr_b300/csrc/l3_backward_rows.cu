// Backward pass of bf16 layers at batch scale, with the table gradients kept for the rows
// the batch touches ("L³: Large Lookup Layers", gist.science explainer, Technical Summary:
// "Core Architecture" gives the formula this differentiates; "Systems-Friendly Design":
// the batch sorted by token id, so each id's tokens form one segment and each table row
// belongs to exactly one segment, whose tokens alone contribute to the row's gradient).
//
// For token i (id t, rows R = offs[t] ..) with the forward's saved m_i, l_i, a_i, and
// da_i = W_upᵀ du_i from the GEMMs:
//   s_j = K_j · x_i,  p_j = exp(s_j - m_i) / l_i,  dp_j = V_j · da_i,
//   ds_j = p_j (dp_j - δ_i) with δ_i = a_i · da_i (which equals Σ_j p_j dp_j),
//   dx_i += Σ_j ds_j K_j,  dK_j = Σ_{i of t} ds_ij x_i,  dV_j = Σ_{i of t} p_ij da_i.
//
// Phase A (attend_bwd_kernel) takes the routing plan's groups of at most 8 tokens of one id,
// whole groups per CTA (cut by the plan's cost units: a chunk and a group start each cost
// a fixed share). Per group it streams the id's rows (TMA, as the forward's split-row
// kernel) and computes the scores and dp with warp MMAs (x and da fragments loaded straight
// from the sorted rows, which the producer prefetches into L2 when it reaches the group; da
// as bf16 hi + lo, so that dp and δ = a · da agree to about 2^-17 and ds = p (dp - δ) keeps
// its digits), p and ds in fp32 (stored per sorted position and row), and the attention
// term of dx with a warp MMA over Kᵀ with ds as bf16 hi + lo, stored to dx (the direct term
// is added afterwards). No group is split, so no merge is needed.
// Phase B (seg_rows_kernel) takes, per id segment, 64-row blocks x 256-column blocks of
// [dK | dV]: the sums over the segment's tokens (x or da rows in sorted order, p or ds as
// bf16 hi + lo), written in segment order to the compact row outputs with each row's table
// index. Both phases are deterministic: fixed summation orders and no floating atomics.
#include "l3_internal.h"
#include "l3_mma.cuh"

namespace l3 {

namespace {

using namespace wmma;

// ---- Phase A ------------------------------------------------------------------------------

constexpr int kAThreads = 256;           // consumer threads (8 warps)
constexpr int kAWarps = kAThreads / 32;
constexpr int kACta = kAThreads + 32;    // + the producer warp
constexpr int kAMaxStages = 6;
constexpr int kAMaxKS = 16;              // 16-wide k-steps of d per warp (d <= 2048)
constexpr int kAMaxKSV = 4;              // of d_v (d_v <= 512)
constexpr int kAMaxDT = 16;              // 16-column tiles of dx per warp
constexpr int kARedLd = 36;
constexpr int kAEld = 40;
constexpr int kASmemLimit = 232448;

// A stage's group (written by the producer before it arms the stage).
struct BMeta {
  int32_t q0, mt, n, c0, c1, pad0, pad1, pad2;
  int32_t tok[kPlanMT];
  float m[kPlanMT], inv_l[kPlanMT], delta[kPlanMT];
};

struct BMisc {
  BMeta meta[kAMaxStages];
  uint64_t meta_full[kAMaxStages];
  uint64_t full[kAMaxStages];
  uint64_t empty[kAMaxStages];
  float red_s[kAWarps][kPlanMT][kARedLd];  // score partials per warp
  float red_p[kAWarps][kPlanMT][kARedLd];  // dp partials per warp
  float e_buf[kPlanMT][kAEld];             // the step's ds per token and row
  int gb, ge, nk;                          // this CTA's groups and their chunks
  int abort;
};

struct BShape {
  int ch, stages, k_bytes, stage_bytes, smem;
};

BShape bwd_shape(int d, int d_v) {
  BShape s{};
  s.ch = 16 * 2 * (d + d_v) <= 49152 ? 16 : 8;
  s.k_bytes = s.ch * 2 * d;
  s.stage_bytes = int(align_up(size_t(s.ch) * 2 * size_t(d + d_v), 1024));
  const int fixed = 1024 + int(align_up(sizeof(BMisc), 128));
  s.stages = (kASmemLimit - fixed) / s.stage_bytes;
  if (s.stages > kAMaxStages) s.stages = kAMaxStages;
  s.smem = fixed + s.stages * s.stage_bytes;
  return s;
}

__device__ __forceinline__ void abar() {
  asm volatile("bar.sync 1, %0;" ::"n"(kAThreads) : "memory");
}

__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(p)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ uint32_t ld_u32(const __nv_bfloat16* p) {
  return __ldg(reinterpret_cast<const unsigned int*>(p));
}

// First group whose cost offset w0 is >= c, by a 32-way search of the producer warp (w0
// increases along the groups; entry NG holds the total).
__device__ int first_group_at(const AttendGroup* groups, int NG, int64_t c, int lane) {
  int lo = 0, hi = NG;  // answer in [lo, hi]
  while (hi - lo > 32) {
    const int step = (hi - lo + 31) / 32;
    const int probe = lo + lane * step;
    const bool below = probe <= hi && groups[probe < hi ? probe : hi].w0 < c;
    const unsigned m = __ballot_sync(0xffffffffu, below && probe < hi);
    // lanes whose probe lies below c form a prefix
    const int nb = __popc(m);
    const int nlo = lo + (nb > 0 ? (nb - 1) * step + 1 : 0);
    const int nhi = lo + nb * step < hi ? lo + nb * step : hi;
    lo = nlo;
    hi = nhi;
  }
  const int probe = lo + lane;
  const bool below = probe < hi && groups[probe].w0 < c;
  return lo + __popc(__ballot_sync(0xffffffffu, below));
}

template <int CH, int KSW, int KSVW, int DTW>
__global__ void __launch_bounds__(kACta, 1)
    attend_bwd_kernel(const __grid_constant__ CUtensorMap mapK,
                      const __grid_constant__ CUtensorMap mapV, const AttendBwdRowsArgs a,
                      const BShape sh) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* ring = base;
  BMisc* ms = reinterpret_cast<BMisc*>(base + sh.stages * sh.stage_bytes);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g8 = lane >> 2, t4 = lane & 3;
  const int b = blockIdx.x;
  const int d = a.d, dv = a.d_v, S = sh.stages;
  const uint32_t ring_s = tc::smem_u32(ring);

  if (warp == kAWarps) {
    // this CTA's groups: those whose cost offset lies in [W b / n, W (b + 1) / n)
    const int NG = a.hdr[kPlanGroups];
    const int64_t W = a.groups[NG].w0;
    const int64_t lo = W * b / gridDim.x, hi = W * (b + 1) / gridDim.x;
    const int gb = first_group_at(a.groups, NG, lo, lane);
    const int ge = first_group_at(a.groups, NG, hi, lane);
    if (lane == 0) {
      ms->gb = gb;
      ms->ge = ge;
      ms->nk = a.groups[ge].c0 - a.groups[gb].c0;
      tc::tma_prefetch_desc(&mapK);
      tc::tma_prefetch_desc(&mapV);
    }
  }
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
  const int nk = ms->nk;
  if (nk <= 0) return;
  volatile int* abort_flag = &ms->abort;

  if (warp == kAWarps) {
    // Producer: per group, an L2 prefetch of its x and da rows (the consumers load their
    // fragments from there when they reach the group), then its chunks' K and V rows.
    const uint32_t tx = uint32_t(CH) * 2u * uint32_t(d + dv);
    int issued = 0;
    bool ok = true;
    for (int g = ms->gb; ok && g < ms->ge; ++g) {
      const AttendGroup G = a.groups[g];
      const int nc = a.groups[g + 1].c0 - G.c0;
      if (nc <= 0) continue;
      float tm = 0.f, tl = 1.f, td = 0.f;
      int tok = 0;
      if (lane < G.mt) {
        tok = G.tok[lane];
        tm = a.ml[2 * int64_t(tok)];
        tl = a.ml[2 * int64_t(tok) + 1];
        td = a.delta[tok];
      }
      if (lane == 0) {
        const int64_t q0 = G.q0;
        prefetch_l2(a.x_sorted + q0 * d, uint32_t(G.mt) * 2u * uint32_t(d));
        prefetch_l2(a.da16 + q0 * dv, uint32_t(G.mt) * 2u * uint32_t(dv));
        prefetch_l2(a.da16_lo + q0 * dv, uint32_t(G.mt) * 2u * uint32_t(dv));
      }
      for (int c = 0; c < nc; ++c, ++issued) {
        const int s = issued % S;
        int oke = 1;
        if (lane == 0)
          oke = tc::mbar_wait_watch(&ms->empty[s], ((issued / S) & 1) ^ 1, abort_flag, a.st,
                                    0x200000)
                    ? 1
                    : 0;
        if (!__shfl_sync(0xffffffffu, oke, 0)) {
          ok = false;
          break;
        }
        BMeta* m = &ms->meta[s];
        if (lane < kPlanMT) {
          m->tok[lane] = tok;
          m->m[lane] = tm;
          m->inv_l[lane] = 1.f / tl;
          m->delta[lane] = td;
        }
        if (lane == 0) {
          m->q0 = G.q0;
          m->mt = G.mt;
          m->n = G.n;
          m->c0 = G.c0;
          m->c1 = G.c0 + nc;
        }
        __syncwarp();
        if (lane == 0) {
          tc::mbar_arrive(&ms->meta_full[s]);
          const int r0 = G.row0 + c * CH;
          const uint32_t st = ring_s + uint32_t(s * sh.stage_bytes);
          tc::mbar_arrive_expect_tx(&ms->full[s], tx);
          tma_load_3d(&mapK, &ms->full[s], st, 0, r0, 0);
          tma_load_3d(&mapV, &ms->full[s], st + uint32_t(sh.k_bytes), 0, r0, 0);
        }
      }
    }
    if (!ok && lane == 0) {
      // Stopped early: let the copies in flight land before the CTA's memory goes away.
      volatile int no_abort = 0;
      for (int j = issued - S > 0 ? issued - S : 0; j < issued; ++j)
        tc::mbar_wait(&ms->full[j % S], (j / S) & 1, &no_abort, a.st, 0x400000, 100000000ull);
    }
    return;
  }

  // ---- consumers ----
  constexpr int KS = KSW ? KSW : kAMaxKS;
  constexpr int KSV = KSVW ? KSVW : kAMaxKSV;
  constexpr int DT = DTW ? DTW : kAMaxDT;
  constexpr int RS = 2 * CH;
  constexpr int MS = RS / 16;
  const int nks = d / 16, nksv = dv / 16, ndt = d / 16;
  float acc[DT][4];
  uint32_t bx[KS][2], bda[KSV][2], bdl[KSV][2];
  int q0 = 0, mt = 0, gn = 0;
  int64_t gc0 = 0, c_next = -1, i0 = 0, i1 = 0;
  bool ok = true, started = false;
  const int64_t cbase = a.groups[ms->gb].c0;

  auto finish = [&]() {  // dx of the group's tokens = the attention term
    const int n0 = 2 * t4, n1 = 2 * t4 + 1;
#pragma unroll
    for (int mi = 0; mi < DT; ++mi) {
      const int mtile = warp + kAWarps * mi;
      if (!DTW && mtile >= ndt) break;
      const int col0 = 16 * mtile + g8, col1 = col0 + 8;
      if (n0 < mt) {
        a.dx[i0 * d + col0] = acc[mi][0];
        a.dx[i0 * d + col1] = acc[mi][2];
      }
      if (n1 < mt) {
        a.dx[i1 * d + col0] = acc[mi][1];
        a.dx[i1 * d + col1] = acc[mi][3];
      }
    }
  };

  for (int k = 0; k < nk;) {
    const int64_t c = cbase + k;
    if (c >= c_next) {  // the chunk opens the next group
      if (started) {
        finish();
        abar();
      }
      const bool got =
          tc::mbar_wait(&ms->meta_full[k % S], (k / S) & 1, abort_flag, a.st, 0x10000);
      const BMeta* m = &ms->meta[k % S];
      if (got) {
        q0 = m->q0;
        mt = m->mt;
        gn = m->n;
        gc0 = m->c0;
        c_next = m->c1;
      } else {
        mt = gn = 0;
        gc0 = c;
        c_next = c + 1;
      }
      started = true;
      i0 = 2 * t4 < mt ? int64_t(m->tok[2 * t4]) : 0;
      i1 = 2 * t4 + 1 < mt ? int64_t(m->tok[2 * t4 + 1]) : 0;
      // x and da fragments of token g8 of the group (zero past mt): B[k][n] = row n at
      // columns 16 s + 2 t4 (+1) and 16 s + 8 + 2 t4 (+1)
#pragma unroll
      for (int i = 0; i < KS; ++i) bx[i][0] = bx[i][1] = 0u;
#pragma unroll
      for (int i = 0; i < KSV; ++i) bda[i][0] = bda[i][1] = bdl[i][0] = bdl[i][1] = 0u;
      if (g8 < mt) {
        const int64_t q = q0 + g8;
        const __nv_bfloat16* xr = a.x_sorted + q * d + 2 * t4;
        const __nv_bfloat16* dr = a.da16 + q * dv + 2 * t4;
        const __nv_bfloat16* dl = a.da16_lo + q * dv + 2 * t4;
#pragma unroll
        for (int i = 0; i < KS; ++i) {
          const int s16 = warp + kAWarps * i;
          if (KSW || s16 < nks) {
            bx[i][0] = ld_u32(xr + 16 * s16);
            bx[i][1] = ld_u32(xr + 16 * s16 + 8);
          }
        }
#pragma unroll
        for (int i = 0; i < KSV; ++i) {
          const int s16 = warp + kAWarps * i;
          if (KSVW || s16 < nksv) {
            bda[i][0] = ld_u32(dr + 16 * s16);
            bda[i][1] = ld_u32(dr + 16 * s16 + 8);
            bdl[i][0] = ld_u32(dl + 16 * s16);
            bdl[i][1] = ld_u32(dl + 16 * s16 + 8);
          }
        }
      }
#pragma unroll
      for (int mi = 0; mi < DT; ++mi) acc[mi][0] = acc[mi][1] = acc[mi][2] = acc[mi][3] = 0.f;
    }
    const int j0 = int(c - gc0);
    const int nr0 = gn - j0 * CH < CH ? gn - j0 * CH : CH;
    const bool pair = k + 1 < nk && c + 1 < c_next;
    const int nr1 = pair ? (gn - (j0 + 1) * CH < CH ? gn - (j0 + 1) * CH : CH) : 0;
    tc::mbar_wait(&ms->full[k % S], (k / S) & 1, abort_flag, a.st, 0x10000);
    if (pair) tc::mbar_wait(&ms->full[(k + 1) % S], ((k + 1) / S) & 1, abort_flag, a.st, 0x10000);
    abar();
    if (*abort_flag) {
      ok = false;
      break;
    }
    const uint32_t st0 = ring_s + uint32_t((k % S) * sh.stage_bytes);
    const uint32_t st1 = pair ? ring_s + uint32_t(((k + 1) % S) * sh.stage_bytes) : st0;
    auto stage_of = [&](int R) { return R < CH ? st0 : st1; };
    const BMeta* m = &ms->meta[k % S];

    // scores s = K x and dp = V da for the step's rows: warps split d and d_v
    {
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
      float sc[MS][4][4], dq[MS][2][4];
#pragma unroll
      for (int t = 0; t < MS; ++t) {
#pragma unroll
        for (int u = 0; u < 4; ++u) sc[t][u][0] = sc[t][u][1] = sc[t][u][2] = sc[t][u][3] = 0.f;
#pragma unroll
        for (int u = 0; u < 2; ++u) dq[t][u][0] = dq[t][u][1] = dq[t][u][2] = dq[t][u][3] = 0.f;
      }
#pragma unroll
      for (int i = 0; i < KS; ++i) {
        const int s16 = warp + kAWarps * i;
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
      for (int i = 0; i < KSV; ++i) {
        const int s16 = warp + kAWarps * i;
        if (KSVW || s16 < nksv) {
#pragma unroll
          for (int t = 0; t < MS; ++t) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4(abase[t] + uint32_t(sh.k_bytes) + sw128(CH, arow[t], s16 * 16 + akof), a0, a1,
                    a2, a3);
            mma16(dq[t][0], a0, a1, a2, a3, bda[i][0], bda[i][1]);
            mma16(dq[t][1], a0, a1, a2, a3, bdl[i][0], bdl[i][1]);
          }
        }
      }
#pragma unroll
      for (int t = 0; t < MS; ++t) {
        float r4[4], p4[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          r4[i] = (sc[t][0][i] + sc[t][1][i]) + (sc[t][2][i] + sc[t][3][i]);
          p4[i] = dq[t][0][i] + dq[t][1][i];
        }
        ms->red_s[warp][2 * t4][16 * t + g8] = r4[0];
        ms->red_s[warp][2 * t4 + 1][16 * t + g8] = r4[1];
        ms->red_s[warp][2 * t4][16 * t + g8 + 8] = r4[2];
        ms->red_s[warp][2 * t4 + 1][16 * t + g8 + 8] = r4[3];
        ms->red_p[warp][2 * t4][16 * t + g8] = p4[0];
        ms->red_p[warp][2 * t4 + 1][16 * t + g8] = p4[1];
        ms->red_p[warp][2 * t4][16 * t + g8 + 8] = p4[2];
        ms->red_p[warp][2 * t4 + 1][16 * t + g8 + 8] = p4[3];
      }
    }
    abar();
    // p and ds per token and row (fp32), stored by sorted position and row within the id
    if (tid < RS * kPlanMT) {
      const int j = tid / RS, r = tid % RS;
      const bool rv = r < CH ? r < nr0 : r - CH < nr1;
      float s = 0.f, dp = 0.f;
#pragma unroll
      for (int w = 0; w < kAWarps; ++w) {
        s += ms->red_s[w][j][r];
        dp += ms->red_p[w][j][r];
      }
      const bool valid = rv && j < mt;
      const float p = valid ? expf(s - m->m[j]) * m->inv_l[j] : 0.f;
      const float ds = valid ? p * (dp - m->delta[j]) : 0.f;
      if (valid) {
        const int64_t o = int64_t(q0 + j) * a.k_max + j0 * CH + r;
        a.p_buf[o] = p;
        a.ds_buf[o] = ds;
      }
      ms->e_buf[j][r] = ds;
    }
    abar();
    // dxᵀ += Kᵀ dsᵀ over the step's rows (K columns as M, ds as bf16 hi + lo)
    {
      uint32_t bh[MS][2], bl[MS][2];
#pragma unroll
      for (int t = 0; t < MS; ++t) {
        const float2 e0 = *reinterpret_cast<const float2*>(&ms->e_buf[g8][16 * t + 2 * t4]);
        const float2 e1 = *reinterpret_cast<const float2*>(&ms->e_buf[g8][16 * t + 2 * t4 + 8]);
        split_pair(e0.x, e0.y, bh[t][0], bl[t][0]);
        split_pair(e1.x, e1.y, bh[t][1], bl[t][1]);
      }
      const int vl = (lane & 7) + (lane >> 4) * 8;
      const int vcol = ((lane >> 3) & 1) * 8;
#pragma unroll
      for (int t = 0; t < MS; ++t) {
        const int R = 16 * t + vl;
        const uint32_t kb = stage_of(R);
        const int krow = R % CH;
#pragma unroll
        for (int mi = 0; mi < DT; ++mi) {
          const int mtile = warp + kAWarps * mi;
          if (DTW || mtile < ndt) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4_t(kb + sw128(CH, krow, 16 * mtile + vcol), a0, a1, a2, a3);
            mma16(acc[mi], a0, a1, a2, a3, bh[t][0], bh[t][1]);
            mma16(acc[mi], a0, a1, a2, a3, bl[t][0], bl[t][1]);
          }
        }
      }
    }
    abar();
    if (tid == 0) {
      tc::mbar_arrive(&ms->empty[k % S]);
      if (pair) tc::mbar_arrive(&ms->empty[(k + 1) % S]);
    }
    k += pair ? 2 : 1;
  }
  if (ok && started) finish();
}

// ---- Phase B ------------------------------------------------------------------------------

constexpr int kBRows = 64;   // table rows per unit
constexpr int kBCols = 256;  // output columns per unit
constexpr int kBTok = 32;    // tokens per step
constexpr int kBThreads = 256;
constexpr int kYld = kBCols + 8;  // bf16 row stride of the token tile (ldmatrix rows 528 B apart)
constexpr int kWld = kBTok + 8;   // bf16 row stride of the weight tiles (80 B apart)
constexpr int kBUnitFixed = 2;    // cost of a unit's setup and stores, in steps

struct SegSmem {
  __nv_bfloat16 ys[2][kBTok][kYld];   // Y rows of the step's tokens, double-buffered
  __nv_bfloat16 wh[2][kBRows][kWld];  // W transposed (row, token), bf16 hi
  __nv_bfloat16 wl[2][kBRows][kWld];  // and lo
};

__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool full) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(tc::smem_u32(dst)),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(full ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}

// One unit: segment s, rows [r0, r0 + 64) of its id, columns [col0, col0 + 256) of dK
// (part 0) or dV (part 1). D[row][col] = sum_q W[q][row] Y[q][col] over the segment's
// sorted positions q, Y = x (dK) or da (dV), W = ds (dK) or p (dV). A step takes 32 tokens:
// Y by cp.async into one of two buffers, W through registers (split into bf16 hi + lo and
// transposed into one of two buffers), so one barrier a step suffices. Warp w owns columns
// [32 w, 32 w + 32) of the unit and all 64 rows.
__global__ void __launch_bounds__(kBThreads, 2) seg_rows_kernel(const SegRowsArgs a) {
  extern __shared__ __align__(128) unsigned char seg_smem_raw[];
  SegSmem& sm = *reinterpret_cast<SegSmem*>(seg_smem_raw);
  __shared__ int s_first[2];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g8 = lane >> 2, t4 = lane & 3;
  const int S = *a.n_seg;
  const int ncb_k = (a.d + kBCols - 1) / kBCols, ncb_v = (a.d_v + kBCols - 1) / kBCols;
  const int ncb = ncb_k + ncb_v;
  // This CTA's units: those whose cost interval starts in [C b / G, C (b + 1) / G) of the
  // total cost C (a unit of segment s costs ceil(tokens / 32) + kBUnitFixed). The first is
  // found by one binary search; the rest follow in order.
  const int64_t C = a.seg_cost0[S];
  const int64_t clo = C * blockIdx.x / gridDim.x, chi = C * (blockIdx.x + 1) / gridDim.x;
  if (tid == 0) {
    int lo = 0, hi = S;  // first segment whose cost interval ends past clo
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (a.seg_cost0[mid + 1] <= clo)
        lo = mid + 1;
      else
        hi = mid;
    }
    s_first[0] = lo;
    int k0 = 0;
    if (lo < S) {
      const int64_t uc = (a.seg_cost0[lo + 1] - a.seg_cost0[lo]) /
                         (a.seg_unit0[lo + 1] - a.seg_unit0[lo]);  // cost of each unit
      k0 = int((clo - a.seg_cost0[lo] + uc - 1) / uc);  // first unit starting at or after clo
    }
    s_first[1] = k0;
  }
  __syncthreads();
  int s = s_first[0];
  int64_t local = s_first[1];
  // W loads: row wr of the unit, tokens 8 wg .. 8 wg + 7 of the step
  const int wr = tid & 63, wg = tid >> 6;
  // the current segment's description, loaded once per segment (its loads form a chain of
  // dependent global round trips: seg_start -> sorted key -> offsets)
  int cur = -1, qs = 0, qe = 0, rbase = 0, n = 0;
  int64_t nu = 0, uc = 0, cost_s = 0, srow0 = 0;
  while (s < S) {
    if (s != cur) {
      nu = a.seg_unit0[s + 1] - a.seg_unit0[s];
      cost_s = a.seg_cost0[s];
      uc = nu > 0 ? (a.seg_cost0[s + 1] - cost_s) / nu : 0;
      qs = a.seg_start[s];
      qe = a.seg_start[s + 1];
      srow0 = a.seg_row0[s];
      const int t = int(a.sorted_keys[qs] >> 32);
      rbase = a.offs[t];
      n = a.offs[t + 1] - rbase;
      cur = s;
    }
    if (local >= nu) {
      ++s;
      local = 0;
      continue;
    }
    if (cost_s + local * uc >= chi) break;
    const int rb = int(local / ncb), cb = int(local % ncb);
    ++local;
    const int part = cb < ncb_k ? 0 : 1;
    const int width = part ? a.d_v : a.d;
    const int col0 = (part ? cb - ncb_k : cb) * kBCols;
    const int r0 = rb * kBRows;
    const int64_t orow0 = srow0 + r0;  // output row of row r0
    const __nv_bfloat16* Y = part ? a.da_sorted : a.x_sorted;
    const float* Wsrc = part ? a.p_buf : a.ds_buf;
    float* out = part ? a.dV_rows : a.dK_rows;
    if (part == 0 && cb == 0)
      for (int r = tid; r < kBRows && r0 + r < n; r += kBThreads) {
        if (orow0 + r < a.max_rows)
          a.row_index[orow0 + r] = rbase + r0 + r;
        else
          atomicOr(&a.st->capacity, 1);
      }
    const bool wcols = col0 + 32 * warp < width;  // the warp's 32 columns exist (width % 64 == 0)
    float acc[4][4][4];
#pragma unroll
    for (int mt = 0; mt < 4; ++mt)
#pragma unroll
      for (int nt = 0; nt < 4; ++nt) acc[mt][nt][0] = acc[mt][nt][1] = acc[mt][nt][2] = acc[mt][nt][3] = 0.f;
    auto load_y = [&](int q, int buf) {  // tokens q .. q + 31: 1024 pieces of 16 bytes
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int pc = tid + kBThreads * j;
        const int tk = pc >> 5, cp = (pc & 31) * 8;
        const bool ok = q + tk < qe && col0 + cp < width;
        const __nv_bfloat16* src = ok ? Y + int64_t(q + tk) * width + col0 + cp : Y;
        cp_async16(&sm.ys[buf][tk][cp], src, ok);
      }
      cp_async_commit();
    };
    float wv[8];
    auto load_w = [&](int q) {
      const bool rv = r0 + wr < n;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int qq = q + 8 * wg + j;
        wv[j] = (rv && qq < qe) ? __ldg(Wsrc + int64_t(qq) * a.k_max + r0 + wr) : 0.f;
      }
    };
    auto store_w = [&](int buf) {
      uint32_t h[4], l[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) split_pair(wv[2 * j], wv[2 * j + 1], h[j], l[j]);
      *reinterpret_cast<uint4*>(&sm.wh[buf][wr][8 * wg]) = make_uint4(h[0], h[1], h[2], h[3]);
      *reinterpret_cast<uint4*>(&sm.wl[buf][wr][8 * wg]) = make_uint4(l[0], l[1], l[2], l[3]);
    };
    load_y(qs, 0);
    load_w(qs);
    store_w(0);
    int buf = 0;
    for (int q = qs; q < qe; q += kBTok, buf ^= 1) {
      cp_async_wait_all();
      __syncthreads();  // step q's tiles are in place; every warp is past the previous step
      const bool more = q + kBTok < qe;
      if (more) {
        load_y(q + kBTok, buf ^ 1);
        load_w(q + kBTok);
      }
      if (wcols) {
#pragma unroll
        for (int ks = 0; ks < kBTok / 16; ++ks) {
          uint32_t b[4][2];
          const int yt = 16 * ks + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
          for (int pr = 0; pr < 2; ++pr) {
            const int yc = 32 * warp + 16 * pr + ((lane >> 4) & 1) * 8;
            ldsm_x4_t(tc::smem_u32(&sm.ys[buf][yt][yc]), b[2 * pr][0], b[2 * pr][1],
                      b[2 * pr + 1][0], b[2 * pr + 1][1]);
          }
          const int ar = lane & 15, ak = 16 * ks + (lane >> 4) * 8;
#pragma unroll
          for (int mt = 0; mt < 4; ++mt) {
            uint32_t h0, h1, h2, h3, l0, l1, l2, l3;
            ldsm_x4(tc::smem_u32(&sm.wh[buf][16 * mt + ar][ak]), h0, h1, h2, h3);
            ldsm_x4(tc::smem_u32(&sm.wl[buf][16 * mt + ar][ak]), l0, l1, l2, l3);
#pragma unroll
            for (int nt = 0; nt < 4; ++nt) {
              mma16(acc[mt][nt], h0, h1, h2, h3, b[nt][0], b[nt][1]);
              mma16(acc[mt][nt], l0, l1, l2, l3, b[nt][0], b[nt][1]);
            }
          }
        }
      }
      if (more) store_w(buf ^ 1);
    }
    __syncthreads();  // the buffers are free for the next unit
    // D[row][col]: lane (g8, t4) holds rows 16 mt + g8 (+ 8), columns 8 nt + 2 t4 (+ 1)
    if (wcols) {
#pragma unroll
      for (int mt = 0; mt < 4; ++mt)
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          const int row = 16 * mt + g8 + 8 * hr;
          if (r0 + row < n && orow0 + row < a.max_rows) {
            float* o = out + (orow0 + row) * width + col0 + 32 * warp + 2 * t4;
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
              *reinterpret_cast<float2*>(o + 8 * nt) =
                  make_float2(acc[mt][nt][2 * hr], acc[mt][nt][2 * hr + 1]);
          }
        }
    }
  }
}

// ---- small kernels ------------------------------------------------------------------------

// LayerNorm of the fp32 rows U = W_up a (one warp per row): mu, rstd (biased variance, eps)
// and h = (U - mu) rstd, written over U in fp32 and as bf16 to h16. Recomputed here rather
// than taken from the forward, whose statistics are those of U rounded to bf16: when
// |mean u| is large against its spread, that rounding moves h by far more than 2^-9.
__global__ void bwd_ln_kernel(float* __restrict__ U, int64_t T, int d, float eps,
                              __nv_bfloat16* __restrict__ h16, float* __restrict__ rstd_out) {
  const int lane = threadIdx.x & 31;
  const int64_t row = int64_t(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (row >= T) return;
  float* u = U + row * d;
  float s = 0.f;
  for (int c = lane; c < d; c += 32) s += u[c];
  const float mean = warp_sum(s) / float(d);
  float m2 = 0.f;
  for (int c = lane; c < d; c += 32) {
    const float e = u[c] - mean;
    m2 = fmaf(e, e, m2);
  }
  const float rstd = 1.f / sqrtf(warp_sum(m2) / float(d) + eps);
  for (int c = lane; c < d; c += 32) {
    const float h = (u[c] - mean) * rstd;
    u[c] = h;
    h16[row * d + c] = __float2bfloat16_rn(h);
  }
  if (lane == 0) rstd_out[row] = rstd;
}

// du = rstd (dh - mean(dh) - h mean(dh h)) per row (one warp per row), fp32, written as
// bf16 hi + lo (du_hi = bf16(du), du_lo = bf16(du - du_hi)).
__global__ void ln_bwd_split_kernel(const float* __restrict__ dh, const float* __restrict__ H,
                                    const float* __restrict__ rstd, int64_t T, int d,
                                    __nv_bfloat16* __restrict__ du_hi,
                                    __nv_bfloat16* __restrict__ du_lo) {
  const int lane = threadIdx.x & 31;
  const int64_t row = int64_t(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (row >= T) return;
  const float* g = dh + row * d;
  const float* h = H + row * d;
  float s1 = 0.f, s2 = 0.f;
  for (int c = lane; c < d; c += 32) {
    s1 += g[c];
    s2 = fmaf(g[c], h[c], s2);
  }
  const float mg = warp_sum(s1) / float(d), mgh = warp_sum(s2) / float(d);
  const float r = rstd[row];
  for (int c = lane; c < d; c += 32) {
    const float du = r * (g[c] - mg - h[c] * mgh);
    const __nv_bfloat16 hi = __float2bfloat16_rn(du);
    du_hi[row * d + c] = hi;
    du_lo[row * d + c] = __float2bfloat16_rn(du - __bfloat162float(hi));
  }
}

// fp32 -> bf16 hi + lo, n elements.
__global__ void split_hilo_kernel(const float* __restrict__ src, int64_t n,
                                  __nv_bfloat16* __restrict__ hi, __nv_bfloat16* __restrict__ lo) {
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += int64_t(gridDim.x) * blockDim.x) {
    const float v = src[i];
    const __nv_bfloat16 h = __float2bfloat16_rn(v);
    hi[i] = h;
    lo[i] = __float2bfloat16_rn(v - __bfloat162float(h));
  }
}

// Per sorted position q (one warp): the x row and da as bf16 hi + lo in sorted order, and
// δ_i = a_i · da_i for the token i = perm(q).
__global__ void bwd_prep_kernel(const uint64_t* __restrict__ keys, int64_t T,
                                const __nv_bfloat16* __restrict__ x, const float* __restrict__ a,
                                const float* __restrict__ da, int d, int d_v,
                                __nv_bfloat16* __restrict__ x_sorted,
                                __nv_bfloat16* __restrict__ da16,
                                __nv_bfloat16* __restrict__ da16_lo, float* __restrict__ delta) {
  const int lane = threadIdx.x & 31;
  const int64_t q = int64_t(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (q >= T) return;
  const int64_t i = int64_t(uint32_t(keys[q]));
  const uint4* xs = reinterpret_cast<const uint4*>(x + i * d);
  uint4* xd = reinterpret_cast<uint4*>(x_sorted + q * d);
  for (int c = lane; c < d / 8; c += 32) xd[c] = __ldg(xs + c);
  float dot = 0.f;
  for (int c = lane; c < d_v; c += 32) {
    const float g = da[i * d_v + c];
    dot = fmaf(a[i * d_v + c], g, dot);
    const __nv_bfloat16 gb = __float2bfloat16_rn(g);
    da16[q * d_v + c] = gb;
    da16_lo[q * d_v + c] = __float2bfloat16_rn(g - __bfloat162float(gb));
  }
  dot = warp_sum(dot);
  if (lane == 0) delta[i] = dot;
}

// Output rows and Phase B units of every segment: exclusive sums of n_t and of the units
// (64-row blocks x column blocks) over the segments, in one CTA of 1024 threads.
__global__ void __launch_bounds__(1024) row_plan_kernel(const uint64_t* __restrict__ keys,
                                                        const int32_t* __restrict__ seg_start,
                                                        const int32_t* __restrict__ n_seg,
                                                        const int32_t* __restrict__ offs, int ncb,
                                                        int32_t* seg_row0, int32_t* seg_unit0,
                                                        int64_t* seg_cost0, int32_t* n_rows,
                                                        int64_t max_rows, DevStatus* st) {
  __shared__ int2 wt[32];
  __shared__ int2 tot;
  __shared__ long long wc[32];
  __shared__ long long totc;
  const int S = *n_seg;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int64_t carry_r = 0, carry_u = 0, carry_c = 0;
  for (int base = 0; base < S; base += blockDim.x) {
    const int s = base + threadIdx.x;
    int nr = 0, nu = 0;
    long long nc = 0;
    if (s < S) {
      const int q0 = seg_start[s];
      const int t = int(keys[q0] >> 32);
      nr = offs[t + 1] - offs[t];
      nu = (nr + kBRows - 1) / kBRows * ncb;
      nc = (long long)nu * ((seg_start[s + 1] - q0 + kBTok - 1) / kBTok + kBUnitFixed);
    }
    long long inc = nc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long u = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += u;
    }
    int2 incl = make_int2(nr, nu);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int ux = __shfl_up_sync(0xffffffffu, incl.x, o);
      const int uy = __shfl_up_sync(0xffffffffu, incl.y, o);
      if (lane >= o) {
        incl.x += ux;
        incl.y += uy;
      }
    }
    if (lane == 31) {
      wt[wid] = incl;
      wc[wid] = inc;
    }
    __syncthreads();
    if (wid == 0) {
      const long long wcv = wc[lane];
      long long wci = wcv;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const long long u = __shfl_up_sync(0xffffffffu, wci, o);
        if (lane >= o) wci += u;
      }
      wc[lane] = wci - wcv;
      if (lane == 31) totc = wci;
      const int2 w = wt[lane];
      int2 wi = w;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int ux = __shfl_up_sync(0xffffffffu, wi.x, o);
        const int uy = __shfl_up_sync(0xffffffffu, wi.y, o);
        if (lane >= o) {
          wi.x += ux;
          wi.y += uy;
        }
      }
      wt[lane] = make_int2(wi.x - w.x, wi.y - w.y);
      if (lane == 31) tot = wi;
    }
    __syncthreads();
    if (s < S) {
      seg_row0[s] = int32_t(carry_r + wt[wid].x + incl.x - nr);
      seg_unit0[s] = int32_t(carry_u + wt[wid].y + incl.y - nu);
      seg_cost0[s] = carry_c + wc[wid] + inc - nc;
    }
    carry_r += tot.x;
    carry_u += tot.y;
    carry_c += totc;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    seg_unit0[S] = int32_t(carry_u);
    seg_cost0[S] = carry_c;
    *n_rows = int32_t(carry_r);
    if (carry_r > max_rows) atomicOr(&st->capacity, 1);
  }
}

}  // namespace

int attend_bwd_rows_per_chunk(int d, int d_v) { return bwd_shape(d, d_v).ch; }

template <int CH, int KSW, int KSVW, int DTW>
cudaError_t launch_bwd_a(const AttendBwdRowsArgs& a, const BShape& sh, cudaStream_t stream) {
  CUtensorMap mk, mv;
  if (!make_row_block_map(&mk, a.K, a.v, a.d, CH) || !make_row_block_map(&mv, a.V, a.v, a.d_v, CH))
    return cudaErrorInvalidValue;
  const cudaError_t attr = ensure_smem_attr(attend_bwd_kernel<CH, KSW, KSVW, DTW>, kASmemLimit);
  if (attr != cudaSuccess) return attr;
  attend_bwd_kernel<CH, KSW, KSVW, DTW><<<a.n_cta, kACta, sh.smem, stream>>>(mk, mv, a, sh);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_attend_bwd_rows(const AttendBwdRowsArgs& a, cudaStream_t stream) {
  const BShape sh = bwd_shape(a.d, a.d_v);
  if (sh.stages < 2 || sh.smem > kASmemLimit || sh.ch != a.ch || a.d % 64 || a.d_v % 64 ||
      a.d > 16 * kAWarps * kAMaxKS || a.d_v > 16 * kAWarps * kAMaxKSV ||
      (reinterpret_cast<uintptr_t>(a.x_sorted) & 15) ||
      (reinterpret_cast<uintptr_t>(a.da16) & 15) || (reinterpret_cast<uintptr_t>(a.da16_lo) & 15))
    return cudaErrorInvalidValue;
  if (sh.ch == 8 && a.d == 2048 && a.d_v == 512) return launch_bwd_a<8, 16, 4, 16>(a, sh, stream);
  if (sh.ch == 16 && a.d == 1024 && a.d_v == 256) return launch_bwd_a<16, 8, 2, 8>(a, sh, stream);
  return sh.ch == 16 ? launch_bwd_a<16, 0, 0, 0>(a, sh, stream)
                     : launch_bwd_a<8, 0, 0, 0>(a, sh, stream);
}

cudaError_t launch_seg_rows(const SegRowsArgs& a, cudaStream_t stream) {
  if (a.d % 64 || a.d_v % 64) return cudaErrorInvalidValue;
  const cudaError_t attr = ensure_smem_attr(seg_rows_kernel, int(sizeof(SegSmem)));
  if (attr != cudaSuccess) return attr;
  seg_rows_kernel<<<unsigned(device_sm_count() * 2), kBThreads, sizeof(SegSmem), stream>>>(a);
  count_launch();
  return cudaGetLastError();
}

int seg_rows_col_blocks(int d, int d_v) {
  return (d + kBCols - 1) / kBCols + (d_v + kBCols - 1) / kBCols;
}

cudaError_t launch_row_plan(const uint64_t* keys, const int32_t* seg_start, const int32_t* n_seg,
                            const int32_t* offs, int d, int d_v, int32_t* seg_row0,
                            int32_t* seg_unit0, int64_t* seg_cost0, int32_t* n_rows,
                            int64_t max_rows, DevStatus* st, cudaStream_t stream) {
  row_plan_kernel<<<1, 1024, 0, stream>>>(keys, seg_start, n_seg, offs,
                                          seg_rows_col_blocks(d, d_v), seg_row0, seg_unit0,
                                          seg_cost0, n_rows, max_rows, st);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_bwd_small(const BwdSmallArgs& a, cudaStream_t stream) {
  if (a.T <= 0) return cudaSuccess;
  const unsigned rows_grid = unsigned((a.T + 7) / 8);
  if (a.stage == 0) {
    bwd_ln_kernel<<<rows_grid, 256, 0, stream>>>(a.U32, a.T, a.d, a.eps, a.h16, a.rstd_out);
  } else if (a.stage == 1) {
    ln_bwd_split_kernel<<<rows_grid, 256, 0, stream>>>(a.dh, a.U32, a.rstd_out, a.T, a.d,
                                                       a.du, a.du_lo);
  } else if (a.stage == 2) {
    bwd_prep_kernel<<<rows_grid, 256, 0, stream>>>(a.keys, a.T, a.x, a.a, a.da, a.d, a.d_v,
                                                   a.x_sorted, a.da16, a.da16_lo, a.delta);
  } else {
    const int64_t n = a.T * a.d_v;
    int64_t g = (n + 255) / 256;
    if (g > int64_t(device_sm_count()) * 16) g = int64_t(device_sm_count()) * 16;
    split_hilo_kernel<<<unsigned(g), 256, 0, stream>>>(a.a, n, a.a_hi, a.a_lo);
  }
  count_launch();
  return cudaGetLastError();
}

}  // namespace l3
