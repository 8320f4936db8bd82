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
// whole groups per CTA (cut by chunk count). Per group it streams the id's rows (TMA, as
// the forward's split-row kernel) and computes the scores and dp with warp MMAs (x and da
// fragments from shared-memory slots the producer fills; da as bf16 hi + lo, so that dp and
// δ = a · da agree to about 2^-17 and ds = p (dp - δ) keeps its digits), p and ds in fp32
// (stored per sorted position and row), and dx with a warp MMA over Kᵀ with ds as bf16
// hi + lo; dx is added to the direct term the GEMMs left there. No group is split, so no
// merge is needed.
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
constexpr int kAMaxStages = 4;
constexpr int kASlots = 2;               // groups whose x and da rows are in shared memory
constexpr int kAMaxKS = 16;              // 16-wide k-steps of d per warp (d <= 2048)
constexpr int kAMaxKSV = 4;              // of d_v (d_v <= 512)
constexpr int kAMaxDT = 16;              // 16-column tiles of dx per warp
constexpr int kARedLd = 36;
constexpr int kAEld = 40;
constexpr int kASmemLimit = 232448;

// A stage's group (written by the producer before it arms the stage).
struct BMeta {
  int32_t q0, mt, n, c0, c1, slot, pad0, pad1;
  int32_t tok[kPlanMT];
  float m[kPlanMT], inv_l[kPlanMT], delta[kPlanMT];
};

struct BMisc {
  BMeta meta[kAMaxStages];
  uint64_t meta_full[kAMaxStages];
  uint64_t full[kAMaxStages];
  uint64_t empty[kAMaxStages];
  uint64_t x_full[kASlots];
  uint64_t x_empty[kASlots];
  float red_s[kAWarps][kPlanMT][kARedLd];  // score partials per warp
  float red_p[kAWarps][kPlanMT][kARedLd];  // dp partials per warp
  float e_buf[kPlanMT][kAEld];             // the step's ds per token and row
  int gb, ge, nk;                          // this CTA's groups and their chunks
  int abort;
};

struct BShape {
  int ch, stages, k_bytes, stage_bytes, x_row, da_row, slot_bytes, smem;
};

BShape bwd_shape(int d, int d_v) {
  BShape s{};
  s.ch = 16 * 2 * (d + d_v) <= 49152 ? 16 : 8;
  s.k_bytes = s.ch * 2 * d;
  s.stage_bytes = int(align_up(size_t(s.ch) * 2 * size_t(d + d_v), 1024));
  s.x_row = 2 * d + 16;
  s.da_row = 2 * d_v + 16;
  s.slot_bytes = int(align_up(size_t(kPlanMT) * size_t(s.x_row + 2 * s.da_row), 128));
  const int fixed = 1024 + int(align_up(sizeof(BMisc), 128)) + kASlots * s.slot_bytes;
  s.stages = (kASmemLimit - fixed) / s.stage_bytes;
  if (s.stages > kAMaxStages) s.stages = kAMaxStages;
  s.smem = fixed + s.stages * s.stage_bytes;
  return s;
}

__device__ __forceinline__ void abar() {
  asm volatile("bar.sync 1, %0;" ::"n"(kAThreads) : "memory");
}

__device__ __forceinline__ void bulk_copy(uint32_t dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(tc::smem_u32(bar))
      : "memory");
}

// First group whose first chunk is >= c, by a 32-way search of the producer warp (groups
// are ordered by first chunk; entry NG holds the total).
__device__ int first_group_at(const AttendGroup* groups, int NG, int64_t c, int lane) {
  int lo = 0, hi = NG;  // answer in [lo, hi]
  while (hi - lo > 32) {
    const int step = (hi - lo + 31) / 32;
    const int probe = lo + lane * step;
    const bool below = probe <= hi && groups[probe < hi ? probe : hi].c0 < c;
    const unsigned m = __ballot_sync(0xffffffffu, below && probe < hi);
    // lanes whose probe lies below c form a prefix
    const int nb = __popc(m);
    const int nlo = lo + (nb > 0 ? (nb - 1) * step + 1 : 0);
    const int nhi = lo + nb * step < hi ? lo + nb * step : hi;
    lo = nlo;
    hi = nhi;
  }
  const int probe = lo + lane;
  const bool below = probe < hi && groups[probe].c0 < c;
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
  unsigned char* slots = base + sh.stages * sh.stage_bytes;
  BMisc* ms = reinterpret_cast<BMisc*>(slots + kASlots * sh.slot_bytes);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g8 = lane >> 2, t4 = lane & 3;
  const int b = blockIdx.x;
  const int d = a.d, dv = a.d_v, S = sh.stages;
  const uint32_t ring_s = tc::smem_u32(ring), slots_s = tc::smem_u32(slots);

  if (warp == kAWarps) {
    // this CTA's groups: those whose first chunk lies in [C b / n, C (b + 1) / n)
    const int NG = a.hdr[kPlanGroups];
    const int64_t C = a.hdr[kPlanChunks];
    const int64_t lo = C * b / gridDim.x, hi = C * (b + 1) / gridDim.x;
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
    for (int s = 0; s < kASlots; ++s) {
      tc::mbar_init(&ms->x_full[s], 1);
      tc::mbar_init(&ms->x_empty[s], 1);
    }
    ms->abort = 0;
    tc::fence_barrier_init();
  }
  __syncthreads();
  const int nk = ms->nk;
  if (nk <= 0) return;
  volatile int* abort_flag = &ms->abort;

  if (warp == kAWarps) {
    // Producer: per group, its x and da rows into a slot, then its chunks' K and V rows.
    const uint32_t tx = uint32_t(CH) * 2u * uint32_t(d + dv);
    int issued = 0, ns = 0;
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
      const int xsl = ns % kASlots;
      int okx = 1;
      if (lane == 0) {
        okx = tc::mbar_wait_watch(&ms->x_empty[xsl], ((ns / kASlots) & 1) ^ 1, abort_flag, a.st,
                                  0x100000)
                  ? 1
                  : 0;
        if (okx)
          tc::mbar_arrive_expect_tx(&ms->x_full[xsl],
                                    uint32_t(G.mt) * 2u * uint32_t(d + 2 * dv));
      }
      if (!__shfl_sync(0xffffffffu, okx, 0)) {
        ok = false;
        break;
      }
      __syncwarp();
      if (lane < G.mt) {
        const uint32_t sb = slots_s + uint32_t(xsl * sh.slot_bytes);
        bulk_copy(sb + uint32_t(lane * sh.x_row), a.x + int64_t(tok) * d, uint32_t(2 * d),
                  &ms->x_full[xsl]);
        bulk_copy(sb + uint32_t(kPlanMT * sh.x_row + lane * sh.da_row), a.da16 + int64_t(tok) * dv,
                  uint32_t(2 * dv), &ms->x_full[xsl]);
        bulk_copy(sb + uint32_t(kPlanMT * (sh.x_row + sh.da_row) + lane * sh.da_row),
                  a.da16_lo + int64_t(tok) * dv, uint32_t(2 * dv), &ms->x_full[xsl]);
      }
      ++ns;
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
          m->slot = xsl;
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
      for (int j = ns - kASlots > 0 ? ns - kASlots : 0; j < ns; ++j)
        tc::mbar_wait(&ms->x_full[j % kASlots], (j / kASlots) & 1, &no_abort, a.st, 0x400000,
                      100000000ull);
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
  int q0 = 0, mt = 0, gn = 0, ngc = 0, x_release = -1;
  int64_t gc0 = 0, c_next = -1, i0 = 0, i1 = 0;
  bool ok = true, started = false;
  const int64_t cbase = a.groups[ms->gb].c0;

  auto finish = [&]() {  // dx of the group's tokens += the attention term
    const int n0 = 2 * t4, n1 = 2 * t4 + 1;
#pragma unroll
    for (int mi = 0; mi < DT; ++mi) {
      const int mtile = warp + kAWarps * mi;
      if (!DTW && mtile >= ndt) break;
      const int col0 = 16 * mtile + g8, col1 = col0 + 8;
      if (n0 < mt) {
        a.dx[i0 * d + col0] += acc[mi][0];
        a.dx[i0 * d + col1] += acc[mi][2];
      }
      if (n1 < mt) {
        a.dx[i1 * d + col0] += acc[mi][1];
        a.dx[i1 * d + col1] += acc[mi][3];
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
      const int slot = got ? m->slot : 0;
      // x and da fragments from the slot (token slots past mt zeroed)
#pragma unroll
      for (int i = 0; i < KS; ++i) bx[i][0] = bx[i][1] = 0u;
#pragma unroll
      for (int i = 0; i < KSV; ++i) bda[i][0] = bda[i][1] = bdl[i][0] = bdl[i][1] = 0u;
      if (got &&
          tc::mbar_wait(&ms->x_full[slot], (ngc / kASlots) & 1, abort_flag, a.st, 0x20000)) {
        const uint32_t sb = slots_s + uint32_t(slot * sh.slot_bytes);
        const uint32_t xr = sb + uint32_t((lane & 7) * sh.x_row + ((lane >> 3) & 1) * 16);
        const uint32_t dr =
            sb + uint32_t(kPlanMT * sh.x_row + (lane & 7) * sh.da_row + ((lane >> 3) & 1) * 16);
        const uint32_t dl = dr + uint32_t(kPlanMT * sh.da_row);
#pragma unroll
        for (int i = 0; i < KS; ++i) {
          const int s16 = warp + kAWarps * i;
          if (KSW || s16 < nks) ldsm_x2(xr + uint32_t(s16 * 32), bx[i][0], bx[i][1]);
        }
#pragma unroll
        for (int i = 0; i < KSV; ++i) {
          const int s16 = warp + kAWarps * i;
          if (KSVW || s16 < nksv) {
            ldsm_x2(dr + uint32_t(s16 * 32), bda[i][0], bda[i][1]);
            ldsm_x2(dl + uint32_t(s16 * 32), bdl[i][0], bdl[i][1]);
          }
        }
        if (g8 >= mt) {
#pragma unroll
          for (int i = 0; i < KS; ++i) bx[i][0] = bx[i][1] = 0u;
#pragma unroll
          for (int i = 0; i < KSV; ++i) bda[i][0] = bda[i][1] = bdl[i][0] = bdl[i][1] = 0u;
        }
        x_release = slot;
      }
      ++ngc;
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
    if (x_release >= 0) {  // every warp holds its fragments
      if (tid == 0) tc::mbar_arrive(&ms->x_empty[x_release]);
      x_release = -1;
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
constexpr int kBThreads = 256;
constexpr int kYld = kBCols + 8;  // bf16 row stride of the token tile (conflict-free)
constexpr int kWld = 24;          // bf16 row stride of the weight tiles

// One unit: segment s, rows [r0, r0 + 64) of its id, columns [col0, col0 + 256) of dK
// (part 0) or dV (part 1). D[col][row] = sum_q Y[q][col] W[q][row] over the segment's
// sorted positions q, Y = x (dK) or da (dV), W = ds (dK) or p (dV).
__global__ void __launch_bounds__(kBThreads) seg_rows_kernel(const SegRowsArgs a) {
  __shared__ __align__(16) __nv_bfloat16 ys[16][kYld];
  __shared__ __align__(16) __nv_bfloat16 wh[kBRows][kWld];
  __shared__ __align__(16) __nv_bfloat16 wl[kBRows][kWld];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g8 = lane >> 2, t4 = lane & 3;
  const int S = *a.n_seg;
  const int64_t units = a.seg_unit0[S];
  const int ncb_k = (a.d + kBCols - 1) / kBCols, ncb_v = (a.d_v + kBCols - 1) / kBCols;
  const int ncb = ncb_k + ncb_v;
  for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
    // segment of unit u: the last s with seg_unit0[s] <= u
    int lo = 0, hi = S - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (a.seg_unit0[mid] <= u)
        lo = mid;
      else
        hi = mid - 1;
    }
    const int s = lo;
    const int64_t local = u - a.seg_unit0[s];
    const int rb = int(local / ncb), cb = int(local % ncb);
    const int part = cb < ncb_k ? 0 : 1;
    const int width = part ? a.d_v : a.d;
    const int col0 = (part ? cb - ncb_k : cb) * kBCols;
    const int qs = a.seg_start[s], qe = a.seg_start[s + 1];
    const int t = int(a.sorted_keys[qs] >> 32);
    const int rbase = a.offs[t];
    const int n = a.offs[t + 1] - rbase;
    const int r0 = rb * kBRows;
    const int64_t orow0 = int64_t(a.seg_row0[s]) + r0;  // output row of row r0
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
    float acc[2][8][4];
#pragma unroll
    for (int mi = 0; mi < 2; ++mi)
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) acc[mi][nt][0] = acc[mi][nt][1] = acc[mi][nt][2] = acc[mi][nt][3] = 0.f;
    // tile loads: thread tid takes token tid / 16: 16 columns (two 16-byte pieces) of Y and
    // 4 rows of W
    const int lt = tid >> 4, lc = (tid & 15) * 16, lr = (tid & 15) * 4;
    uint4 yv[2];
    float wv[4];
    auto load = [&](int q) {  // tile of tokens q .. q + 15
      const int qq = q + lt;
      yv[0] = yv[1] = make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int j = 0; j < 4; ++j) wv[j] = 0.f;
      if (qq < qe) {
        const int c = col0 + lc;
        const __nv_bfloat16* yr = Y + int64_t(qq) * width + c;
        if (c < width) yv[0] = __ldg(reinterpret_cast<const uint4*>(yr));
        if (c + 8 < width) yv[1] = __ldg(reinterpret_cast<const uint4*>(yr + 8));
        const float* wr = Wsrc + int64_t(qq) * a.k_max + r0 + lr;
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (r0 + lr + j < n) wv[j] = __ldg(wr + j);
      }
    };
    load(qs);
    for (int q = qs; q < qe; q += 16) {
      *reinterpret_cast<uint4*>(&ys[lt][lc]) = yv[0];
      *reinterpret_cast<uint4*>(&ys[lt][lc + 8]) = yv[1];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const __nv_bfloat16 h = __float2bfloat16_rn(wv[j]);
        wh[lr + j][lt] = h;
        wl[lr + j][lt] = __float2bfloat16_rn(wv[j] - __bfloat162float(h));
      }
      __syncthreads();
      if (q + 16 < qe) load(q + 16);  // the next tile is in flight during the products
      // warp w: column tiles 2w, 2w + 1 (16 columns each), all 8 row tiles
      const int vl = (lane & 7) + (lane >> 4) * 8;
      const int vcol = ((lane >> 3) & 1) * 8;
#pragma unroll
      for (int mi = 0; mi < 2; ++mi) {
        const int cl = 16 * (2 * warp + mi);
        if (col0 + cl >= width) break;
        uint32_t a0, a1, a2, a3;
        ldsm_x4_t(tc::smem_u32(&ys[vl][cl + vcol]), a0, a1, a2, a3);
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
          const int row = 8 * nt + g8;
          const uint32_t h0 = *reinterpret_cast<const uint32_t*>(&wh[row][2 * t4]);
          const uint32_t h1 = *reinterpret_cast<const uint32_t*>(&wh[row][2 * t4 + 8]);
          const uint32_t l0 = *reinterpret_cast<const uint32_t*>(&wl[row][2 * t4]);
          const uint32_t l1 = *reinterpret_cast<const uint32_t*>(&wl[row][2 * t4 + 8]);
          mma16(acc[mi][nt], a0, a1, a2, a3, h0, h1);
          mma16(acc[mi][nt], a0, a1, a2, a3, l0, l1);
        }
      }
      __syncthreads();
    }
    // D[col][row]: lane (g8, t4) holds cols cl + g8 (+ 8) and rows 8 nt + 2 t4 (+ 1)
#pragma unroll
    for (int mi = 0; mi < 2; ++mi) {
      const int c0 = col0 + 16 * (2 * warp + mi) + g8;
      if (col0 + 16 * (2 * warp + mi) >= width) break;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        const int rr = 8 * nt + 2 * t4;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int row = rr + (e & 1), col = c0 + (e >> 1) * 8;
          if (r0 + row < n && orow0 + row < a.max_rows)
            out[(orow0 + row) * width + col] = acc[mi][nt][e];
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

// Per sorted position q (one warp): x and da rows in sorted order (bf16), da in batch order
// as bf16 hi + lo, and δ_i = a_i · da_i for the token i = perm(q).
__global__ void bwd_prep_kernel(const uint64_t* __restrict__ keys, int64_t T,
                                const __nv_bfloat16* __restrict__ x, const float* __restrict__ a,
                                const float* __restrict__ da, int d, int d_v,
                                __nv_bfloat16* __restrict__ x_sorted,
                                __nv_bfloat16* __restrict__ da_sorted,
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
    da_sorted[q * d_v + c] = gb;
    da16[i * d_v + c] = gb;
    da16_lo[i * d_v + c] = __float2bfloat16_rn(g - __bfloat162float(gb));
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
                                                        int32_t* n_rows, int64_t max_rows,
                                                        DevStatus* st) {
  __shared__ int2 wt[32];
  __shared__ int2 tot;
  const int S = *n_seg;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int64_t carry_r = 0, carry_u = 0;
  for (int base = 0; base < S; base += blockDim.x) {
    const int s = base + threadIdx.x;
    int nr = 0, nu = 0;
    if (s < S) {
      const int t = int(keys[seg_start[s]] >> 32);
      nr = offs[t + 1] - offs[t];
      nu = (nr + kBRows - 1) / kBRows * ncb;
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
    if (lane == 31) wt[wid] = incl;
    __syncthreads();
    if (wid == 0) {
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
    }
    carry_r += tot.x;
    carry_u += tot.y;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    seg_unit0[S] = int32_t(carry_u);
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
      (reinterpret_cast<uintptr_t>(a.x) & 15) || (reinterpret_cast<uintptr_t>(a.da16) & 15) ||
      (reinterpret_cast<uintptr_t>(a.da16_lo) & 15))
    return cudaErrorInvalidValue;
  if (sh.ch == 8 && a.d == 2048 && a.d_v == 512) return launch_bwd_a<8, 16, 4, 16>(a, sh, stream);
  if (sh.ch == 16 && a.d == 1024 && a.d_v == 256) return launch_bwd_a<16, 8, 2, 8>(a, sh, stream);
  return sh.ch == 16 ? launch_bwd_a<16, 0, 0, 0>(a, sh, stream)
                     : launch_bwd_a<8, 0, 0, 0>(a, sh, stream);
}

cudaError_t launch_seg_rows(const SegRowsArgs& a, cudaStream_t stream) {
  seg_rows_kernel<<<unsigned(device_sm_count() * 4), kBThreads, 0, stream>>>(a);
  count_launch();
  return cudaGetLastError();
}

int seg_rows_col_blocks(int d, int d_v) {
  return (d + kBCols - 1) / kBCols + (d_v + kBCols - 1) / kBCols;
}

cudaError_t launch_row_plan(const uint64_t* keys, const int32_t* seg_start, const int32_t* n_seg,
                            const int32_t* offs, int d, int d_v, int32_t* seg_row0,
                            int32_t* seg_unit0, int32_t* n_rows, int64_t max_rows,
                            DevStatus* st, cudaStream_t stream) {
  row_plan_kernel<<<1, 1024, 0, stream>>>(keys, seg_start, n_seg, offs,
                                          seg_rows_col_blocks(d, d_v), seg_row0, seg_unit0,
                                          n_rows, max_rows, st);
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
                                                   a.x_sorted, a.da_sorted, a.da16, a.da16_lo,
                                                   a.delta);
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
