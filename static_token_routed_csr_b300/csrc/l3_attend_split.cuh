// Pieces shared by the two split-row gather-attend kernels (CUDA cores for fp32 layers,
// warp-level tensor cores for bf16 layers): the bulk copy that fills a stage, the output
// and partial slots, and the merge of the partial (m, l, acc) of a group whose chunks
// several CTAs processed ("L³: Large Lookup Layers", gist.science explainer,
// Technical Summary, "Core Architecture": a = V_tᵀ softmax(K_t x), here assembled from
// row blocks by the usual rescaling m = max m_b, l = sum_b l_b e^(m_b - m),
// acc = sum_b acc_b e^(m_b - m), a = acc / l).
#pragma once

#include <math.h>

#include "l3_internal.h"
#include "l3_tc.cuh"

namespace l3 {
namespace split {

constexpr int kThreads = 256;
constexpr int kMT = kPlanMT;
constexpr int kMaxCtas = kPlanMaxCtas;
constexpr int kSmemLimit = 232448;  // 227 KB of opt-in shared memory per CTA

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(tc::smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(tc::smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void write_a(const AttendArgs& a, int64_t i, int col, float v) {
  if (a.a_f32) a.a_f32[i * a.d_v + col] = v;
  if (a.a_bf16) a.a_bf16[i * a.d_v + col] = __float2bfloat16_rn(v);
}

// Partial of CTA b for a group: slot 0 if the group holds the CTA's first chunk, else 1
// (only the group still open at the end of the range can be the second). Each slot holds
// kMT token entries of (m, l, acc[d_v]).
__device__ __forceinline__ float* part_entry(const AttendArgs& a, int64_t b, bool second, int j) {
  return a.part + ((2 * b + (second ? 1 : 0)) * kMT + j) * int64_t(a.d_v + 2);
}

// Shared memory of a merge: the CTAs holding chunks of the group (in CTA order) and, for up
// to kMergeW of them, each token's weight e^(m_b - M) / L.
constexpr int kMergeCap = 128;  // holders of a group: at most k_max / ch <= 128 chunks
constexpr int kMergeW = 16;
struct MergeSmem {
  int hold[kMergeCap];
  float w[kMT][kMergeW];  // a holder's m, then its weight
  float l[kMT][kMergeW];
  float M[kMT], inv_l[kMT];
  int64_t tok[kMT];       // batch index of each of the group's tokens
  int nh, first_second, last;
};

template <typename Bar>
__device__ __noinline__ void merge_held(const AttendArgs& a, int q0, int mt, MergeSmem* sm,
                                        int tid, int nthr, Bar bar);

// After this CTA (chunks [cb, ce)) wrote its partial for group g (chunks [c0, c1)): count
// the group's chunks done and, in the CTA that completes the count, merge all partials in
// CTA order and write the group's outputs. Called by the CTA's `nthr` working threads,
// numbered tid = 0 .. nthr-1 (nthr >= 32); `bar()` is a barrier over exactly those threads.
// Kept out of line: the merge is rare and its registers must not weigh on the caller's loop.
template <typename Bar>
__device__ __noinline__ void arrive_and_merge(const AttendArgs& a, int g, int64_t c0, int64_t c1,
                                        int64_t cb, int64_t ce, int q0, int mt, MergeSmem* sm,
                                        int tid, int nthr, Bar bar) {
  const int32_t* cs = a.cta_start;
  __threadfence();
  bar();
  if (tid == 0) {
    const int mine = int((c1 < ce ? c1 : ce) - (c0 > cb ? c0 : cb));
    sm->last = atomicAdd(&a.counters[g], mine) + mine == int(c1 - c0) ? 1 : 0;
  }
  bar();
  if (!sm->last) return;
  __threadfence();
  // Holders: the CTAs whose non-empty range meets [c0, c1), contiguous around this one.
  // Warp 0 looks at the 32 CTAs on each side at once; a longer run is walked one by one.
  if (tid < 32) {
    const int b = int(blockIdx.x), n = a.n_cta;
    auto holds = [&](int bb) {
      return bb >= 0 && bb < n && cs[bb] < cs[bb + 1] && cs[bb] < c1 && cs[bb + 1] > c0;
    };
    const unsigned lo = __ballot_sync(0xffffffffu, holds(b - 32 + tid));  // b-32 .. b-1
    const unsigned hi = __ballot_sync(0xffffffffu, holds(b + 1 + tid));   // b+1 .. b+32
    if (tid == 0) {
      int b0 = b, b1 = b;
      // holders are contiguous among the non-empty ranges; empty ranges may sit between
      if (c0 < cb) {
        b0 = -1;
        for (int k = 31; k >= 0; --k)
          if (lo >> k & 1u) b0 = b - 32 + k;  // lowest holder in the window
        // until the holder of chunk c0 is found, step down past the window
        for (int bb = (b0 < 0 ? b - 33 : b0 - 1); bb >= 0 && (b0 < 0 || cs[b0] > c0); --bb)
          if (cs[bb] < cs[bb + 1]) b0 = bb;
      }
      if (c1 > ce) {
        b1 = -1;
        for (int k = 0; k < 32; ++k)
          if (hi >> k & 1u) b1 = b + 1 + k;  // highest holder in the window
        // until the holder of chunk c1 - 1 is found, step up past the window
        for (int bb = (b1 < 0 ? b + 33 : b1 + 1); bb < n && (b1 < 0 || cs[b1 + 1] < c1); ++bb)
          if (cs[bb] < cs[bb + 1]) b1 = bb;
      }
      int nh = 0;
      for (int bb = b0; bb <= b1; ++bb)
        if (cs[bb] < cs[bb + 1] && nh < kMergeCap) sm->hold[nh++] = bb;
      sm->nh = nh;
      sm->first_second = c0 > cs[b0] ? 1 : 0;  // the group is CTA b0's second slot
    }
  }
  merge_held(a, q0, mt, sm, tid, nthr, bar);
}

// Merge the partials of a group (tokens q0 .. q0 + mt - 1 in sorted order) held by the CTAs
// sm->hold[0 .. sm->nh) in CTA order (holder 0 keeps it in its second slot if
// sm->first_second), and write the group's outputs. Same caller rules as arrive_and_merge.
template <typename Bar>
__device__ __noinline__ void merge_held(const AttendArgs& a, int q0, int mt, MergeSmem* sm,
                                        int tid, int nthr, Bar bar) {
  bar();
  const int nh = sm->nh;
  const bool fs = sm->first_second != 0;
  auto entry = [&](int h, int j) { return part_entry(a, sm->hold[h], h == 0 && fs, j); };
  // every holder's (m, l) for every token, loaded at once (the first kMergeW holders)
  const int nw = nh < kMergeW ? nh : kMergeW;
  for (int e = tid; e < mt * nw; e += nthr) {
    const int j = e / nw, h = e - j * nw;
    const float* pp = entry(h, j);
    sm->w[j][h] = __ldcg(pp);
    sm->l[j][h] = __ldcg(pp + 1);
  }
  bar();
  // token j: max and denominator over the holders, then the holders' weights
  if (tid < mt) {
    const int j = tid;
    float M = -INFINITY;
    for (int h = 0; h < nh; ++h) M = fmaxf(M, h < kMergeW ? sm->w[j][h] : __ldcg(entry(h, j)));
    float L = 0.f;
    for (int h = 0; h < nh; ++h) {
      const float m = h < kMergeW ? sm->w[j][h] : __ldcg(entry(h, j));
      const float l = h < kMergeW ? sm->l[j][h] : __ldcg(entry(h, j) + 1);
      L = fmaf(l, expf(m - M), L);
    }
    const float inv = 1.f / L;
    for (int h = 0; h < nw; ++h) sm->w[j][h] = expf(sm->w[j][h] - M) * inv;
    sm->M[j] = M;
    sm->inv_l[j] = inv;
    const int64_t i = int64_t(uint32_t(a.sorted_keys[q0 + j]));
    sm->tok[j] = i;
    if (a.ml) {
      a.ml[2 * i] = M;
      a.ml[2 * i + 1] = L;
    }
  }
  bar();
  // a = sum_h w_h acc_h. Thread tid takes the column pair cp = tid % half of the tokens
  // tid / half, + nthr / half, ... (d_v <= 512, so half <= nthr). The code is kept compact:
  // a merge runs at most once per group, often with the instruction cache cold, and four
  // holders' loads are in flight per step.
  const int half = a.d_v / 2;
  const int jstep = nthr / half;
  const int cp = tid % half;
#pragma unroll 1
  for (int j = tid / half; j < mt; j += jstep) {
    float s0 = 0.f, s1 = 0.f;
    int h = 0;
#pragma unroll 1
    for (; h + 4 <= nw; h += 4) {
      float2 v[4];
#pragma unroll
      for (int e = 0; e < 4; ++e)
        v[e] = __ldcg(reinterpret_cast<const float2*>(entry(h + e, j) + 2 + 2 * cp));
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float wt = sm->w[j][h + e];
        s0 = fmaf(v[e].x, wt, s0);
        s1 = fmaf(v[e].y, wt, s1);
      }
    }
#pragma unroll 1
    for (; h < nh; ++h) {
      const float* pp = entry(h, j);
      const float wt = h < kMergeW ? sm->w[j][h] : expf(__ldcg(pp) - sm->M[j]) * sm->inv_l[j];
      const float2 v = __ldcg(reinterpret_cast<const float2*>(pp + 2 + 2 * cp));
      s0 = fmaf(v.x, wt, s0);
      s1 = fmaf(v.y, wt, s1);
    }
    write_a(a, sm->tok[j], 2 * cp, s0);
    write_a(a, sm->tok[j], 2 * cp + 1, s1);
  }
}

int sm_count();

}  // namespace split
}  // namespace l3
