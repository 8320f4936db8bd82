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
  // Holders: the CTAs whose non-empty range meets [c0, c1), in CTA order around this one
  // (CTAs with empty ranges may sit between them). Warp 0 looks at the 32 CTAs on each side
  // at once (one pair of range bounds per lane and side) and takes the holders from the
  // two ballots; only when the holders found do not cover [c0, c1) (more lie outside the
  // windows) is the run walked one CTA at a time.
  if (tid < 32) {
    const int b = int(blockIdx.x), n = a.n_cta;
    auto holds = [&](int bb, int32_t& s0, int32_t& s1) {
      const bool in = bb >= 0 && bb < n;
      s0 = in ? cs[bb] : 0;
      s1 = in ? cs[bb + 1] : 0;
      return in && s0 < s1 && s0 < c1 && s1 > c0;
    };
    int32_t s_lo = 0, e_lo = 0, s_hi = 0, e_hi = 0;
    const bool h_lo = holds(b - 32 + tid, s_lo, e_lo);  // b-32 .. b-1
    const bool h_hi = holds(b + 1 + tid, s_hi, e_hi);   // b+1 .. b+32
    const unsigned lo = __ballot_sync(0xffffffffu, h_lo);
    const unsigned hi = __ballot_sync(0xffffffffu, h_hi);
    // holder CTAs in order: the set bits of lo, then b, then the set bits of hi
    const int nlo = __popc(lo), nhi = __popc(hi);
    if (h_lo) {
      const int k = __popc(lo & ((1u << tid) - 1u));
      if (k < kMergeCap) sm->hold[k] = b - 32 + tid;
    }
    if (h_hi) {
      const int k = nlo + 1 + __popc(hi & ((1u << tid) - 1u));
      if (k < kMergeCap) sm->hold[k] = b + 1 + tid;
    }
    // range start of the lowest holder and range end of the highest one, from the lanes
    // that looked at them
    const int low_lane = lo ? __ffs(lo) - 1 : 0;
    const int high_lane = hi ? 31 - __clz(hi) : 0;
    const int32_t s_low = __shfl_sync(0xffffffffu, s_lo, low_lane);
    const int32_t e_high = __shfl_sync(0xffffffffu, e_hi, high_lane);
    (void)s_hi;
    (void)e_lo;
    if (tid == 0) {
      sm->hold[nlo < kMergeCap ? nlo : kMergeCap - 1] = b;
      int nh = nlo + 1 + nhi;
      int64_t start0 = lo ? s_low : cb;  // range start of the first holder
      const int64_t end1 = hi ? e_high : ce;  // range end of the last holder
      if (start0 > c0 || end1 < c1) {
        // holders outside the windows: list them again, walking from the first
        int b0 = lo ? b - 32 + low_lane : b;
        for (int bb = b0 - 1; bb >= 0 && cs[b0] > c0; --bb)
          if (cs[bb] < cs[bb + 1]) b0 = bb;
        int b1 = b;
        for (int bb = b + 1; bb < n && cs[bb] < c1; ++bb)
          if (cs[bb] < cs[bb + 1]) b1 = bb;
        nh = 0;
        for (int bb = b0; bb <= b1; ++bb)
          if (cs[bb] < cs[bb + 1] && nh < kMergeCap) sm->hold[nh++] = bb;
        start0 = cs[b0];
      }
      sm->nh = nh < kMergeCap ? nh : kMergeCap;
      sm->first_second = c0 > start0 ? 1 : 0;  // the group is the first holder's second slot
    }
  }
  merge_held(a, q0, mt, sm, tid, nthr, bar);
}

// Merge the partials of a group (tokens q0 .. q0 + mt - 1 in sorted order) held by the CTAs
// sm->hold[0 .. sm->nh) in CTA order (holder 0 keeps it in its second slot if
// sm->first_second), and write the group's outputs. Same caller rules as arrive_and_merge.
// Thread tid takes the column pair cp = tid % half (half = d_v / 2) of the tokens tid / half,
// + nthr / half, ... Every load that does not depend on another goes out in one phase: the
// holders' (m, l), the tokens' batch indices and the thread's share of the first kMergeW
// holders' partial sums for its first token; the weights follow, then the sums.
template <typename Bar>
__device__ __noinline__ void merge_held(const AttendArgs& a, int q0, int mt, MergeSmem* sm,
                                        int tid, int nthr, Bar bar) {
  bar();
  const int nh = sm->nh;
  const bool fs = sm->first_second != 0;
  auto entry = [&](int h, int j) { return part_entry(a, sm->hold[h], h == 0 && fs, j); };
  const int nw = nh < kMergeW ? nh : kMergeW;
  const int half = a.d_v / 2;
  const int jstep = nthr / half;
  const int cp = tid % half, j0 = tid / half;
  for (int e = tid; e < mt * nw; e += nthr) {
    const int j = e / nw, h = e - j * nw;
    const float* pp = entry(h, j);
    sm->w[j][h] = __ldcg(pp);
    sm->l[j][h] = __ldcg(pp + 1);
  }
  if (tid < mt) sm->tok[tid] = int64_t(uint32_t(a.sorted_keys[q0 + tid]));
  float2 pre[kMergeW];
#pragma unroll
  for (int h = 0; h < kMergeW; ++h)
    pre[h] = j0 < mt && h < nw ? __ldcg(reinterpret_cast<const float2*>(entry(h, j0) + 2 + 2 * cp))
                               : make_float2(0.f, 0.f);
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
    if (a.ml) {
      const int64_t i = sm->tok[j];
      a.ml[2 * i] = M;
      a.ml[2 * i + 1] = L;
    }
  }
  bar();
  // a = sum_h w_h acc_h: the first token from the registers loaded above, each further token
  // with one batch of loads; holders past kMergeW one by one
#pragma unroll 1
  for (int j = j0; j < mt; j += jstep) {
    if (j != j0) {
#pragma unroll
      for (int h = 0; h < kMergeW; ++h)
        pre[h] = h < nw ? __ldcg(reinterpret_cast<const float2*>(entry(h, j) + 2 + 2 * cp))
                        : make_float2(0.f, 0.f);
    }
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int h = 0; h < kMergeW; ++h) {
      const float wt = h < nw ? sm->w[j][h] : 0.f;
      s0 = fmaf(pre[h].x, wt, s0);
      s1 = fmaf(pre[h].y, wt, s1);
    }
#pragma unroll 1
    for (int h = kMergeW; h < nh; ++h) {
      const float* pp = entry(h, j);
      const float wt = expf(__ldcg(pp) - sm->M[j]) * sm->inv_l[j];
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
