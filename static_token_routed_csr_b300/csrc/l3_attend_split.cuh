// Pieces shared by the two split-row gather-attend kernels (CUDA cores for fp32 layers,
// warp-level tensor cores for bf16 layers): the walk over the plan's chunk list, the bulk
// copies that fill a stage, and the merge of the partial (m, l, acc) of a group whose
// chunks several CTAs processed ("L³: Large Lookup Layers", gist.science explainer,
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
constexpr int kMaxCtas = 256;
constexpr int kSmemLimit = 232448;  // 227 KB of opt-in shared memory per CTA

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(tc::smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(tc::smem_u32(bar))
      : "memory");
}

// CTA b of G covers chunks [b C / G, (b+1) C / G); the CTA that holds chunk c:
__device__ __forceinline__ int cta_of(int64_t c, int64_t C, int64_t G) {
  return int(((c + 1) * G - 1) / C);
}

// Largest group g in [0, n_groups) with groups[g].c0 <= c.
__device__ __forceinline__ int find_group(const AttendGroup* groups, int n_groups, int64_t c) {
  int lo = 0, hi = n_groups - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (groups[mid].c0 <= c)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
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

// After this CTA wrote its partial for group g (chunks [c0, c1)): count it and, in the CTA
// that completes the group, merge all partials in CTA order and write the group's outputs.
// Called by the CTA's `nthr` working threads, numbered tid = 0 .. nthr-1; `bar()` is a
// barrier over exactly those threads; `last` is a shared-memory flag.
template <typename Bar>
__device__ inline void arrive_and_merge(const AttendArgs& a, int g, int64_t c0, int64_t c1,
                                        int64_t C, int64_t G, int q0, int mt, int* last,
                                        int tid, int nthr, Bar bar) {
  __threadfence();
  bar();
  const int b0 = cta_of(c0, C, G), b1 = cta_of(c1 - 1, C, G);
  if (tid == 0) *last = atomicAdd(&a.counters[g], 1) == b1 - b0;
  bar();
  if (!*last) return;
  __threadfence();
  const int64_t cs0 = int64_t(b0) * C / G;  // first chunk of CTA b0
  const bool first_second = c0 > cs0;       // the group is CTA b0's second slot
  for (int j = 0; j < mt; ++j) {
    float M = -INFINITY;
    for (int bb = b0; bb <= b1; ++bb)
      M = fmaxf(M, __ldcg(part_entry(a, bb, bb == b0 && first_second, j)));
    float L = 0.f;
    for (int bb = b0; bb <= b1; ++bb) {
      const float* pp = part_entry(a, bb, bb == b0 && first_second, j);
      L = fmaf(__ldcg(pp + 1), expf(__ldcg(pp) - M), L);
    }
    const int64_t i = int64_t(uint32_t(a.sorted_keys[q0 + j]));
    const float inv = 1.f / L;
    for (int col = tid; col < a.d_v; col += nthr) {
      float s = 0.f;
      for (int bb = b0; bb <= b1; ++bb) {
        const float* pp = part_entry(a, bb, bb == b0 && first_second, j);
        s = fmaf(__ldcg(pp + 2 + col), expf(__ldcg(pp) - M), s);
      }
      write_a(a, i, col, s * inv);
    }
    if (a.ml && tid == 0) {
      a.ml[2 * i] = M;
      a.ml[2 * i + 1] = L;
    }
  }
}

int sm_count();

}  // namespace split
}  // namespace l3
