// Batch sorting by token id ("L³: Large Lookup Layers", gist.science explainer,
// Technical Summary, "Systems-Friendly Design": sorting a batch by token id turns the
// layer's attention mask block-diagonal).
//
// Keys are (id << 32) | batch position. They are unique, so any correct sort of the keys
// is the stable sort of the ids. Batches of at most 256 tokens are ranked in one pass by one
// CTA. Larger ones: with ids below 2^19, blocks of 8192 tokens are sorted by one CTA each
// with a stable radix sort on the ids; otherwise blocks of 4096 keys are sorted by a
// shared-memory bitonic network. Blocks are then merged pairwise (each key
// finds its rank in the other run by binary search).
// A last pass marks segment starts and numbers the segments, and (for the forward) lays out
// the work plan of the split-row gather-attend.
#include "l3_internal.h"
#include "l3_tc.cuh"

namespace l3 {

namespace {

constexpr int kChunk = 4096;  // keys per CTA sort (32 KB of shared memory)

__device__ inline uint64_t make_key(const int32_t* ids, int64_t T, int64_t vocab, int64_t i,
                                    DevStatus* st) {
  if (i >= T) return ~0ull;
  int32_t id = ids[i];
  if (id < 0 || int64_t(id) >= vocab) {
    atomicOr(&st->token_range, 1);
    id = 0;  // keep every later access in bounds; the row's output is unspecified
  }
  return (uint64_t(uint32_t(id)) << 32) | uint64_t(i);
}

// Bitonic sort of n (power of two, <= kChunk) keys in shared memory by the whole CTA.
__device__ void block_bitonic(uint64_t* s, int n) {
  for (int k = 2; k <= n; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < n; i += blockDim.x) {
        int p = i ^ j;
        if (p > i) {
          uint64_t a = s[i], b = s[p];
          bool up = (i & k) == 0;
          if ((a > b) == up) {
            s[i] = b;
            s[p] = a;
          }
        }
      }
      __syncthreads();
    }
  }
}

// Exclusive scan of one int per thread across the CTA (blockDim.x == 1024).
__device__ int block_exclusive_scan(int v, int* warp_tot, int* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) warp_tot[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    int w = lane < (int)(blockDim.x >> 5) ? warp_tot[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int u = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += u;
    }
    warp_tot[lane] = wi - w;
    if (lane == 31) *total = wi;
  }
  __syncthreads();
  int r = warp_tot[wid] + incl - v;
  __syncthreads();
  return r;
}

// Exclusive scan of four ints per thread at once (blockDim.x == 1024); *total gets the sums.
__device__ int4 block_exclusive_scan4(int4 v, int4* warp_tot, int4* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int4 incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int ux = __shfl_up_sync(0xffffffffu, incl.x, o);
    const int uy = __shfl_up_sync(0xffffffffu, incl.y, o);
    const int uz = __shfl_up_sync(0xffffffffu, incl.z, o);
    const int uw = __shfl_up_sync(0xffffffffu, incl.w, o);
    if (lane >= o) {
      incl.x += ux;
      incl.y += uy;
      incl.z += uz;
      incl.w += uw;
    }
  }
  if (lane == 31) warp_tot[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    const int4 w = lane < (int)(blockDim.x >> 5) ? warp_tot[lane] : make_int4(0, 0, 0, 0);
    int4 wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int ux = __shfl_up_sync(0xffffffffu, wi.x, o);
      const int uy = __shfl_up_sync(0xffffffffu, wi.y, o);
      const int uz = __shfl_up_sync(0xffffffffu, wi.z, o);
      const int uw = __shfl_up_sync(0xffffffffu, wi.w, o);
      if (lane >= o) {
        wi.x += ux;
        wi.y += uy;
        wi.z += uz;
        wi.w += uw;
      }
    }
    warp_tot[lane] = make_int4(wi.x - w.x, wi.y - w.y, wi.z - w.z, wi.w - w.w);
    if (lane == 31) *total = wi;
  }
  __syncthreads();
  const int4 b = warp_tot[wid];
  const int4 r = make_int4(b.x + incl.x - v.x, b.y + incl.y - v.y, b.z + incl.z - v.z,
                           b.w + incl.w - v.w);
  __syncthreads();
  return r;
}

// CTA b's head: group gh, which holds chunk c (the first of b's range); an empty head
// when there is no such group (gh >= NG: the range is empty).
__device__ void write_head(const PlanOut& pl, int64_t b, int gh, int64_t c, int NG) {
  CtaHead h{};
  h.cb = int32_t(c);  // ce is filled in once every range start is known
  if (gh >= NG) {
    pl.cta_head[b] = h;
    return;
  }
  const AttendGroup& gr = pl.groups[gh];
  h.g = gh;
  h.q0 = gr.q0;
  h.mt = gr.mt;
  h.n = gr.n;
  h.row0 = gr.row0;
  h.c0 = gr.c0;
  h.c1 = pl.groups[gh + 1].c0;
  h.row = gr.row0 + int32_t(c - gr.c0) * pl.ch;
#pragma unroll
  for (int j = 0; j < kPlanMT; ++j) h.tok[j] = gr.tok[j];
  pl.cta_head[b] = h;
}

// Work plan of the gather-attend (see PlanOut), from the finished segment table.
__device__ void plan_pass(const uint64_t* keys, int64_t T, const int32_t* seg_start, int S,
                          const PlanOut& pl, DevStatus* st, int* warp_tot, int* total) {
  int gcarry = 0, ccarry = 0, icarry = 0, wcarry = 0;
  for (int base = 0; base < S; base += blockDim.x) {
    const int s = base + threadIdx.x;
    int ng = 0, nc = 0, ni = 0, nw = 0, q0 = 0, m = 0, t = 0, row0 = 0, n = 0, per = 0;
    if (s < S) {
      q0 = seg_start[s];
      m = seg_start[s + 1] - q0;
      t = int(keys[q0] >> 32);
      row0 = pl.offs[t];
      n = pl.offs[t + 1] - row0;
      if (n < 1 || n > pl.k_max || row0 < 0 || int64_t(row0) + n > pl.v) {
        atomicOr(&st->layer_bad, 1);
        n = 0;  // no rows are read for this id; its tokens' outputs are unspecified
      }
      if (m >= pl.th) {
        ni = n > 0 ? (m + kTcNT - 1) / kTcNT : 0;
      } else {
        ng = (m + pl.mt_max - 1) / pl.mt_max;
        per = n > 0 ? (n + pl.ch - 1) / pl.ch : 0;
        nc = ng * per;
        nw = per > 0 ? ng : 0;  // groups with chunks
      }
    }
    __shared__ int4 wt4[32], tot4;
    const int4 ex = block_exclusive_scan4(make_int4(ng, nc, ni, nw), wt4, &tot4);
    const int4 tot = tot4;
    const int gex = ex.x, cex = ex.y, iex = ex.z, wex = ex.w;
    const int gtot = tot.x, ctot = tot.y, itot = tot.z, wtot = tot.w;
    for (int k = 0; k < ng; ++k) {
      AttendGroup g;
      g.q0 = q0 + k * pl.mt_max;
      g.mt = m - k * pl.mt_max < pl.mt_max ? m - k * pl.mt_max : pl.mt_max;
      g.t = t;
      g.row0 = row0;
      g.n = n;
      g.c0 = ccarry + cex + k * per;
      g.w0 = g.c0 * pl.w_chunk + (wcarry + wex + (per > 0 ? k : 0)) * pl.w_group;
      g.pad = 0;
#pragma unroll
      for (int j = 0; j < kPlanMT; ++j)
        g.tok[j] = j < g.mt ? int32_t(uint32_t(keys[g.q0 + j])) : 0;
      pl.groups[gcarry + gex + k] = g;
      pl.counters[gcarry + gex + k] = 0;
    }
    for (int k = 0; k < ni; ++k) {
      AttendItem it;
      it.q0 = q0 + k * kTcNT;
      it.nt = m - k * kTcNT < kTcNT ? m - k * kTcNT : kTcNT;
      it.t = t;
      it.pad = 0;
      pl.items[icarry + iex + k] = it;
    }
    gcarry += gtot;
    ccarry += ctot;
    icarry += itot;
    wcarry += wtot;
  }
  if (threadIdx.x == 0) {
    AttendGroup end{};
    end.q0 = int32_t(T);
    end.c0 = ccarry;
    end.w0 = ccarry * pl.w_chunk + wcarry * pl.w_group;
    pl.groups[gcarry] = end;
    pl.hdr[kPlanGroups] = gcarry;
    pl.hdr[kPlanChunks] = ccarry;
    pl.hdr[kPlanItems] = icarry;
    pl.hdr[3] = 0;
  }
  if (!pl.cta_start) return;
  // Cost-balanced split of the chunk list. Chunk c covers the cost units
  // [UB(c), UB(c + 1)), UB(c) = c w_chunk + (groups with chunks that start before c) w_group,
  // so the group holding chunk c0 of its first chunk covers [w0, w0 + w_group + n_c w_chunk).
  // CTA b starts at the first chunk with UB(c) >= tau_b = b U / n_cta (U = UB(C)): chunk 0
  // if tau_b = 0, else one past the chunk covering unit tau_b - 1. Each group fills in the
  // CTAs whose unit tau_b - 1 it covers.
  __syncthreads();
  const int NG = gcarry;
  const int64_t C = ccarry;
  const int64_t n = pl.n_cta;
  const int64_t U = C * pl.w_chunk + int64_t(wcarry) * pl.w_group;
  if (U == 0) {
    for (int b = threadIdx.x; b <= n; b += blockDim.x) {
      pl.cta_start[b] = 0;
      if (b < n) {
        pl.cta_group[b] = 0;
        pl.cta_head[b] = CtaHead{};
      }
    }
    return;
  }
  // CTAs with tau_b = 0: b U < n
  const int64_t b_zero = (n + U - 1) / U;  // smallest b with b U >= n
  // the first group with chunks (groups without rows have none)
  int g_first = 0;
  while (g_first < NG && pl.groups[g_first + 1].c0 == pl.groups[g_first].c0) ++g_first;
  for (int64_t b = threadIdx.x; b < b_zero && b <= n; b += blockDim.x) {
    pl.cta_start[b] = 0;
    if (b < n) {
      pl.cta_group[b] = 0;
      write_head(pl, b, g_first, 0, NG);
    }
  }
  for (int g = threadIdx.x; g < NG; g += blockDim.x) {
    const int64_t c0 = pl.groups[g].c0, c1 = pl.groups[g + 1].c0;
    if (c1 <= c0) continue;
    const int64_t W0 = pl.groups[g].w0;
    const int64_t W1 = W0 + pl.w_group + (c1 - c0) * pl.w_chunk;
    // b with W0 <= tau_b - 1 < W1, i.e. W0 + 1 <= floor(b U / n) <= W1
    const int64_t b_lo = ((W0 + 1) * n + U - 1) / U;
    const int64_t b_hi = ((W1 + 1) * n + U - 1) / U - 1;
    for (int64_t b = b_lo; b <= b_hi && b <= n; ++b) {
      const int64_t u1 = b * U / n - 1;  // the unit tau_b - 1
      const int64_t r = u1 - W0 - pl.w_group;
      const int64_t cs = r < 0 ? c0 : c0 + r / pl.w_chunk;  // chunk covering u1
      pl.cta_start[b] = int32_t(cs + 1);
      // group holding chunk cs + 1: this one, or (at its end) the search starts at the next
      if (b < n) {
        pl.cta_group[b] = cs + 1 < c1 ? g : g + 1;
        int gh = g;
        if (cs + 1 >= c1) {  // the range starts at the next group with chunks
          gh = g + 1;
          while (gh < NG && pl.groups[gh + 1].c0 == pl.groups[gh].c0) ++gh;
        }
        write_head(pl, b, gh, cs + 1, NG);
      }
    }
  }
  __syncthreads();
  for (int64_t b = threadIdx.x; b < n; b += blockDim.x) pl.cta_head[b].ce = pl.cta_start[b + 1];
}

// Segment pass over sorted keys: perm, seg_start, seg_id, n_seg (and the attend plan).
// One CTA of 1024 threads walks the batch in tiles of 1024*kItems keys, carrying the
// segment count across tiles.
constexpr int kItems = 4;

__device__ void segment_pass(const uint64_t* keys, int64_t T, int32_t* perm,
                             int32_t* seg_start, int32_t* seg_id, int32_t* n_seg,
                             const PlanOut* plan, DevStatus* st, int* warp_tot, int* total) {
  if (!perm && !seg_start && !seg_id && !n_seg) return;  // (the many-CTA pass follows)
  int carry = 0;
  const int64_t tile = int64_t(blockDim.x) * kItems;
  for (int64_t base = 0; base < T; base += tile) {
    int flags[kItems];
    int cnt = 0;
#pragma unroll
    for (int u = 0; u < kItems; ++u) {
      int64_t q = base + int64_t(threadIdx.x) * kItems + u;
      flags[u] = 0;
      if (q < T) {
        uint64_t k = keys[q];
        flags[u] = (q == 0 || (keys[q - 1] >> 32) != (k >> 32)) ? 1 : 0;
        if (perm) perm[q] = int32_t(uint32_t(k));
      }
      cnt += flags[u];
    }
    int ex = block_exclusive_scan(cnt, warp_tot, total);
    int s = carry + ex;
#pragma unroll
    for (int u = 0; u < kItems; ++u) {
      int64_t q = base + int64_t(threadIdx.x) * kItems + u;
      if (flags[u]) {
        if (seg_start) seg_start[s] = int32_t(q);
        if (seg_id) seg_id[s] = int32_t(keys[q] >> 32);
        ++s;
      }
    }
    carry += *total;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    if (seg_start) seg_start[carry] = int32_t(T);
    if (n_seg) *n_seg = carry;
  }
  if (plan && seg_start) {
    __syncthreads();  // seg_start complete and visible to the whole CTA
    plan_pass(keys, T, seg_start, carry, *plan, st, warp_tot, total);
  }
}

__global__ void __launch_bounds__(1024) route_small_kernel(const int32_t* __restrict__ ids,
                                                           int64_t T, int64_t vocab,
                                                           uint64_t* keys_out, int32_t* perm,
                                                           int32_t* seg_start, int32_t* seg_id,
                                                           int32_t* n_seg, DevStatus* st,
                                                           const PlanOut plan, int with_plan) {
  __shared__ uint64_t s[kChunk];
  __shared__ int warp_tot[32];
  __shared__ int total;
  int n = 1;
  while (n < T) n <<= 1;
  for (int i = threadIdx.x; i < n; i += blockDim.x) s[i] = make_key(ids, T, vocab, i, st);
  __syncthreads();
  block_bitonic(s, n);
  for (int i = threadIdx.x; i < T; i += blockDim.x) keys_out[i] = s[i];
  __syncthreads();
  segment_pass(s, T, perm, seg_start, seg_id, n_seg, with_plan ? &plan : nullptr, st, warp_tot,
               &total);
}

// T <= kRankN: one CTA; each thread ranks its key among all keys of the batch (keys are
// unique, so the ranks are a permutation: the stable sort), then the segment and plan passes.
// One pass over shared memory instead of the radix passes' many CTA-wide barriers.
constexpr int kRankN = 256;
__global__ void __launch_bounds__(kRankN) route_rank_kernel(const int32_t* __restrict__ ids,
                                                            int64_t T, int64_t vocab,
                                                            uint64_t* keys_out, int32_t* perm,
                                                            int32_t* seg_start, int32_t* seg_id,
                                                            int32_t* n_seg, DevStatus* st,
                                                            const PlanOut plan, int with_plan) {
  grid_dep_release();  // as in the one-CTA radix kernel
  __shared__ uint64_t kin[kRankN], kout[kRankN];
  __shared__ int warp_tot[32];
  __shared__ int total;
  const int i = threadIdx.x;
  const uint64_t key = make_key(ids, T, vocab, i, st);  // all ones past the batch
  kin[i] = key;
  __syncthreads();
  if (i < T) {
    int r = 0;
    for (int j = 0; j < int(T); ++j) r += kin[j] < key ? 1 : 0;
    kout[r] = key;
    keys_out[r] = key;
  }
  __syncthreads();
  segment_pass(kout, T, perm, seg_start, seg_id, n_seg, with_plan ? &plan : nullptr, st, warp_tot,
               &total);
}

__global__ void __launch_bounds__(1024) route_chunk_kernel(const int32_t* __restrict__ ids,
                                                           int64_t T, int64_t vocab,
                                                           uint64_t* keys_out, DevStatus* st) {
  __shared__ uint64_t s[kChunk];
  const int64_t base = int64_t(blockIdx.x) * kChunk;
  for (int i = threadIdx.x; i < kChunk; i += blockDim.x) s[i] = make_key(ids, T, vocab, base + i, st);
  __syncthreads();
  block_bitonic(s, kChunk);
  for (int i = threadIdx.x; i < kChunk; i += blockDim.x)
    if (base + i < T) keys_out[base + i] = s[i];
}

// ---- one-CTA stable radix sort of up to 8192 ids ----------------------------------------------
//
// 32-bit keys (id << 13 | index within the CTA's block of 8192); an LSD radix sort on the
// id bits, 8 bits per pass, keeps equal ids in index order. Per pass each warp ranks its
// 256 keys in index order (warp w holds indices 256 w + 32 e + lane, e = 0..7) with
// __match_any_sync over the digit, a per-digit prefix over the 32 warps and a scan over the
// 256 digits place every key, and the keys are scattered to the other buffer.
constexpr int kRadixN = 8192;
constexpr int kIdxBits = 13;

struct RadixSmem {
  uint32_t buf[2][kRadixN];
  uint32_t cnt[32][256];
  uint32_t dstart[256];
  int warp_tot[32];
};

// Sorts buf[0][0 .. 256 nw) by key >> 13 (stable; warps nw .. 31 sit out: keys past the
// batch are all-ones and stay last, so the first T results never depend on them); returns
// the buffer that holds the result.
__device__ int block_radix_sort(RadixSmem& sm, int passes, int nw) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t lt = (1u << lane) - 1u;
  const bool active = warp < nw;
  int cur = 0;
  for (int p = 0; p < passes; ++p) {
    const int sh = kIdxBits + 8 * p;
    for (int i = tid; i < nw * 256; i += 1024) (&sm.cnt[0][0])[i] = 0;
    __syncthreads();
    uint32_t key[8];
    int dig[8], rank[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      if (!active) {
        key[e] = 0;
        dig[e] = rank[e] = 0;
        continue;
      }
      key[e] = sm.buf[cur][warp * 256 + e * 32 + lane];
      dig[e] = int((key[e] >> sh) & 255u);
      const uint32_t peers = __match_any_sync(0xffffffffu, dig[e]);
      const uint32_t before = sm.cnt[warp][dig[e]];
      rank[e] = int(before + __popc(peers & lt));
      __syncwarp();
      if ((peers & lt) == 0) sm.cnt[warp][dig[e]] = before + __popc(peers);  // lowest lane
      __syncwarp();
    }
    __syncthreads();
    int tot = 0, incl = 0;
    if (tid < 256) {
      uint32_t run = 0;
      for (int w = 0; w < nw; ++w) {
        const uint32_t c = sm.cnt[w][tid];
        sm.cnt[w][tid] = run;
        run += c;
      }
      tot = int(run);
      incl = tot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
      }
      if (lane == 31) sm.warp_tot[warp] = incl;
    }
    __syncthreads();
    if (tid < 256) {
      int off = 0;
      for (int w = 0; w < warp; ++w) off += sm.warp_tot[w];
      sm.dstart[tid] = uint32_t(off + incl - tot);
    }
    __syncthreads();
    if (active)
#pragma unroll
      for (int e = 0; e < 8; ++e)
        sm.buf[cur ^ 1][sm.dstart[dig[e]] + sm.cnt[warp][dig[e]] + rank[e]] = key[e];
    __syncthreads();
    cur ^= 1;
  }
  return cur;
}

// Keys of the block [base, base + 8192) of the batch: (id << 13 | local index); past T all
// bits set (they sort last). Ids outside [0, vocab) are reported and treated as id 0.
__device__ void radix_load(RadixSmem& sm, const int32_t* ids, int64_t T, int64_t vocab,
                           int64_t base, DevStatus* st, int n) {
#pragma unroll 8
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    uint32_t key = 0xffffffffu;
    if (base + i < T) {
      int32_t id = ids[base + i];
      if (id < 0 || int64_t(id) >= vocab) {
        atomicOr(&st->token_range, 1);
        id = 0;
      }
      key = (uint32_t(id) << kIdxBits) | uint32_t(i);
    }
    sm.buf[0][i] = key;
  }
  __syncthreads();
}

__device__ __forceinline__ uint64_t wide_key(uint32_t k, int64_t base) {
  return (uint64_t(k >> kIdxBits) << 32) | uint64_t(base + (k & (kRadixN - 1)));
}

// T <= 8192: sort, segments and plan in one CTA.
__global__ void __launch_bounds__(1024) route_radix_small_kernel(
    const int32_t* __restrict__ ids, int64_t T, int64_t vocab, int passes, uint64_t* keys_out,
    int32_t* perm, int32_t* seg_start, int32_t* seg_id, int32_t* n_seg, DevStatus* st,
    const PlanOut plan, int with_plan) {
  // the attend kernel that follows (launched as a programmatic dependent) may set up its CTAs
  // now; it reads nothing of this kernel's before this grid completes
  grid_dep_release();
  extern __shared__ __align__(16) unsigned char dyn[];
  RadixSmem& sm = *reinterpret_cast<RadixSmem*>(dyn);
  uint64_t* k64 = reinterpret_cast<uint64_t*>(dyn + sizeof(RadixSmem));
  __shared__ int warp_tot[32];
  __shared__ int total;
  const int nw = int((T + 255) / 256);  // warps holding keys of the batch
  radix_load(sm, ids, T, vocab, 0, st, 256 * nw);
  const int cur = block_radix_sort(sm, passes, nw);
  for (int i = threadIdx.x; i < T; i += blockDim.x) {
    const uint64_t k = wide_key(sm.buf[cur][i], 0);
    k64[i] = k;
    keys_out[i] = k;
  }
  __syncthreads();
  segment_pass(k64, T, perm, seg_start, seg_id, n_seg, with_plan ? &plan : nullptr, st, warp_tot,
               &total);
}

// T > 8192: each CTA sorts one block of 8192 keys (merged afterwards).
__global__ void __launch_bounds__(1024) route_radix_chunk_kernel(const int32_t* __restrict__ ids,
                                                                 int64_t T, int64_t vocab,
                                                                 int passes, uint64_t* keys_out,
                                                                 DevStatus* st) {
  extern __shared__ __align__(16) unsigned char dyn[];
  RadixSmem& sm = *reinterpret_cast<RadixSmem*>(dyn);
  const int64_t base = int64_t(blockIdx.x) * kRadixN;
  radix_load(sm, ids, T, vocab, base, st, kRadixN);
  const int cur = block_radix_sort(sm, passes, 32);
  for (int i = threadIdx.x; i < kRadixN; i += blockDim.x)
    if (base + i < T) keys_out[base + i] = wide_key(sm.buf[cur][i], base);
}

constexpr size_t kRadixSmallSmem = sizeof(RadixSmem) + kRadixN * sizeof(uint64_t);

// Number of keys in a[0..n) smaller than key (a sorted ascending).
__device__ inline int64_t lower_bound(const uint64_t* a, int64_t n, uint64_t key) {
  int64_t lo = 0, hi = n;
  while (lo < hi) {
    int64_t mid = (lo + hi) >> 1;
    if (a[mid] < key)
      lo = mid + 1;
    else
      hi = mid;
  }
  return lo;
}

// Merge sorted runs of width w pairwise: in -> out.
__global__ void route_merge_kernel(const uint64_t* __restrict__ in, uint64_t* __restrict__ out,
                                   int64_t T, int64_t w) {
  const int64_t p = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (p >= T) return;
  const int64_t L = p / (2 * w) * (2 * w);
  const int64_t mid = L + w < T ? L + w : T;
  const int64_t R = L + 2 * w < T ? L + 2 * w : T;
  const uint64_t key = in[p];
  int64_t rank;
  if (p < mid)
    rank = (p - L) + lower_bound(in + mid, R - mid, key);
  else
    rank = (p - mid) + lower_bound(in + L, mid - L, key);
  out[L + rank] = key;
}

__global__ void __launch_bounds__(1024) route_segment_kernel(const uint64_t* __restrict__ keys,
                                                             int64_t T, int32_t* perm,
                                                             int32_t* seg_start, int32_t* seg_id,
                                                             int32_t* n_seg, DevStatus* st,
                                                             const PlanOut plan, int with_plan) {
  grid_dep_release();  // as in the one-CTA routing kernel
  __shared__ int warp_tot[32];
  __shared__ int total;
  segment_pass(keys, T, perm, seg_start, seg_id, n_seg, with_plan ? &plan : nullptr, st,
               warp_tot, &total);
}

// ---- many-CTA segment and plan pass (batches above kRankN tokens with a work plan) ---------
//
// One cooperative launch of G CTAs (all co-resident) does what segment_pass and plan_pass
// do in one CTA, each step split over the CTAs and separated by grid barriers:
//   1. CTA b counts the segment starts in its contiguous share of the sorted keys;
//   2. it scans the CTAs' counts (each CTA itself), numbers its segments and writes
//      perm, seg_start, seg_id (CTA G-1 also seg_start[S] and n_seg);
//   3. it counts (groups, chunks, items, groups with chunks) of its share of the segments;
//   4. it scans those per CTA and writes its segments' groups and items, the whole CTA
//      sharing out each tile's groups (a segment of m tokens has m / 8 of them);
//   5. the cost-balanced split of the chunk list over the attend CTAs and their heads,
//      groups shared out over the CTAs as in the one-CTA pass;
//   6. the heads' range ends.
// The barriers are bounded: a CTA that waits too long records it (status word code
// 0x2000000) and stops.
constexpr int kCoopThreads = 1024;
constexpr int kCoopMaxCtas = 256;

struct CoopScratch {
  int32_t cnt[kCoopMaxCtas];
  int4 tot4[kCoopMaxCtas];
  unsigned bar;  // arrivals: zeroed before the launch, k G after the k-th barrier
};

size_t coop_scratch_bytes() { return align_up(sizeof(CoopScratch), kAlign); }

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ bool coop_barrier(CoopScratch* cs, unsigned target, DevStatus* st, int* s_ok) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(&cs->bar, 1u);
    const uint64_t t0 = tc::global_ns();
    int ok = 1;
    for (uint32_t i = 0;; ++i) {
      if (ld_acquire(&cs->bar) >= target) break;
      if ((i & 255) == 255 && tc::global_ns() - t0 > 1000000000ull) {
        atomicOr(&st->timeout, 0x2000000);
        ok = 0;
        break;
      }
    }
    __threadfence();
    *s_ok = ok;
  }
  __syncthreads();
  return *s_ok != 0;
}

// Sum of v[0 .. n) (n <= kCoopMaxCtas) below index `below`, and the total, by warp 0;
// returned to every thread through shared memory.
__device__ int2 coop_prefix(const int32_t* v, int n, int below, int2* sh) {
  if (threadIdx.x < 32) {
    int a = 0, t = 0;
    for (int i = threadIdx.x; i < n; i += 32) {
      const int x = __ldcg(v + i);
      t += x;
      if (i < below) a += x;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      a += __shfl_xor_sync(0xffffffffu, a, o);
      t += __shfl_xor_sync(0xffffffffu, t, o);
    }
    if (threadIdx.x == 0) *sh = make_int2(a, t);
  }
  __syncthreads();
  const int2 r = *sh;
  __syncthreads();
  return r;
}

__device__ void coop_prefix4(const int4* v, int n, int below, int4* sh_before, int4* sh_total) {
  if (threadIdx.x < 32) {
    int4 a = make_int4(0, 0, 0, 0), t = make_int4(0, 0, 0, 0);
    for (int i = threadIdx.x; i < n; i += 32) {
      const int4 x = __ldcg(v + i);
      t.x += x.x, t.y += x.y, t.z += x.z, t.w += x.w;
      if (i < below) a.x += x.x, a.y += x.y, a.z += x.z, a.w += x.w;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      a.x += __shfl_xor_sync(0xffffffffu, a.x, o);
      a.y += __shfl_xor_sync(0xffffffffu, a.y, o);
      a.z += __shfl_xor_sync(0xffffffffu, a.z, o);
      a.w += __shfl_xor_sync(0xffffffffu, a.w, o);
      t.x += __shfl_xor_sync(0xffffffffu, t.x, o);
      t.y += __shfl_xor_sync(0xffffffffu, t.y, o);
      t.z += __shfl_xor_sync(0xffffffffu, t.z, o);
      t.w += __shfl_xor_sync(0xffffffffu, t.w, o);
    }
    if (threadIdx.x == 0) {
      *sh_before = a;
      *sh_total = t;
    }
  }
  __syncthreads();
}

// A segment's share of the plan (as in plan_pass).
struct SegPlan {
  int q0, m, t, row0, n, per, ng, nc, ni, nw;
};
__device__ SegPlan seg_plan(const uint64_t* keys, const int32_t* seg_start, int s,
                            const PlanOut& pl, DevStatus* st) {
  SegPlan r{};
  r.q0 = seg_start[s];
  r.m = seg_start[s + 1] - r.q0;
  r.t = int(keys[r.q0] >> 32);
  r.row0 = pl.offs[r.t];
  r.n = pl.offs[r.t + 1] - r.row0;
  if (r.n < 1 || r.n > pl.k_max || r.row0 < 0 || int64_t(r.row0) + r.n > pl.v) {
    atomicOr(&st->layer_bad, 1);
    r.n = 0;
  }
  if (r.m >= pl.th) {
    r.ni = r.n > 0 ? (r.m + kTcNT - 1) / kTcNT : 0;
  } else {
    r.ng = (r.m + pl.mt_max - 1) / pl.mt_max;
    r.per = r.n > 0 ? (r.n + pl.ch - 1) / pl.ch : 0;
    r.nc = r.ng * r.per;
    r.nw = r.per > 0 ? r.ng : 0;
  }
  return r;
}

// Index i with off[i] <= x < off[i + 1] in the ascending off[0 .. n] (shared memory).
__device__ __forceinline__ int find_seg(const int* off, int n, int x) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (off[mid] <= x)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

struct CoopSmem {
  int warp_tot[32];
  int total;
  int4 wt4[32];
  int4 tot4;
  int4 before4, all4;
  int2 pre;
  int ok;
  // one tile of segments: exclusive offsets of its groups and items, and their fields
  int goff[kCoopThreads + 1], ioff[kCoopThreads + 1];
  int q0[kCoopThreads], m[kCoopThreads], t[kCoopThreads], row0[kCoopThreads], n[kCoopThreads];
  int per[kCoopThreads], cex[kCoopThreads], wex[kCoopThreads];
};

__global__ void __launch_bounds__(kCoopThreads, 1)
    route_plan_coop_kernel(const uint64_t* __restrict__ keys, int64_t T, int32_t* perm,
                           int32_t* seg_start, int32_t* seg_id, int32_t* n_seg, DevStatus* st,
                           const PlanOut pl, CoopScratch* cs) {
  grid_dep_release();
  __shared__ CoopSmem sm;
  const int G = gridDim.x, b = blockIdx.x, tid = threadIdx.x;
  // 1. segment starts in keys [k0, k1)
  const int64_t k0 = T * b / G, k1 = T * (b + 1) / G;
  constexpr int kPer = 4;
  int cnt = 0;
  for (int64_t q = k0 + tid; q < k1; q += kCoopThreads)
    cnt += (q == 0 || (keys[q - 1] >> 32) != (keys[q] >> 32)) ? 1 : 0;
  {
    const int ex = block_exclusive_scan(cnt, sm.warp_tot, &sm.total);
    (void)ex;
    if (tid == 0) cs->cnt[b] = sm.total;
  }
  if (!coop_barrier(cs, 1u * G, st, &sm.ok)) return;
  // 2. numbering: this CTA's first segment is the number of starts before k0
  const int2 pre = coop_prefix(cs->cnt, G, b, &sm.pre);
  const int S = pre.y;
  int carry = pre.x;
  for (int64_t base = k0; base < k1; base += int64_t(kCoopThreads) * kPer) {
    int flags[kPer], c = 0;
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int64_t q = base + int64_t(tid) * kPer + u;
      flags[u] = 0;
      if (q < k1) {
        const uint64_t k = keys[q];
        flags[u] = (q == 0 || (keys[q - 1] >> 32) != (k >> 32)) ? 1 : 0;
        if (perm) perm[q] = int32_t(uint32_t(k));
      }
      c += flags[u];
    }
    int s = carry + block_exclusive_scan(c, sm.warp_tot, &sm.total);
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int64_t q = base + int64_t(tid) * kPer + u;
      if (flags[u]) {
        seg_start[s] = int32_t(q);
        if (seg_id) seg_id[s] = int32_t(keys[q] >> 32);
        ++s;
      }
    }
    carry += sm.total;
    __syncthreads();
  }
  if (b == G - 1 && tid == 0) {
    seg_start[S] = int32_t(T);
    if (n_seg) *n_seg = S;
  }
  if (!coop_barrier(cs, 2u * G, st, &sm.ok)) return;
  // 3. plan counts of segments [s0, s1); when the CTA has at most kCoopThreads of them,
  // thread tid keeps its segment's plan for step 4
  const int s0 = int(int64_t(S) * b / G), s1 = int(int64_t(S) * (b + 1) / G);
  const bool one_tile = s1 - s0 <= kCoopThreads;
  SegPlan kept{};
  int4 mine = make_int4(0, 0, 0, 0);
  for (int s = s0 + tid; s < s1; s += kCoopThreads) {
    const SegPlan r = seg_plan(keys, seg_start, s, pl, st);
    mine.x += r.ng, mine.y += r.nc, mine.z += r.ni, mine.w += r.nw;
    kept = r;
  }
  {
    const int4 ex = block_exclusive_scan4(mine, sm.wt4, &sm.tot4);
    (void)ex;
    if (tid == 0) cs->tot4[b] = sm.tot4;
  }
  if (!coop_barrier(cs, 3u * G, st, &sm.ok)) return;
  // 4. groups and items of segments [s0, s1), one tile of kCoopThreads segments at a time
  coop_prefix4(cs->tot4, G, b, &sm.before4, &sm.all4);
  const int4 all = sm.all4;
  int4 run = sm.before4;  // (groups, chunks, items, groups with chunks) before the tile
  for (int base = s0; base < s1; base += kCoopThreads) {
    const int s = base + tid;
    SegPlan r{};
    if (s < s1) r = one_tile ? kept : seg_plan(keys, seg_start, s, pl, st);
    const int4 ex = block_exclusive_scan4(make_int4(r.ng, r.nc, r.ni, r.nw), sm.wt4, &sm.tot4);
    const int4 tt = sm.tot4;
    sm.goff[tid] = ex.x;
    sm.ioff[tid] = ex.z;
    sm.q0[tid] = r.q0;
    sm.m[tid] = r.m;
    sm.t[tid] = r.t;
    sm.row0[tid] = r.row0;
    sm.n[tid] = r.n;
    sm.per[tid] = r.per;
    sm.cex[tid] = ex.y;
    sm.wex[tid] = ex.w;
    if (tid == 0) {
      sm.goff[kCoopThreads] = tt.x;
      sm.ioff[kCoopThreads] = tt.z;
    }
    __syncthreads();
    const int nseg = s1 - base < kCoopThreads ? s1 - base : kCoopThreads;
    for (int gi = tid; gi < tt.x; gi += kCoopThreads) {
      const int i = find_seg(sm.goff, nseg, gi);
      const int k = gi - sm.goff[i];
      AttendGroup g;
      g.q0 = sm.q0[i] + k * pl.mt_max;
      g.mt = sm.m[i] - k * pl.mt_max < pl.mt_max ? sm.m[i] - k * pl.mt_max : pl.mt_max;
      g.t = sm.t[i];
      g.row0 = sm.row0[i];
      g.n = sm.n[i];
      g.c0 = run.y + sm.cex[i] + k * sm.per[i];
      g.w0 = g.c0 * pl.w_chunk + (run.w + sm.wex[i] + (sm.per[i] > 0 ? k : 0)) * pl.w_group;
      g.pad = 0;
#pragma unroll
      for (int j = 0; j < kPlanMT; ++j)
        g.tok[j] = j < g.mt ? int32_t(uint32_t(keys[g.q0 + j])) : 0;
      pl.groups[run.x + gi] = g;
      pl.counters[run.x + gi] = 0;
    }
    for (int ii = tid; ii < tt.z; ii += kCoopThreads) {
      int i = 0;
      {  // the segment of item ii
        int lo = 0, hi = nseg - 1;
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (sm.ioff[mid] <= ii)
            lo = mid;
          else
            hi = mid - 1;
        }
        i = lo;
      }
      const int k = ii - sm.ioff[i];
      AttendItem it;
      it.q0 = sm.q0[i] + k * kTcNT;
      it.nt = sm.m[i] - k * kTcNT < kTcNT ? sm.m[i] - k * kTcNT : kTcNT;
      it.t = sm.t[i];
      it.pad = 0;
      pl.items[run.z + ii] = it;
    }
    run.x += tt.x, run.y += tt.y, run.z += tt.z, run.w += tt.w;
    __syncthreads();
  }
  if (b == G - 1 && tid == 0) {
    AttendGroup end{};
    end.q0 = int32_t(T);
    end.c0 = all.y;
    end.w0 = all.y * pl.w_chunk + all.w * pl.w_group;
    pl.groups[all.x] = end;
    pl.hdr[kPlanGroups] = all.x;
    pl.hdr[kPlanChunks] = all.y;
    pl.hdr[kPlanItems] = all.z;
    pl.hdr[3] = 0;
  }
  if (!pl.cta_start) return;
  if (!coop_barrier(cs, 4u * G, st, &sm.ok)) return;
  // 5. the split (as in plan_pass), groups [NG b / G, NG (b + 1) / G) here
  const int NG = all.x;
  const int64_t C = all.y;
  const int64_t n = pl.n_cta;
  const int64_t U = C * pl.w_chunk + int64_t(all.w) * pl.w_group;
  if (U == 0) {
    for (int64_t bb = int64_t(b) * kCoopThreads + tid; bb <= n; bb += int64_t(G) * kCoopThreads) {
      pl.cta_start[bb] = 0;
      if (bb < n) {
        pl.cta_group[bb] = 0;
        pl.cta_head[bb] = CtaHead{};
      }
    }
    return;
  }
  if (b == 0) {
    const int64_t b_zero = (n + U - 1) / U;
    int g_first = 0;
    while (g_first < NG && pl.groups[g_first + 1].c0 == pl.groups[g_first].c0) ++g_first;
    for (int64_t bb = tid; bb < b_zero && bb <= n; bb += kCoopThreads) {
      pl.cta_start[bb] = 0;
      if (bb < n) {
        pl.cta_group[bb] = 0;
        write_head(pl, bb, g_first, 0, NG);
      }
    }
  }
  const int g0 = int(int64_t(NG) * b / G), g1 = int(int64_t(NG) * (b + 1) / G);
  for (int g = g0 + tid; g < g1; g += kCoopThreads) {
    const int64_t c0 = pl.groups[g].c0, c1 = pl.groups[g + 1].c0;
    if (c1 <= c0) continue;
    const int64_t W0 = pl.groups[g].w0;
    const int64_t W1 = W0 + pl.w_group + (c1 - c0) * pl.w_chunk;
    const int64_t b_lo = ((W0 + 1) * n + U - 1) / U;
    const int64_t b_hi = ((W1 + 1) * n + U - 1) / U - 1;
    for (int64_t bb = b_lo; bb <= b_hi && bb <= n; ++bb) {
      const int64_t u1 = bb * U / n - 1;
      const int64_t r = u1 - W0 - pl.w_group;
      const int64_t cs0 = r < 0 ? c0 : c0 + r / pl.w_chunk;
      pl.cta_start[bb] = int32_t(cs0 + 1);
      if (bb < n) {
        pl.cta_group[bb] = cs0 + 1 < c1 ? g : g + 1;
        int gh = g;
        if (cs0 + 1 >= c1) {
          gh = g + 1;
          while (gh < NG && pl.groups[gh + 1].c0 == pl.groups[gh].c0) ++gh;
        }
        write_head(pl, bb, gh, cs0 + 1, NG);
      }
    }
  }
  if (!coop_barrier(cs, 5u * G, st, &sm.ok)) return;
  // 6. the heads' range ends
  for (int64_t bb = int64_t(b) * kCoopThreads + tid; bb < n; bb += int64_t(G) * kCoopThreads)
    pl.cta_head[bb].ce = pl.cta_start[bb + 1];
}

}  // namespace

size_t route_scratch_bytes(int64_t T) {
  return 2 * align_up(size_t(T) * sizeof(uint64_t), kAlign) + coop_scratch_bytes();
}

// Sorted keys end up in the returned buffer (one of the two scratch halves). With a work plan
// and more than kRadixN tokens, the sort kernels only sort and the many-CTA pass
// (route_plan_coop_kernel) finds the segments and lays out the plan; smaller batches keep
// the sort, the segments and the plan in one CTA (a dependent global round trip costs a
// microsecond or two, which is about what a step of the one-CTA pass costs at that size).
cudaError_t launch_route(const int32_t* ids, int64_t T, int64_t vocab, void* scratch,
                         RouteOut out, DevStatus* st, cudaStream_t stream,
                         const uint64_t** sorted_keys, const PlanOut* plan) {
  const PlanOut pl = plan ? *plan : PlanOut{};
  const bool with_plan = plan && out.seg_start;
  const bool coop = with_plan && T > kRadixN;
  uint64_t* k0 = static_cast<uint64_t*>(scratch);
  uint64_t* k1 = reinterpret_cast<uint64_t*>(static_cast<char*>(scratch) +
                                             align_up(size_t(T) * sizeof(uint64_t), kAlign));
  if (T <= kRankN) {
    route_rank_kernel<<<1, kRankN, 0, stream>>>(ids, T, vocab, k0, out.perm, out.seg_start,
                                                out.seg_id, out.n_seg, st, pl, with_plan ? 1 : 0);
    count_launch();
    *sorted_keys = k0;
    return cudaGetLastError();
  }
  // the sort; the segments and the plan in the same kernels unless the many-CTA pass follows
  const RouteOut sort_out = coop ? RouteOut{nullptr, nullptr, nullptr, nullptr} : out;
  const int sort_plan = with_plan && !coop ? 1 : 0;
  const uint64_t* sorted = nullptr;
  // bits of the largest id; the radix path packs (id, index) into 32 bits
  int idbits = 1;
  while (idbits < 31 && (int64_t(1) << idbits) < vocab) ++idbits;
  if (idbits + kIdxBits <= 32) {
    const cudaError_t a1 = ensure_smem_attr(route_radix_small_kernel, int(kRadixSmallSmem));
    if (a1 != cudaSuccess) return a1;
    const cudaError_t a2 = ensure_smem_attr(route_radix_chunk_kernel, int(sizeof(RadixSmem)));
    if (a2 != cudaSuccess) return a2;
    const int passes = (idbits + 7) / 8;
    if (T <= kRadixN) {
      route_radix_small_kernel<<<1, 1024, kRadixSmallSmem, stream>>>(
          ids, T, vocab, passes, k0, sort_out.perm, sort_out.seg_start, sort_out.seg_id,
          sort_out.n_seg, st, pl, sort_plan);
      count_launch();
      sorted = k0;
    } else {
      const int64_t nblk = (T + kRadixN - 1) / kRadixN;
      route_radix_chunk_kernel<<<unsigned(nblk), 1024, sizeof(RadixSmem), stream>>>(
          ids, T, vocab, passes, k0, st);
      count_launch();
      uint64_t *src = k0, *dst = k1;
      for (int64_t w = kRadixN; w < T; w *= 2) {
        route_merge_kernel<<<unsigned((T + 255) / 256), 256, 0, stream>>>(src, dst, T, w);
        count_launch();
        uint64_t* t = src;
        src = dst;
        dst = t;
      }
      sorted = src;
      if (!coop) {
        route_segment_kernel<<<1, 1024, 0, stream>>>(src, T, out.perm, out.seg_start,
                                                     out.seg_id, out.n_seg, st, pl, sort_plan);
        count_launch();
      }
    }
  } else if (T <= kChunk) {
    route_small_kernel<<<1, 1024, 0, stream>>>(ids, T, vocab, k0, sort_out.perm,
                                               sort_out.seg_start, sort_out.seg_id,
                                               sort_out.n_seg, st, pl, sort_plan);
    count_launch();
    sorted = k0;
  } else {
    const int64_t nchunks = (T + kChunk - 1) / kChunk;
    route_chunk_kernel<<<unsigned(nchunks), 1024, 0, stream>>>(ids, T, vocab, k0, st);
    count_launch();
    uint64_t *src = k0, *dst = k1;
    for (int64_t w = kChunk; w < T; w *= 2) {
      route_merge_kernel<<<unsigned((T + 255) / 256), 256, 0, stream>>>(src, dst, T, w);
      count_launch();
      uint64_t* t = src;
      src = dst;
      dst = t;
    }
    sorted = src;
    if (!coop) {
      route_segment_kernel<<<1, 1024, 0, stream>>>(src, T, out.perm, out.seg_start, out.seg_id,
                                                   out.n_seg, st, pl, sort_plan);
      count_launch();
    }
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  *sorted_keys = sorted;
  if (!coop) return cudaSuccess;
  // the many-CTA segment and plan pass: one cooperative launch, its barrier counter zeroed
  CoopScratch* cs = reinterpret_cast<CoopScratch*>(
      static_cast<char*>(scratch) + 2 * align_up(size_t(T) * sizeof(uint64_t), kAlign));
  e = cudaMemsetAsync(&cs->bar, 0, sizeof(unsigned), stream);
  if (e != cudaSuccess) return e;
  int G = int((T + 511) / 512);
  const int sms = device_sm_count();
  if (G > sms) G = sms;
  if (G > kCoopMaxCtas) G = kCoopMaxCtas;
  if (G < 1) G = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(unsigned(G));
  cfg.blockDim = dim3(kCoopThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeCooperative;
  at[0].val.cooperative = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, route_plan_coop_kernel, sorted, T, out.perm, out.seg_start,
                         out.seg_id, out.n_seg, st, pl, cs);
  count_launch();
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace l3
