// Token frequencies of a stream of token ids ("L³: Large Lookup Layers", gist.science
// explainer, Technical Summary, "Information-Theoretic Embedding Allocation": rows are
// spread over the vocabulary by how often each token occurs). The counts feed
// l3_alloc_offsets_counts, which turns them into the CSR offsets of the static routing.
//
// The stream is HBM-bound (4 bytes per token read once). Token frequencies are heavy-
// tailed, so most occurrences hit a few ids: ids below kHead are counted per CTA in
// shared memory (one warp-aggregated atomic per distinct id in a warp) and added to the
// global counts once per CTA; the rare ids above go straight to global atomics, where they
// meet little contention. Integer atomics make the counts exact whatever the order.
#include "l3_internal.h"

namespace l3 {

namespace {

constexpr int kHead = 8192;  // ids counted in shared memory (32 KB)
constexpr int kCountThreads = 512;

__device__ __forceinline__ void count_one(int32_t t, int64_t vocab, int head, uint32_t* h,
                                          unsigned long long* counts, int& bad) {
  const bool ok = t >= 0 && int64_t(t) < vocab;
  if (!ok) bad = 1;
  // lanes with the same id count it once, with the number of lanes that hold it
  const int key = ok ? t : -1;
  const unsigned peers = __match_any_sync(__activemask(), key);
  const int lead = __ffs(peers) - 1;
  if (!ok || (threadIdx.x & 31) != lead) return;
  const uint32_t k = uint32_t(__popc(peers));
  if (t < head)
    atomicAdd(&h[t], k);
  else
    atomicAdd(&counts[t], static_cast<unsigned long long>(k));
}

__global__ void __launch_bounds__(kCountThreads) count_ids_kernel(
    const int32_t* __restrict__ ids, int64_t n, int64_t vocab, unsigned long long* counts,
    DevStatus* st) {
  __shared__ uint32_t h[kHead];
  const int head = vocab < kHead ? int(vocab) : kHead;
  for (int i = threadIdx.x; i < head; i += blockDim.x) h[i] = 0;
  __syncthreads();
  int bad = 0;
  // 16-byte loads over the aligned body, single loads for the ragged ends
  const uintptr_t addr = reinterpret_cast<uintptr_t>(ids);
  int64_t pre = int64_t(((16 - (addr & 15)) & 15) / 4);
  if (pre > n) pre = n;
  const int64_t body = (n - pre) / 4;
  const int4* v4 = reinterpret_cast<const int4*>(ids + pre);
  const int64_t stride = int64_t(gridDim.x) * blockDim.x;
  const int64_t start = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  // Every lane of a warp runs the same number of iterations (bounds rounded up to whole
  // warps), so __match_any_sync sees full warps; lanes past the end carry no id.
  const int64_t body_w = (body + 31) / 32 * 32;
  for (int64_t i = start; i < body_w; i += stride) {
    int4 q = make_int4(-1, -1, -1, -1);
    const bool in = i < body;
    if (in) q = __ldg(v4 + i);
    const int32_t e[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      int b2 = 0;
      count_one(in ? e[j] : -1, vocab, head, h, counts, b2);
      if (in) bad |= b2;
    }
  }
  const int64_t tail0 = pre + 4 * body;
  const int64_t rest = pre + (n - tail0);  // the unaligned head and the tail
  for (int64_t i = start; i < (rest + 31) / 32 * 32; i += stride) {
    const bool in = i < rest;
    const int64_t pos = i < pre ? i : tail0 + (i - pre);
    int b2 = 0;
    count_one(in ? ids[pos] : -1, vocab, head, h, counts, b2);
    if (in) bad |= b2;
  }
  if (bad) atomicOr(&st->token_range, 1);
  __syncthreads();
  for (int i = threadIdx.x; i < head; i += blockDim.x)
    if (h[i]) atomicAdd(&counts[i], static_cast<unsigned long long>(h[i]));
}

}  // namespace

cudaError_t launch_count_ids(const int32_t* ids, int64_t n, int64_t vocab, int64_t* counts,
                             DevStatus* st, cudaStream_t stream) {
  cudaError_t e = cudaMemsetAsync(counts, 0, size_t(vocab) * sizeof(int64_t), stream);
  if (e != cudaSuccess || n == 0) return e;
  // every CTA clears and flushes its shared histogram: enough CTAs to fill the SMs twice,
  // fewer when the stream is short
  int64_t grid = (n / 4 + kCountThreads - 1) / kCountThreads;
  const int64_t cap = int64_t(device_sm_count()) * 2;
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  count_ids_kernel<<<unsigned(grid), kCountThreads, 0, stream>>>(
      ids, n, vocab, reinterpret_cast<unsigned long long*>(counts), st);
  count_launch();
  return cudaGetLastError();
}

}  // namespace l3
