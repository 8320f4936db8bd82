// Staging of a batch's table rows from host memory into device memory, for tables too large
// to keep in HBM ("L³: Large Lookup Layers", gist.science explainer, Technical Summary,
// "Systems-Friendly Design": the tables can live in CPU memory, and because routing is
// static the rows a batch needs are known from its token ids alone, so they can be fetched
// ahead of the layer, for instance while earlier layers run).
//
// The batch is sorted by id; its S distinct ids become the ids 0 .. S-1 of a compact staged
// layer whose offsets are the prefix sums of their n_t, and each token's id is replaced by
// its segment index. The rows themselves are copied by warps reading the host-resident
// (pinned, device-mapped) tables directly, 16 bytes per lane with many loads in flight.
// The staged layer keeps the order of ids and their row counts, so the forward over it
// makes the same plan and computes the same values as over the full tables.
#include "l3_internal.h"

namespace l3 {

namespace {

constexpr int kStageThreads = 256;

// One CTA per segment s < S: the id's K and V rows to the staged tables at row seg_row0[s];
// the staged offsets, and the staged ids of the segment's tokens.
__global__ void __launch_bounds__(kStageThreads) stage_rows_kernel(
    const uint64_t* __restrict__ keys, const int32_t* __restrict__ seg_start,
    const int32_t* __restrict__ n_seg, const int32_t* __restrict__ offs,
    const int32_t* __restrict__ seg_row0, const unsigned char* __restrict__ K_host,
    const unsigned char* __restrict__ V_host, int64_t k_row_bytes, int64_t v_row_bytes,
    unsigned char* __restrict__ K_st, unsigned char* __restrict__ V_st, int64_t max_rows,
    int32_t* __restrict__ offs_st, int32_t* __restrict__ ids_st, DevStatus* st) {
  const int S = *n_seg;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int s = blockIdx.x; s < S; s += gridDim.x) {
    const int q0 = seg_start[s], q1 = seg_start[s + 1];
    const int t = int(keys[q0] >> 32);
    const int64_t r0 = offs[t];
    const int n = offs[t + 1] - int(r0);
    const int64_t o0 = seg_row0[s];
    if (threadIdx.x == 0) {
      offs_st[s] = int32_t(o0);
      if (s == S - 1) offs_st[S] = int32_t(o0 + n);
    }
    for (int q = q0 + int(threadIdx.x); q < q1; q += kStageThreads)
      ids_st[uint32_t(keys[q])] = s;
    if (o0 + n > max_rows) {
      if (threadIdx.x == 0) atomicOr(&st->capacity, 1);
      continue;
    }
    // rows of the segment, one warp per row; 16-byte pieces, four loads in flight per lane
    for (int j = warp; j < n; j += kStageThreads / 32) {
      const uint4* ks = reinterpret_cast<const uint4*>(K_host + (r0 + j) * k_row_bytes);
      uint4* kd = reinterpret_cast<uint4*>(K_st + (o0 + j) * k_row_bytes);
      const int kp = int(k_row_bytes / 16);
      for (int c = lane; c < kp; c += 128) {
        uint4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (c + 32 * u < kp) v[u] = ks[c + 32 * u];
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (c + 32 * u < kp) kd[c + 32 * u] = v[u];
      }
      const uint4* vs = reinterpret_cast<const uint4*>(V_host + (r0 + j) * v_row_bytes);
      uint4* vd = reinterpret_cast<uint4*>(V_st + (o0 + j) * v_row_bytes);
      const int vp = int(v_row_bytes / 16);
      for (int c = lane; c < vp; c += 32) vd[c] = vs[c];
    }
  }
}

// Offsets of the unused staged ids S+1 .. T: one row each past the staged rows, so that the
// staged offsets stay increasing (no token refers to those ids). The 128 rows after the
// staged ones are zeroed: the forward's copies of an id's last rows read whole boxes of up to
// 128 rows and mask the rows past the id, which must hold finite values.
__global__ void stage_tail_kernel(const int32_t* __restrict__ n_seg,
                                  const int32_t* __restrict__ n_rows, int32_t* offs_st,
                                  int64_t T, unsigned char* K_st, unsigned char* V_st,
                                  int64_t k_row_bytes, int64_t v_row_bytes, int64_t max_rows) {
  const int S = *n_seg;
  const int64_t U = *n_rows;
  const int64_t tid = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t nthr = int64_t(gridDim.x) * blockDim.x;
  for (int64_t u = S + 1 + tid; u <= T; u += nthr) offs_st[u] = int32_t(U + (u - S));
  const int64_t z1 = U + 128 < max_rows ? U + 128 : max_rows;
  if (U >= z1) return;
  const int64_t kq = (z1 - U) * k_row_bytes / 16, vq = (z1 - U) * v_row_bytes / 16;
  uint4* kz = reinterpret_cast<uint4*>(K_st + U * k_row_bytes);
  uint4* vz = reinterpret_cast<uint4*>(V_st + U * v_row_bytes);
  for (int64_t i = tid; i < kq; i += nthr) kz[i] = make_uint4(0, 0, 0, 0);
  for (int64_t i = tid; i < vq; i += nthr) vz[i] = make_uint4(0, 0, 0, 0);
}

}  // namespace

cudaError_t launch_stage_rows(const StageArgs& a, cudaStream_t stream) {
  unsigned grid = unsigned(a.T < int64_t(device_sm_count()) * 8 ? a.T : device_sm_count() * 8);
  if (grid < 1) grid = 1;
  stage_rows_kernel<<<grid, kStageThreads, 0, stream>>>(
      a.sorted_keys, a.seg_start, a.n_seg, a.offs, a.seg_row0,
      static_cast<const unsigned char*>(a.K_host), static_cast<const unsigned char*>(a.V_host),
      a.k_row_bytes, a.v_row_bytes, static_cast<unsigned char*>(a.K_st),
      static_cast<unsigned char*>(a.V_st), a.max_rows, a.offs_st, a.ids_st, a.st);
  count_launch();
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  stage_tail_kernel<<<256, 256, 0, stream>>>(a.n_seg, a.n_rows, a.offs_st, a.T,
                                             static_cast<unsigned char*>(a.K_st),
                                             static_cast<unsigned char*>(a.V_st), a.k_row_bytes,
                                             a.v_row_bytes, a.max_rows);
  count_launch();
  return cudaGetLastError();
}

}  // namespace l3
