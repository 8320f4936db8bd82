// Gather-attend forward on CUDA cores with the rows of every id split across the GPU:
//   for each token i with id t (rows R = offs[t] .. offs[t+1]-1):
//   s = K_R x_i,  p = softmax(s),  a_i = V_Rᵀ p
// ("L³: Large Lookup Layers", gist.science explainer, Technical Summary, "Core
// Architecture": context-dependent aggregation of the token's keys and values;
// "Systems-Friendly Design": the batch sorted by id, so the tokens of one id share its
// rows).
//
// Work: the routing pass cuts each segment of equal ids (every segment of a small batch;
// the short segments of a large bf16 batch, whose long ones go to the tensor-core kernel)
// into groups of at most 8 tokens and each group's n_t rows into chunks of `ch` rows (see
// PlanOut). The chunks of all groups form one list that the plan cuts into one contiguous
// range per persistent CTA (one per SM), of about equal cost, so a decode batch with a few
// dozen tokens still streams its rows with every SM.
//
// Per CTA: thread 0 keeps a ring of up to 4 stages in flight, each filled by two bulk
// copies (cp.async.bulk) of the chunk's contiguous K rows and V rows. Eight warps compute
// the chunk's scores (warp w: row w, all tokens of the group, x from shared memory), then
// an online (single-pass) softmax update: m' = max(m, max s), l' = l e^(m-m') + sum e^(s-m'),
// acc' = acc e^(m-m') + sum_r e^(s_r-m') V_r, all in fp32. When a group ends inside the
// CTA's range its tokens are finished there; otherwise the CTA writes its partial
// (m, l, acc), and the CTA whose chunks complete the group's count (an atomic counter, no
// waiting) merges the partials in CTA order, so results are deterministic.
// Every wait on a copy is bounded: on a timeout the CTA records it, waits (bounded) for the
// copies it issued and returns.
#include "l3_attend_split.cuh"

namespace l3 {

namespace {

using namespace split;

constexpr int kMaxCh = 8;
constexpr int kMaxStages = 4;
constexpr int kChunkBytes = 40960;  // K and V bytes per chunk (at most)

struct Misc {
  uint64_t full[kMaxStages];
  float s_buf[kMaxCh][kMT];
  float e_buf[kMaxCh][kMT];
  float m_run[2][kMT];
  float l_run[2][kMT];
  float scale[kMT];
  MergeSmem merge;
  int abort;
};

struct SplitShape {
  int ch;           // rows per chunk
  int stages;       // ring depth
  int stage_bytes;  // ch rows of K, then ch rows of V
  int x_bytes;      // kMT rows of x
  int smem;         // dynamic shared memory of the launch
};

int esize(int dtype) { return dtype == L3_BF16 ? 2 : 4; }

SplitShape split_shape(int d, int d_v, int dtype) {
  SplitShape s{};
  const int es = esize(dtype);
  s.ch = attend_rows_per_chunk(d, d_v, dtype);
  s.stage_bytes = int(align_up(size_t(s.ch) * size_t(d + d_v) * es, 128));
  s.x_bytes = kMT * d * es;
  const int fixed = 128 + s.x_bytes + int(align_up(sizeof(Misc), 128));
  s.stages = (kSmemLimit - fixed) / s.stage_bytes;
  if (s.stages > kMaxStages) s.stages = kMaxStages;
  s.smem = fixed + s.stages * s.stage_bytes;
  return s;
}

template <typename TE>
struct Vec;
template <>
struct Vec<float> {
  static constexpr int P = 4;  // elements per 16 bytes
  __device__ static inline void unpack(const uint4 v, float* o) {
    o[0] = __uint_as_float(v.x);
    o[1] = __uint_as_float(v.y);
    o[2] = __uint_as_float(v.z);
    o[3] = __uint_as_float(v.w);
  }
  __device__ static inline float2 pair(const float* p) { return *reinterpret_cast<const float2*>(p); }
};
template <>
struct Vec<__nv_bfloat16> {
  static constexpr int P = 8;
  __device__ static inline void unpack(const uint4 v, float* o) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      o[2 * j] = __uint_as_float(w[j] << 16);
      o[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
    }
  }
  __device__ static inline float2 pair(const __nv_bfloat16* p) {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(p);
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  }
};

template <typename TE>
__device__ __forceinline__ void store_pair(TE* dst, float v0, float v1);
template <>
__device__ __forceinline__ void store_pair<float>(float* dst, float v0, float v1) {
  *reinterpret_cast<float2*>(dst) = make_float2(v0, v1);
}
template <>
__device__ __forceinline__ void store_pair<__nv_bfloat16>(__nv_bfloat16* dst, float v0, float v1) {
  *reinterpret_cast<__nv_bfloat162*>(dst) = __floats2bfloat162_rn(v0, v1);
}

__device__ __forceinline__ void write_a2(const AttendArgs& a, int64_t i, int col, float v0,
                                         float v1) {
  if (a.a_f32) store_pair<float>(a.a_f32 + i * a.d_v + col, v0, v1);
  if (a.a_bf16) store_pair<__nv_bfloat16>(a.a_bf16 + i * a.d_v + col, v0, v1);
}

template <typename TE>
__global__ void __launch_bounds__(kThreads, 1) attend_split_kernel(const AttendArgs a,
                                                                  const SplitShape sh) {
  using Vt = Vec<TE>;
  constexpr int P = Vt::P;
  constexpr int ES = int(sizeof(TE));
  extern __shared__ unsigned char smem_raw[];
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  unsigned char* ring = base;
  TE* xt = reinterpret_cast<TE*>(base + sh.stages * sh.stage_bytes);
  Misc* ms = reinterpret_cast<Misc*>(base + sh.stages * sh.stage_bytes + sh.x_bytes);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.x;
  const int64_t cb = a.cta_start[b], ce = a.cta_start[b + 1];
  if (cb >= ce) return;
  const int nk = int(ce - cb);
  const int d = a.d, dv = a.d_v, ch = sh.ch, S = sh.stages;
  const int npk = d / P;  // 16-byte pieces of a K or x row
  const TE* __restrict__ Kg = static_cast<const TE*>(a.K);
  const TE* __restrict__ Vg = static_cast<const TE*>(a.V);
  const TE* __restrict__ Xg = static_cast<const TE*>(a.x);
  const AttendGroup* __restrict__ groups = a.groups;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) tc::mbar_init(&ms->full[s], 1);
    ms->abort = 0;
    tc::fence_barrier_init();
  }
  tc::fence_proxy_async();
  __syncthreads();

  // Producer state (thread 0): next chunk to issue and its group.
  int issued = 0;
  int pg = a.cta_group[b];
  auto issue = [&](int k) {
    const int64_t c = cb + k;
    while (groups[pg + 1].c0 <= c) ++pg;
    const AttendGroup g = groups[pg];
    const int j = int(c - g.c0);
    const int r0 = g.row0 + j * ch;
    const int nr = g.n - j * ch < ch ? g.n - j * ch : ch;
    unsigned char* st = ring + (k % S) * sh.stage_bytes;
    tc::mbar_arrive_expect_tx(&ms->full[k % S], uint32_t(nr) * uint32_t(d + dv) * ES);
    bulk_load(st, Kg + int64_t(r0) * d, uint32_t(nr) * d * ES, &ms->full[k % S]);
    bulk_load(st + ch * d * ES, Vg + int64_t(r0) * dv, uint32_t(nr) * dv * ES, &ms->full[k % S]);
  };
  if (tid == 0) {
    for (; issued < S - 1 && issued < nk; ++issued) issue(issued);
  }

  const bool col_ok = 2 * tid < dv;
  const int col = 2 * tid;
  float acc[kMT][2];
  int cg = -1, q0 = 0, mt = 0;
  bool ok = true;
  int k = 0;

  // Finish the current group: final outputs if the whole group lay in this CTA's range,
  // else a partial and, for the last CTA of the group, the merge of all partials.
  auto finish = [&](int par) {
    const int64_t c0 = groups[cg].c0, c1 = groups[cg + 1].c0;
    if (c0 >= cb && c1 <= ce) {
#pragma unroll
      for (int j = 0; j < kMT; ++j) {
        if (j >= mt) break;
        const int64_t i = int64_t(uint32_t(a.sorted_keys[q0 + j]));
        const float inv = 1.f / ms->l_run[par][j];
        if (col_ok) write_a2(a, i, col, acc[j][0] * inv, acc[j][1] * inv);
        if (a.ml && tid == 0) {
          a.ml[2 * i] = ms->m_run[par][j];
          a.ml[2 * i + 1] = ms->l_run[par][j];
        }
      }
      return;
    }
    const bool second = c0 > cb;
#pragma unroll
    for (int j = 0; j < kMT; ++j) {
      if (j >= mt) break;
      float* pe = part_entry(a, b, second, j);
      if (col_ok) *reinterpret_cast<float2*>(pe + 2 + col) = make_float2(acc[j][0], acc[j][1]);
      if (tid == 0) {
        pe[0] = ms->m_run[par][j];
        pe[1] = ms->l_run[par][j];
      }
    }
    arrive_and_merge(a, cg, c0, c1, cb, ce, q0, mt, &ms->merge, int(threadIdx.x), kThreads,
                     [] { __syncthreads(); });
  };

  for (; k < nk; ++k) {
    if (tid == 0 && issued < nk) {
      tc::fence_proxy_async();  // the stage refilled here was last read by generic loads
      issue(issued++);
    }
    const int64_t c = cb + k;
    int g = cg < 0 ? a.cta_group[b] : cg;
    while (groups[g + 1].c0 <= c) ++g;
    if (g != cg) {
      if (cg >= 0) {
        finish(k & 1);
        __syncthreads();
      }
      cg = g;
      q0 = groups[g].q0;
      mt = groups[g].mt;
      // x rows of the group's tokens into shared memory
      for (int idx = tid; idx < mt * npk; idx += kThreads) {
        const int j = idx / npk, pc = idx % npk;
        const int64_t i = int64_t(uint32_t(a.sorted_keys[q0 + j]));
        reinterpret_cast<uint4*>(xt + j * d)[pc] =
            __ldg(reinterpret_cast<const uint4*>(Xg + i * d) + pc);
      }
#pragma unroll
      for (int j = 0; j < kMT; ++j) acc[j][0] = acc[j][1] = 0.f;
      if (tid < kMT) {
        ms->m_run[k & 1][tid] = -INFINITY;
        ms->l_run[k & 1][tid] = 0.f;
      }
      __syncthreads();
    }
    const AttendGroup gr = groups[g];
    const int j0 = int(c - gr.c0);
    const int nr = gr.n - j0 * ch < ch ? gr.n - j0 * ch : ch;

    volatile int* abort_flag = &ms->abort;
    const bool got = tc::mbar_wait(&ms->full[k % S], (k / S) & 1, abort_flag, a.st, 0x10000);
    if (!__syncthreads_and(got ? 1 : 0)) {
      ok = false;
      break;
    }
    const unsigned char* stg = ring + (k % S) * sh.stage_bytes;
    const TE* Kc = reinterpret_cast<const TE*>(stg);
    const TE* Vc = reinterpret_cast<const TE*>(stg + ch * d * ES);

    // scores: warp w takes row w of the chunk for every token of the group
    if (warp < nr) {
      float sacc[kMT];
#pragma unroll
      for (int j = 0; j < kMT; ++j) sacc[j] = 0.f;
      const uint4* krow = reinterpret_cast<const uint4*>(Kc + warp * d);
      for (int pc = lane; pc < npk; pc += 32) {
        float kv[P];
        Vt::unpack(krow[pc], kv);
#pragma unroll
        for (int j = 0; j < kMT; ++j) {
          if (j < mt) {
            float xv[P];
            Vt::unpack(reinterpret_cast<const uint4*>(xt + j * d)[pc], xv);
#pragma unroll
            for (int e = 0; e < P; ++e) sacc[j] = fmaf(kv[e], xv[e], sacc[j]);
          }
        }
      }
#pragma unroll
      for (int j = 0; j < kMT; ++j) {
        if (j < mt) {
          const float sj = warp_sum(sacc[j]);
          if (lane == 0) ms->s_buf[warp][j] = sj;
        }
      }
    }
    __syncthreads();
    // softmax update of the running (m, l) and the chunk's weights e
    const int par = k & 1;
    if (tid < ch * kMT) {
      const int r = tid / kMT, j = tid % kMT;
      if (j < mt) {
        const float mo = ms->m_run[par][j];
        float mx = -INFINITY;
        for (int rr = 0; rr < nr; ++rr) mx = fmaxf(mx, ms->s_buf[rr][j]);
        const float mn = fmaxf(mo, mx);
        ms->e_buf[r][j] = r < nr ? expf(ms->s_buf[r][j] - mn) : 0.f;
        if (r == 0) {
          const float sc = expf(mo - mn);
          float sum = 0.f;
          for (int rr = 0; rr < nr; ++rr) sum += expf(ms->s_buf[rr][j] - mn);
          ms->scale[j] = sc;
          ms->m_run[par ^ 1][j] = mn;
          ms->l_run[par ^ 1][j] = fmaf(ms->l_run[par][j], sc, sum);
        }
      }
    }
    __syncthreads();
    // acc = acc * scale + sum_r e_r V_r (two value columns per thread)
    if (col_ok) {
#pragma unroll
      for (int j = 0; j < kMT; ++j) {
        if (j >= mt) break;
        float v0 = acc[j][0] * ms->scale[j], v1 = acc[j][1] * ms->scale[j];
        for (int r = 0; r < nr; ++r) {
          const float e = ms->e_buf[r][j];
          const float2 vv = Vt::pair(Vc + r * dv + col);
          v0 = fmaf(e, vv.x, v0);
          v1 = fmaf(e, vv.y, v1);
        }
        acc[j][0] = v0;
        acc[j][1] = v1;
      }
    }
    __syncthreads();  // the stage and the score buffers are free again
  }

  if (ok) {
    if (cg >= 0) finish(nk & 1);
  } else if (tid == 0) {
    // Let the copies still in flight land before the CTA's shared memory goes away.
    volatile int no_abort = 0;
    for (int j = k; j < issued; ++j)
      tc::mbar_wait(&ms->full[j % S], (j / S) & 1, &no_abort, a.st, 0x20000, 100000000ull);
  }
}

template <typename TE>
cudaError_t launch_split(const AttendArgs& a, cudaStream_t stream) {
  const SplitShape sh = split_shape(a.d, a.d_v, a.dtype);
  if (sh.stages < 2 || sh.ch != a.ch) return cudaErrorInvalidValue;
  const cudaError_t attr = ensure_smem_attr(attend_split_kernel<TE>, kSmemLimit);
  if (attr != cudaSuccess) return attr;
  if (a.n_cta < 1 || a.n_cta > kMaxCtas) return cudaErrorInvalidValue;
  attend_split_kernel<TE><<<a.n_cta, kThreads, sh.smem, stream>>>(a, sh);
  count_launch();
  return cudaGetLastError();
}

}  // namespace

namespace split {
int sm_count() { return device_sm_count(); }
}  // namespace split

cudaError_t launch_attend_mma(const AttendArgs& a, cudaStream_t stream);
int attend_mma_ctas(int d, int d_v);

int attend_split_ctas(int d, int d_v, int dtype) {
  if (dtype == L3_BF16) return attend_mma_ctas(d, d_v);
  return sm_count() < kMaxCtas ? sm_count() : kMaxCtas;
}

// Cost units of the plan's CTA split, in about 0.2 us of one CTA's time: a chunk, and the
// extra work of a group (its x rows, its outputs, and an unpaired last chunk). A group
// weighs relatively more where chunks are short (8 rows at the widest tables); the two
// settings were measured on the prefill presets (16-row chunks: 1 .. 5 tried, 3 best).
void attend_split_weights(int d, int d_v, int dtype, int* w_chunk, int* w_group) {
  *w_chunk = 4;
  *w_group = attend_rows_per_chunk(d, d_v, dtype) >= 16 ? 3 : 7;
}

int attend_group_tokens(int) { return kPlanMT; }

int attend_rows_per_chunk(int d, int d_v, int dtype) {
  if (dtype == L3_BF16) return attend_mma_rows_per_chunk(d, d_v);
  const int row = (d + d_v) * esize(dtype);
  int ch = kChunkBytes / row;
  if (ch > kMaxCh) ch = kMaxCh;
  return ch < 1 ? 1 : ch;
}

size_t attend_part_floats(int d_v) { return size_t(2 * kMaxCtas) * kMT * size_t(d_v + 2); }

cudaError_t launch_attend_fwd(const AttendArgs& a, cudaStream_t stream) {
  if (a.T <= 0) return cudaSuccess;
  return a.dtype == L3_BF16 ? launch_attend_mma(a, stream) : launch_split<float>(a, stream);
}

}  // namespace l3
