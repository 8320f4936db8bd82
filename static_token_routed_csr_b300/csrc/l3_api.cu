// C-ABI entry points of the L³ library: argument checks, workspace layout, and the order
// of the kernels for the forward pass, the backward pass and batch routing.
#include <atomic>
#include <climits>
#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

#include "l3_internal.h"

namespace l3 {

namespace {

std::atomic<uint64_t> g_launches{0};

// Bump allocator over a caller-provided buffer (base == nullptr: measure only).
struct Carve {
  char* base;
  size_t off = 0;
  explicit Carve(void* b) : base(static_cast<char*>(b)) {}
  template <typename T>
  T* take(size_t n) {
    off = align_up(off, kAlign);
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off += n * sizeof(T);
    return p;
  }
  char* raw(size_t bytes) { return take<char>(bytes); }
};

bool valid_dtype(int dt) { return dt == L3_F32 || dt == L3_BF16; }
size_t esize(int dt) { return dt == L3_BF16 ? 2 : 4; }

l3_status check_layer_args(const l3_layer* L) {
  if (!L) return L3_ERR_INVALID_ARG;
  if (!L->offs || !L->K || !L->V || !L->W_up || !L->W_mix) return L3_ERR_INVALID_ARG;
  if (!valid_dtype(L->dtype) || L->reserved != 0) return L3_ERR_INVALID_ARG;
  if (L->vocab < 1 || L->v < L->vocab || L->v >= (int64_t(1) << 31) ||
      L->vocab >= (int64_t(1) << 31))
    return L3_ERR_INVALID_ARG;
  if (!(L->ln_eps > 0.f) || !std::isfinite(L->ln_eps)) return L3_ERR_INVALID_ARG;
  if (L->k_max < 1 || L->k_max > 512) return L3_ERR_UNSUPPORTED;
  if (L->d < 64 || L->d > 2048 || L->d % 64 != 0) return L3_ERR_UNSUPPORTED;
  if (L->d_v < 64 || L->d_v > 512 || L->d_v % 64 != 0) return L3_ERR_UNSUPPORTED;
  if (L->v > L->vocab * int64_t(L->k_max)) return L3_ERR_INVALID_ARG;
  return L3_OK;
}

// ---- workspace layouts ------------------------------------------------------------------------

struct FwdWs {
  DevStatus* st;
  void* route_scratch;
  int32_t *perm, *seg_start, *seg_id, *n_seg;
  float* part;
  AttendGroup* groups;
  int32_t* plan_hdr;
  int32_t* counters;
  int32_t* cta_start;  // the plan's split of the chunk list over the split-row kernel's CTAs
  int32_t* cta_group;
  CtaHead* cta_head;
  int n_cta;
  AttendItem* items;
  float* a_f32;
  __nv_bfloat16* a_bf16;
  // fp32 layers (CUDA-core GEMMs)
  float* U;
  float* mu;
  float* rstd;
  float* H;
  // bf16 layers (tensor-core GEMMs)
  __nv_bfloat16* U16;
  float* stats;
  float* colsum;
  float* slab;  // split-K parts of the GEMMs (decode-sized batches)
  size_t slab_floats;
  // small batches (T <= 64): warp-MMA GEMMs with their own statistics and halves
  bool small;
  uint32_t* sync;  // arrival counters, zeroed with the status words
  float *q_stats, *q_slab;
  // tensor-core gather-attend of the long segments
  int tc_th;      // segments with at least this many tokens go to tensor cores (0: none)
  int max_items;  // bound on their item count
};

FwdWs carve_fwd(Carve& c, const l3_layer* L, int64_t T) {
  FwdWs w{};
  const size_t t = size_t(T), d = size_t(L->d), dv = size_t(L->d_v);
  w.st = c.take<DevStatus>(1);
  w.sync = c.take<uint32_t>(size_t(kSyncWords));  // zeroed with the status words
  w.route_scratch = c.raw(route_scratch_bytes(T));
  w.perm = c.take<int32_t>(t);
  w.seg_start = c.take<int32_t>(t + 1);
  w.seg_id = c.take<int32_t>(t);
  w.n_seg = c.take<int32_t>(1);
  w.mu = c.take<float>(t);
  w.rstd = c.take<float>(t);
  w.part = c.take<float>(attend_part_floats(int(dv)));
  w.groups = c.take<AttendGroup>(t + 1);
  w.plan_hdr = c.take<int32_t>(kPlanHdrWords);
  w.counters = c.take<int32_t>(t);
  w.n_cta = attend_split_ctas(int(d), int(dv), L->dtype);
  w.cta_start = c.take<int32_t>(size_t(kPlanMaxCtas) + 1);
  w.cta_group = c.take<int32_t>(size_t(kPlanMaxCtas));
  w.cta_head = c.take<CtaHead>(size_t(kPlanMaxCtas));
  w.tc_th = attend_tc_threshold(T, int(d), int(dv), L->dtype);
  if (w.tc_th > 0) {
    w.max_items = int(T / w.tc_th + 1);
    w.items = c.take<AttendItem>(size_t(w.max_items));
  }
  if (L->dtype == L3_BF16) {
    w.a_bf16 = c.take<__nv_bfloat16>(t * dv);
    w.U16 = c.take<__nv_bfloat16>(t * d);
    w.small = small_gemm_fits(T, int(d), int(dv));
    if (w.small) {
      w.q_stats = c.take<float>(d / 32 * 64 * 2);
      w.q_slab = c.take<float>(d * 128);
      w.colsum = c.take<float>(d);
    } else {
      w.stats = c.take<float>(size_t(tc_up_stat_tiles(int(d))) * t * 2);
      w.colsum = c.take<float>(d);
      w.slab_floats = tc_splitk_floats(T, int(d), int(dv));
      if (w.slab_floats) w.slab = c.take<float>(w.slab_floats);
    }
  } else {
    w.a_f32 = c.take<float>(t * dv);
    w.U = c.take<float>(t * d);
    w.H = c.take<float>(t * d);
  }
  return w;
}

struct Saved {
  float* a;     // [T, d_v]
  float* ml;    // [T, 2]
  float* mu;    // [T]
  float* rstd;  // [T]
};

Saved carve_saved(Carve& c, const l3_layer* L, int64_t T) {
  Saved s{};
  s.a = c.take<float>(size_t(T) * size_t(L->d_v));
  s.ml = c.take<float>(size_t(T) * 2);
  s.mu = c.take<float>(size_t(T));
  s.rstd = c.take<float>(size_t(T));
  return s;
}

struct BwdWs {
  DevStatus* st;
  void* route_scratch;
  int32_t *seg_start, *n_seg;
  float *U, *H, *mu, *rstd, *dC, *du, *dA, *p_buf, *ds_buf;
};

BwdWs carve_bwd(Carve& c, const l3_layer* L, int64_t T) {
  BwdWs w{};
  const size_t t = size_t(T), d = size_t(L->d), dv = size_t(L->d_v);
  w.st = c.take<DevStatus>(1);
  w.route_scratch = c.raw(route_scratch_bytes(T));
  w.seg_start = c.take<int32_t>(t + 1);
  w.n_seg = c.take<int32_t>(1);
  w.U = c.take<float>(t * d);
  w.H = c.take<float>(t * d);
  w.mu = c.take<float>(t);
  w.rstd = c.take<float>(t);
  w.dC = c.take<float>(t * 2 * d);
  w.du = c.take<float>(t * d);
  w.dA = c.take<float>(t * dv);
  w.p_buf = c.take<float>(t * size_t(L->k_max));
  w.ds_buf = c.take<float>(t * size_t(L->k_max));
  return w;
}

struct BwdRowsWs {
  DevStatus* st;
  void* route_scratch;
  int32_t *seg_start, *n_seg;
  AttendGroup* groups;
  int32_t* hdr;
  int32_t* counters;
  __nv_bfloat16 *a_hi, *a_lo, *h16, *du_hi, *du_lo, *x_sorted, *da16, *da16_lo;
  float *U32, *rstd, *dh, *da, *delta, *p_buf, *ds_buf;
  int32_t *seg_row0, *seg_unit0;
  int64_t* seg_cost0;
  void* lt_ws;
};

BwdRowsWs carve_bwd_rows(Carve& c, const l3_layer* L, int64_t T) {
  BwdRowsWs w{};
  const size_t t = size_t(T), d = size_t(L->d), dv = size_t(L->d_v), km = size_t(L->k_max);
  w.st = c.take<DevStatus>(1);
  w.route_scratch = c.raw(route_scratch_bytes(T));
  w.seg_start = c.take<int32_t>(t + 1);
  w.n_seg = c.take<int32_t>(1);
  w.groups = c.take<AttendGroup>(t + 1);
  w.hdr = c.take<int32_t>(kPlanHdrWords);
  w.counters = c.take<int32_t>(t + 1);
  w.a_hi = c.take<__nv_bfloat16>(t * dv);
  w.a_lo = c.take<__nv_bfloat16>(t * dv);
  w.h16 = c.take<__nv_bfloat16>(t * d);
  w.du_hi = c.take<__nv_bfloat16>(t * d);
  w.du_lo = c.take<__nv_bfloat16>(t * d);
  w.x_sorted = c.take<__nv_bfloat16>(t * d);
  w.da16 = c.take<__nv_bfloat16>(t * dv);
  w.da16_lo = c.take<__nv_bfloat16>(t * dv);
  w.U32 = c.take<float>(t * d);
  w.rstd = c.take<float>(t);
  w.dh = c.take<float>(t * d);
  w.da = c.take<float>(t * dv);
  w.delta = c.take<float>(t);
  w.p_buf = c.take<float>(t * km);
  w.ds_buf = c.take<float>(t * km);
  w.seg_row0 = c.take<int32_t>(t + 1);
  w.seg_unit0 = c.take<int32_t>(t + 1);
  w.seg_cost0 = c.take<int64_t>(t + 1);
  w.lt_ws = c.raw(kLtWorkspace);
  return w;
}

#define L3_CUDA(call)                      \
  do {                                     \
    if ((call) != cudaSuccess) {           \
      (void)cudaGetLastError();            \
      return L3_ERR_CUDA;                  \
    }                                      \
  } while (0)

// Stage boundary event. Under stream capture the event becomes an event-record node of
// the graph (cudaEventRecordExternal), so graph replays time their stages too.
cudaError_t record_stage(cudaEvent_t ev, cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(s, &cs);
  if (e != cudaSuccess) return e;
  return cs == cudaStreamCaptureStatusActive
             ? cudaEventRecordWithFlags(ev, s, cudaEventRecordExternal)
             : cudaEventRecord(ev, s);
}

__global__ void check_offsets_kernel(const int32_t* __restrict__ offs, int64_t vocab, int64_t v,
                                     int k_max, DevStatus* st) {
  for (int64_t t = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; t < vocab;
       t += int64_t(gridDim.x) * blockDim.x) {
    const int64_t a = offs[t], b = offs[t + 1];
    bool bad = !(b > a) || (b - a) > k_max;
    if (t == 0 && a != 0) bad = true;
    if (t == vocab - 1 && b != v) bad = true;
    if (bad) atomicOr(&st->layer_bad, 1);
  }
}

l3_status forward_impl(const l3_layer* L, const int32_t* ids, int64_t T, const void* x, void* y,
                       int32_t y_dtype, void* saved, void* ws, size_t ws_bytes,
                       cudaStream_t s, cudaEvent_t* ev) {
  l3_status e = check_layer_args(L);
  if (e != L3_OK) return e;
  if (T < 0 || T >= (int64_t(1) << 31)) return L3_ERR_INVALID_ARG;
  if (!(y_dtype == L3_F32 || y_dtype == L->dtype)) return L3_ERR_INVALID_ARG;
  if (T > 0 && (!ids || !x || !y || !ws)) return L3_ERR_INVALID_ARG;
  // x and y rows move through TMA tensor copies, whose global addresses are 16-byte aligned
  if (((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) & 15) != 0)
    return L3_ERR_INVALID_ARG;
  if (ws_bytes < l3_workspace_size(L, T, L3_PASS_FORWARD)) return L3_ERR_WORKSPACE;
  if (T == 0) return L3_OK;

  Carve c(ws);
  FwdWs w = carve_fwd(c, L, T);
  Saved sv{};
  if (saved) {
    Carve cs(saved);
    sv = carve_saved(cs, L, T);
  }
  float* a_f32 = saved ? sv.a : w.a_f32;
  float* mu = saved ? sv.mu : w.mu;
  float* rstd = saved ? sv.rstd : w.rstd;
  const int d = int(L->d), dv = int(L->d_v);

  // the status words and the arrival counters (one zeroing of the workspace's head)
  L3_CUDA(cudaMemsetAsync(w.st, 0,
                          size_t(reinterpret_cast<char*>(w.sync + kSyncWords) -
                                 reinterpret_cast<char*>(w.st)),
                          s));
  if (ev) L3_CUDA(record_stage(ev[L3_STAGE_ROUTE], s));
  const uint64_t* keys = nullptr;
  const int ch = attend_rows_per_chunk(d, dv, L->dtype);
  PlanOut plan{w.groups, w.plan_hdr, w.counters, w.items, L->offs, L->v, L->k_max, ch,
               attend_group_tokens(L->dtype), w.tc_th > 0 ? w.tc_th : INT32_MAX,
               w.cta_start, w.cta_group, w.cta_head, w.n_cta, 0, 0};
  attend_split_weights(d, dv, L->dtype, &plan.w_chunk, &plan.w_group);
  L3_CUDA(launch_route(ids, T, L->vocab, w.route_scratch,
                       RouteOut{w.perm, w.seg_start, w.seg_id, w.n_seg}, w.st, s, &keys, &plan));

  if (ev) L3_CUDA(record_stage(ev[L3_STAGE_ATTEND], s));
  float* a_copy = (L->dtype == L3_F32 || saved) ? a_f32 : nullptr;  // fp32 copy for backward
  float* ml = saved ? sv.ml : nullptr;
  {
    AttendArgs aa{};
    aa.sorted_keys = keys;
    aa.T = T;
    aa.groups = w.groups;
    aa.hdr = w.plan_hdr;
    aa.counters = w.counters;
    aa.K = L->K;
    aa.V = L->V;
    aa.x = x;
    aa.v = L->v;
    aa.d = d;
    aa.d_v = dv;
    aa.ch = ch;
    aa.dtype = L->dtype;
    aa.a_f32 = a_copy;
    aa.a_bf16 = w.a_bf16;
    aa.ml = ml;
    aa.part = w.part;
    aa.cta_start = w.cta_start;
    aa.cta_group = w.cta_group;
    aa.cta_head = w.cta_head;
    aa.n_cta = w.n_cta;
    aa.st = w.st;
    L3_CUDA(launch_attend_fwd(aa, s));
  }
  if (ev) L3_CUDA(record_stage(ev[L3_STAGE_ATTEND_LONG], s));
  if (w.tc_th > 0) {
    AttendTcArgs at{};
    at.sorted_keys = keys;
    at.items = w.items;
    at.hdr = w.plan_hdr;
    at.max_items = w.max_items;
    at.T = T;
    at.offs = L->offs;
    at.K = L->K;
    at.V = L->V;
    at.x = x;
    at.v = L->v;
    at.d = d;
    at.d_v = dv;
    at.a_bf16 = w.a_bf16;
    at.a_f32 = a_copy;
    at.ml = ml;
    at.st = w.st;
    L3_CUDA(launch_attend_tc(at, s));
  }

  if (ev) L3_CUDA(record_stage(ev[L3_STAGE_UP], s));
  if (L->dtype == L3_BF16 && w.small) {
    // small batch: weight-streaming warp-MMA GEMMs
    SmallGemmArgs g{};
    g.T = T;
    g.d = d;
    g.d_v = dv;
    g.eps = L->ln_eps;
    g.a = w.a_bf16;
    g.W_up = static_cast<const __nv_bfloat16*>(L->W_up);
    g.W_mix = static_cast<const __nv_bfloat16*>(L->W_mix);
    g.x = static_cast<const __nv_bfloat16*>(x);
    g.U = w.U16;
    g.tile_stats = w.q_stats;
    g.mu_out = saved ? sv.mu : nullptr;
    g.rstd_out = saved ? sv.rstd : nullptr;
    g.slab = w.q_slab;
    g.colsum = w.colsum;
    g.counters = w.sync;
    g.Y = y;
    g.y_dtype = y_dtype;
    g.st = w.st;
    L3_CUDA(launch_small_up(g, s));
    if (ev) L3_CUDA(record_stage(ev[L3_STAGE_MIX], s));
    L3_CUDA(launch_small_mix(g, s));
    if (ev) L3_CUDA(record_stage(ev[L3_FWD_STAGES], s));
    return L3_OK;
  }
  if (L->dtype == L3_BF16) {
    // Tensor cores: U = bf16(A W_upᵀ) with partial LayerNorm statistics, then
    // y = rstd (U W1ᵀ - mu c) + x W2ᵀ with the statistics merged in the epilogue.
    const auto* Wmix = static_cast<const __nv_bfloat16*>(L->W_mix);
    L3_CUDA(launch_tc_up(w.a_bf16, static_cast<const __nv_bfloat16*>(L->W_up), T, d, dv, w.U16,
                         w.stats, w.slab, w.slab_floats, Wmix, w.colsum, w.st, s));
    if (ev) L3_CUDA(record_stage(ev[L3_STAGE_MIX], s));
    L3_CUDA(launch_tc_mix(w.U16, static_cast<const __nv_bfloat16*>(x), Wmix, T, d, w.stats,
                          w.colsum, L->ln_eps, y, y_dtype, saved ? sv.mu : nullptr,
                          saved ? sv.rstd : nullptr, w.slab, w.slab_floats, w.st, s));
    if (ev) L3_CUDA(record_stage(ev[L3_FWD_STAGES], s));
    return L3_OK;
  }
  // fp32 layers: CUDA-core GEMMs (fp32 parity rules out tf32 tensor cores).
  // u = W_up a: U[i, n] = sum_k A[i, k] W_up[n, k]
  SimtGemm up{};
  up.M = T;
  up.N = d;
  up.K = dv;
  up.A = a_f32;
  up.a_dtype = L3_F32;
  up.a_sm = dv;
  up.a_sk = 1;
  up.B = L->W_up;
  up.b_dtype = L3_F32;
  up.b_sk = 1;
  up.b_sn = dv;
  up.C = w.U;
  up.ldc = d;
  up.alpha = 1.f;
  up.beta = 0.f;
  L3_CUDA(launch_simt_gemm(up, s));
  L3_CUDA(launch_ln_stats(w.U, T, d, L->ln_eps, mu, rstd, s));

  if (ev) L3_CUDA(record_stage(ev[L3_STAGE_MIX], s));
  L3_CUDA(launch_ln_apply(w.U, mu, rstd, T, d, w.H, s));
  // y = W_mix[:, :d] h + W_mix[:, d:] x (fp32 y: y_dtype must be L3_F32 here)
  float* Y = static_cast<float*>(y);
  SimtGemm mix{};
  mix.M = T;
  mix.N = d;
  mix.K = d;
  mix.A = w.H;
  mix.a_dtype = L3_F32;
  mix.a_sm = d;
  mix.a_sk = 1;
  mix.B = L->W_mix;
  mix.b_dtype = L3_F32;
  mix.b_sk = 1;
  mix.b_sn = 2 * d;
  mix.C = Y;
  mix.ldc = d;
  mix.alpha = 1.f;
  mix.beta = 0.f;
  L3_CUDA(launch_simt_gemm(mix, s));
  mix.A = x;
  mix.B = static_cast<const float*>(L->W_mix) + d;
  mix.beta = 1.f;
  L3_CUDA(launch_simt_gemm(mix, s));
  if (ev) L3_CUDA(record_stage(ev[L3_FWD_STAGES], s));
  return L3_OK;
}

}  // namespace

void count_launch(int n) { g_launches.fetch_add(uint64_t(n), std::memory_order_relaxed); }

namespace {
struct SmemAttr {
  const void* kernel;
  int dev;
  int bytes;
};
std::mutex g_attr_mu;
std::vector<SmemAttr> g_attrs;
constexpr int kMaxDevices = 64;
int g_sms[kMaxDevices] = {};
}  // namespace

cudaError_t ensure_smem_attr(const void* kernel, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_attr_mu);
  for (const SmemAttr& a : g_attrs)
    if (a.kernel == kernel && a.dev == dev && a.bytes >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  g_attrs.push_back(SmemAttr{kernel, dev, bytes});
  return cudaSuccess;
}

int device_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
  int n = __atomic_load_n(&g_sms[dev], __ATOMIC_RELAXED);
  if (n > 0) return n;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    n = 148;
  __atomic_store_n(&g_sms[dev], n, __ATOMIC_RELAXED);
  return n;
}

cudaError_t launch_check_offsets(const int32_t* offs, int64_t vocab, int64_t v, int k_max,
                                 DevStatus* st, cudaStream_t stream) {
  int64_t blocks = (vocab + 255) / 256;
  if (blocks > 148 * 8) blocks = 148 * 8;
  check_offsets_kernel<<<unsigned(blocks), 256, 0, stream>>>(offs, vocab, v, k_max, st);
  count_launch();
  return cudaGetLastError();
}

}  // namespace l3

using namespace l3;

extern "C" {

size_t l3_workspace_size(const l3_layer* L, int64_t T, int32_t pass) {
  if (check_layer_args(L) != L3_OK || T < 0) return 0;
  Carve c(nullptr);
  if (pass == L3_PASS_FORWARD || pass == L3_PASS_FORWARD_HOST) {
    carve_fwd(c, L, T);
    if (pass == L3_PASS_FORWARD_HOST) {
      c.take<int32_t>(size_t(T));
      c.raw(size_t(T) * size_t(L->d) * esize(L->dtype));
      c.raw(size_t(T) * size_t(L->d) * 4);
    }
  } else if (pass == L3_PASS_BACKWARD) {
    carve_bwd(c, L, T);
  } else if (pass == L3_PASS_BACKWARD_ROWS) {
    carve_bwd_rows(c, L, T);
  } else if (pass == L3_PASS_STAGE) {
    c.take<DevStatus>(1);
    c.raw(route_scratch_bytes(T));
    for (int k = 0; k < 3; ++k) c.take<int32_t>(size_t(T) + 1);
    c.take<int32_t>(1);
    c.take<int64_t>(size_t(T) + 1);
  } else {
    return 0;
  }
  return align_up(c.off, kAlign);
}

size_t l3_saved_size(const l3_layer* L, int64_t T) {
  if (check_layer_args(L) != L3_OK || T < 0) return 0;
  Carve c(nullptr);
  carve_saved(c, L, T);
  return align_up(c.off, kAlign);
}

l3_status l3_check_layer(const l3_layer* L, void* ws, size_t ws_bytes, l3_stream_t stream) {
  l3_status e = check_layer_args(L);
  if (e != L3_OK) return e;
  if (!ws) return L3_ERR_INVALID_ARG;
  if (ws_bytes < l3_workspace_size(L, 0, L3_PASS_FORWARD)) return L3_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  DevStatus* st = static_cast<DevStatus*>(ws);
  L3_CUDA(cudaMemsetAsync(st, 0, sizeof(DevStatus), s));
  L3_CUDA(launch_check_offsets(L->offs, L->vocab, L->v, L->k_max, st, s));
  DevStatus h{};
  L3_CUDA(cudaMemcpyAsync(&h, st, sizeof(h), cudaMemcpyDeviceToHost, s));
  L3_CUDA(cudaStreamSynchronize(s));
  return h.layer_bad ? L3_ERR_LAYER : L3_OK;
}

l3_status l3_route(const l3_layer* L, const int32_t* ids, int64_t T, int32_t* perm,
                   int32_t* seg_start, int32_t* seg_id, int32_t* n_seg, void* ws,
                   size_t ws_bytes, l3_stream_t stream) {
  l3_status e = check_layer_args(L);
  if (e != L3_OK) return e;
  if (T < 0 || T >= (int64_t(1) << 31) || !ws || (T > 0 && !ids)) return L3_ERR_INVALID_ARG;
  if (ws_bytes < l3_workspace_size(L, T, L3_PASS_FORWARD)) return L3_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  Carve c(ws);
  FwdWs w = carve_fwd(c, L, T);
  L3_CUDA(cudaMemsetAsync(w.st, 0, sizeof(DevStatus), s));
  const uint64_t* keys = nullptr;
  L3_CUDA(launch_route(ids, T, L->vocab, w.route_scratch, RouteOut{perm, seg_start, seg_id, n_seg},
                       w.st, s, &keys));
  return L3_OK;
}

l3_status l3_forward(const l3_layer* L, const int32_t* ids, int64_t T, const void* x, void* y,
                     int32_t y_dtype, void* saved, void* ws, size_t ws_bytes,
                     l3_stream_t stream) {
  return forward_impl(L, ids, T, x, y, y_dtype, saved, ws, ws_bytes,
                      reinterpret_cast<cudaStream_t>(stream), nullptr);
}

l3_status l3_forward_timed(const l3_layer* L, const int32_t* ids, int64_t T, const void* x,
                           void* y, int32_t y_dtype, void* saved, void* ws, size_t ws_bytes,
                           l3_stream_t stream, l3_event_t* events) {
  if (!events) return L3_ERR_INVALID_ARG;
  return forward_impl(L, ids, T, x, y, y_dtype, saved, ws, ws_bytes,
                      reinterpret_cast<cudaStream_t>(stream),
                      reinterpret_cast<cudaEvent_t*>(events));
}

l3_status l3_forward_host(const l3_layer* L, const int32_t* ids_host, int64_t T,
                          const void* x_host, void* y_host, int32_t y_dtype, void* ws,
                          size_t ws_bytes, l3_stream_t stream) {
  l3_status e = check_layer_args(L);
  if (e != L3_OK) return e;
  if (T < 0 || T >= (int64_t(1) << 31)) return L3_ERR_INVALID_ARG;
  if (T == 0) return L3_OK;
  if (!ids_host || !x_host || !y_host || !ws) return L3_ERR_INVALID_ARG;
  if (!(y_dtype == L3_F32 || y_dtype == L->dtype)) return L3_ERR_INVALID_ARG;
  if (ws_bytes < l3_workspace_size(L, T, L3_PASS_FORWARD_HOST)) return L3_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  Carve c(ws);
  carve_fwd(c, L, T);
  const size_t fwd_bytes = align_up(c.off, kAlign);
  const size_t xb = size_t(T) * size_t(L->d) * esize(L->dtype);
  const size_t yb = size_t(T) * size_t(L->d) * esize(y_dtype);
  int32_t* ids_d = c.take<int32_t>(size_t(T));
  void* x_d = c.raw(xb);
  void* y_d = c.raw(size_t(T) * size_t(L->d) * 4);
  L3_CUDA(cudaMemcpyAsync(ids_d, ids_host, size_t(T) * 4, cudaMemcpyHostToDevice, s));
  L3_CUDA(cudaMemcpyAsync(x_d, x_host, xb, cudaMemcpyHostToDevice, s));
  e = forward_impl(L, ids_d, T, x_d, y_d, y_dtype, nullptr, ws, fwd_bytes, s, nullptr);
  if (e != L3_OK) return e;
  L3_CUDA(cudaMemcpyAsync(y_host, y_d, yb, cudaMemcpyDeviceToHost, s));
  return L3_OK;
}

l3_status l3_backward(const l3_layer* L, const int32_t* ids, int64_t T, const void* x,
                      const void* dy, const void* saved, float* dx, float* dK, float* dV,
                      float* dW_up, float* dW_mix, void* ws, size_t ws_bytes,
                      l3_stream_t stream) {
  l3_status e = check_layer_args(L);
  if (e != L3_OK) return e;
  if (T < 0 || T >= (int64_t(1) << 31)) return L3_ERR_INVALID_ARG;
  if (!dK || !dV || !dW_up || !dW_mix || !ws) return L3_ERR_INVALID_ARG;
  if (T > 0 && (!ids || !x || !dy || !saved || !dx)) return L3_ERR_INVALID_ARG;
  if (ws_bytes < l3_workspace_size(L, T, L3_PASS_BACKWARD)) return L3_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int d = int(L->d), dv = int(L->d_v);
  Carve c(ws);
  BwdWs w = carve_bwd(c, L, T);
  L3_CUDA(cudaMemsetAsync(w.st, 0, sizeof(DevStatus), s));
  L3_CUDA(cudaMemsetAsync(dK, 0, size_t(L->v) * size_t(d) * 4, s));
  L3_CUDA(cudaMemsetAsync(dV, 0, size_t(L->v) * size_t(dv) * 4, s));
  if (T == 0) {
    L3_CUDA(cudaMemsetAsync(dW_up, 0, size_t(d) * size_t(dv) * 4, s));
    L3_CUDA(cudaMemsetAsync(dW_mix, 0, size_t(d) * size_t(2 * d) * 4, s));
    return L3_OK;
  }
  Carve cs(const_cast<void*>(saved));
  Saved sv = carve_saved(cs, L, T);

  const uint64_t* keys = nullptr;
  L3_CUDA(launch_route(ids, T, L->vocab, w.route_scratch,
                       RouteOut{nullptr, w.seg_start, nullptr, w.n_seg}, w.st, s, &keys));
  // Recompute u = W_up a (fp32 a from the forward) and h = LayerNorm(u).
  SimtGemm g{};
  g.M = T;
  g.N = d;
  g.K = dv;
  g.A = sv.a;
  g.a_dtype = L3_F32;
  g.a_sm = dv;
  g.a_sk = 1;
  g.B = L->W_up;
  g.b_dtype = L->dtype;
  g.b_sk = 1;
  g.b_sn = dv;
  g.C = w.U;
  g.ldc = d;
  g.alpha = 1.f;
  g.beta = 0.f;
  L3_CUDA(launch_simt_gemm(g, s));
  L3_CUDA(launch_ln_stats(w.U, T, d, L->ln_eps, w.mu, w.rstd, s));
  L3_CUDA(launch_ln_apply(w.U, w.mu, w.rstd, T, d, w.H, s));
  // dW_mix[:, :d] = dyᵀ h, dW_mix[:, d:] = dyᵀ x
  g = SimtGemm{};
  g.M = d;
  g.N = d;
  g.K = T;
  g.A = dy;
  g.a_dtype = L->dtype;
  g.a_sm = 1;
  g.a_sk = d;
  g.B = w.H;
  g.b_dtype = L3_F32;
  g.b_sk = d;
  g.b_sn = 1;
  g.C = dW_mix;
  g.ldc = 2 * d;
  g.alpha = 1.f;
  g.beta = 0.f;
  L3_CUDA(launch_simt_gemm(g, s));
  g.B = x;
  g.b_dtype = L->dtype;
  g.C = dW_mix + d;
  L3_CUDA(launch_simt_gemm(g, s));
  // dC = dy W_mix  [T, 2d]
  g = SimtGemm{};
  g.M = T;
  g.N = 2 * d;
  g.K = d;
  g.A = dy;
  g.a_dtype = L->dtype;
  g.a_sm = d;
  g.a_sk = 1;
  g.B = L->W_mix;
  g.b_dtype = L->dtype;
  g.b_sk = 2 * d;
  g.b_sn = 1;
  g.C = w.dC;
  g.ldc = 2 * d;
  g.alpha = 1.f;
  g.beta = 0.f;
  L3_CUDA(launch_simt_gemm(g, s));
  L3_CUDA(launch_ln_backward(w.dC, 2 * d, w.H, w.rstd, T, d, w.du, s));
  // dW_up = duᵀ a  [d, d_v]
  g = SimtGemm{};
  g.M = d;
  g.N = dv;
  g.K = T;
  g.A = w.du;
  g.a_dtype = L3_F32;
  g.a_sm = 1;
  g.a_sk = d;
  g.B = sv.a;
  g.b_dtype = L3_F32;
  g.b_sk = dv;
  g.b_sn = 1;
  g.C = dW_up;
  g.ldc = dv;
  g.alpha = 1.f;
  g.beta = 0.f;
  L3_CUDA(launch_simt_gemm(g, s));
  // da = du W_up  [T, d_v]
  g = SimtGemm{};
  g.M = T;
  g.N = dv;
  g.K = d;
  g.A = w.du;
  g.a_dtype = L3_F32;
  g.a_sm = d;
  g.a_sk = 1;
  g.B = L->W_up;
  g.b_dtype = L->dtype;
  g.b_sk = dv;
  g.b_sn = 1;
  g.C = w.dA;
  g.ldc = dv;
  g.alpha = 1.f;
  g.beta = 0.f;
  L3_CUDA(launch_simt_gemm(g, s));

  AttendBwdArgs ab{};
  ab.sorted_keys = keys;
  ab.T = T;
  ab.offs = L->offs;
  ab.K = L->K;
  ab.V = L->V;
  ab.x = x;
  ab.d = d;
  ab.d_v = dv;
  ab.k_max = L->k_max;
  ab.dtype = L->dtype;
  ab.da = w.dA;
  ab.dx_in = w.dC + d;
  ab.ldx_in = 2 * d;
  ab.dx = dx;
  ab.p_buf = w.p_buf;
  ab.ds_buf = w.ds_buf;
  L3_CUDA(launch_attend_bwd(ab, s));

  SegReduceArgs sr{};
  sr.sorted_keys = keys;
  sr.T = T;
  sr.seg_start = w.seg_start;
  sr.n_seg = w.n_seg;
  sr.offs = L->offs;
  sr.x = x;
  sr.dtype = L->dtype;
  sr.da = w.dA;
  sr.d = d;
  sr.d_v = dv;
  sr.k_max = L->k_max;
  sr.p_buf = w.p_buf;
  sr.ds_buf = w.ds_buf;
  sr.dK = dK;
  sr.dV = dV;
  L3_CUDA(launch_seg_reduce(sr, s));
  return L3_OK;
}

l3_status l3_count_ids(const int32_t* ids, int64_t n, int64_t vocab, int64_t* counts, void* ws,
                       size_t ws_bytes, l3_stream_t stream) {
  if (n < 0 || n >= (int64_t(1) << 31) || vocab < 1 || vocab >= (int64_t(1) << 31) || !counts ||
      !ws || (n > 0 && !ids))
    return L3_ERR_INVALID_ARG;
  if (ws_bytes < sizeof(DevStatus)) return L3_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  L3_CUDA(cudaMemsetAsync(ws, 0, sizeof(DevStatus), s));
  L3_CUDA(launch_count_ids(ids, n, vocab, counts, static_cast<DevStatus*>(ws), s));
  return L3_OK;
}

l3_status l3_backward_rows(const l3_layer* L, const int32_t* ids, int64_t T, const void* x,
                           const void* dy, const void* saved, float* dx, int32_t* row_index,
                           float* dK_rows, float* dV_rows, int32_t* n_rows, int64_t max_rows,
                           float* dW_up, float* dW_mix, void* ws, size_t ws_bytes,
                           l3_stream_t stream) {
  l3_status e = check_layer_args(L);
  if (e != L3_OK) return e;
  if (L->dtype != L3_BF16) return L3_ERR_UNSUPPORTED;
  if (T < 0 || T >= (int64_t(1) << 31) || max_rows < 0) return L3_ERR_INVALID_ARG;
  if (!dW_up || !dW_mix || !n_rows || !ws) return L3_ERR_INVALID_ARG;
  if (T > 0 && (!ids || !x || !dy || !saved || !dx || !row_index || !dK_rows || !dV_rows))
    return L3_ERR_INVALID_ARG;
  if (ws_bytes < l3_workspace_size(L, T, L3_PASS_BACKWARD_ROWS)) return L3_ERR_WORKSPACE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int d = int(L->d), dv = int(L->d_v);
  Carve c(ws);
  BwdRowsWs w = carve_bwd_rows(c, L, T);
  L3_CUDA(cudaMemsetAsync(w.st, 0, sizeof(DevStatus), s));
  if (T == 0) {
    L3_CUDA(cudaMemsetAsync(dW_up, 0, size_t(d) * size_t(dv) * 4, s));
    L3_CUDA(cudaMemsetAsync(dW_mix, 0, size_t(d) * size_t(2 * d) * 4, s));
    L3_CUDA(cudaMemsetAsync(n_rows, 0, 4, s));
    return L3_OK;
  }
  Carve cs(const_cast<void*>(saved));
  const Saved sv = carve_saved(cs, L, T);
  const int ch = attend_bwd_rows_per_chunk(d, dv);
  // batch sorting and the token groups (every segment in groups of at most 8 tokens); the
  // CTAs of Phase A split the groups by cost: 2 units a chunk, 3 more a group (its fragment
  // loads and its dx stores)
  PlanOut plan{w.groups, w.hdr, w.counters, nullptr, L->offs, L->v, L->k_max, ch, kPlanMT,
               INT32_MAX, nullptr, nullptr, nullptr, 0, 2, 3};
  const uint64_t* keys = nullptr;
  L3_CUDA(launch_route(ids, T, L->vocab, w.route_scratch,
                       RouteOut{nullptr, w.seg_start, nullptr, w.n_seg}, w.st, s, &keys, &plan));
  const int Ti = int(T);
  auto gemm = [&](int m, int n, int k, bool ta, bool tb, const void* A, int64_t lda, const void* B,
                  int64_t ldb, void* C, int64_t ldc, bool c16, bool acc) {
    return lt_gemm(LtGemm{m, n, k, ta, tb, A, lda, B, ldb, C, ldc, c16, acc}, w.lt_ws,
                   kLtWorkspace, s);
  };
  BwdSmallArgs sa{};
  sa.T = T;
  sa.d = d;
  sa.d_v = dv;
  sa.eps = L->ln_eps;
  // u = W_up a in fp32 from a as bf16 hi + lo, and h = LayerNorm(u) (fp32 and bf16)
  sa.stage = 3;
  sa.a = sv.a;
  sa.a_hi = w.a_hi;
  sa.a_lo = w.a_lo;
  L3_CUDA(launch_bwd_small(sa, s));
  L3_CUDA(gemm(d, Ti, dv, true, false, L->W_up, dv, w.a_hi, dv, w.U32, d, false, false));
  L3_CUDA(gemm(d, Ti, dv, true, false, L->W_up, dv, w.a_lo, dv, w.U32, d, false, true));
  sa.stage = 0;
  sa.U32 = w.U32;
  sa.h16 = w.h16;
  sa.rstd_out = w.rstd;
  L3_CUDA(launch_bwd_small(sa, s));
  // dW_mix = dyᵀ [h x]
  L3_CUDA(gemm(d, d, Ti, false, true, w.h16, d, dy, d, dW_mix, 2 * d, false, false));
  L3_CUDA(gemm(d, d, Ti, false, true, x, d, dy, d, dW_mix + d, 2 * d, false, false));
  // dh = dy W_mix[:, :d]
  L3_CUDA(gemm(d, Ti, d, false, false, L->W_mix, 2 * d, dy, d, w.dh, d, false, false));
  // du = LayerNorm backward (bf16 hi + lo); dW_up = duᵀ a; da = du W_up from both parts
  sa.stage = 1;
  sa.dh = w.dh;
  sa.du = w.du_hi;
  sa.du_lo = w.du_lo;
  L3_CUDA(launch_bwd_small(sa, s));
  L3_CUDA(gemm(dv, d, Ti, false, true, w.a_hi, dv, w.du_hi, d, dW_up, dv, false, false));
  L3_CUDA(gemm(dv, Ti, d, false, false, L->W_up, dv, w.du_hi, d, w.da, dv, false, false));
  L3_CUDA(gemm(dv, Ti, d, false, false, L->W_up, dv, w.du_lo, d, w.da, dv, false, true));
  // x and da in sorted order, da as bf16 hi + lo, delta = a . da
  sa.stage = 2;
  sa.keys = keys;
  sa.x = static_cast<const __nv_bfloat16*>(x);
  sa.da = w.da;
  sa.x_sorted = w.x_sorted;
  sa.da16 = w.da16;
  sa.da16_lo = w.da16_lo;
  sa.delta = w.delta;
  L3_CUDA(launch_bwd_small(sa, s));
  // Phase A: p, ds per token and row; dx = sum_j ds_j K_j
  AttendBwdRowsArgs ab{};
  ab.sorted_keys = keys;
  ab.T = T;
  ab.groups = w.groups;
  ab.hdr = w.hdr;
  ab.K = L->K;
  ab.V = L->V;
  ab.v = L->v;
  ab.d = d;
  ab.d_v = dv;
  ab.ch = ch;
  ab.k_max = L->k_max;
  ab.x_sorted = w.x_sorted;
  ab.da16 = w.da16;
  ab.da16_lo = w.da16_lo;
  ab.ml = sv.ml;
  ab.delta = w.delta;
  ab.dx = dx;
  ab.p_buf = w.p_buf;
  ab.ds_buf = w.ds_buf;
  ab.n_cta = device_sm_count();
  ab.st = w.st;
  L3_CUDA(launch_attend_bwd_rows(ab, s));
  // dx += the direct term dy W_mix[:, d:]
  L3_CUDA(gemm(d, Ti, d, false, false, static_cast<const __nv_bfloat16*>(L->W_mix) + d, 2 * d, dy,
               d, dx, d, false, true));
  // Phase B: the touched rows' dK and dV, in segment order
  L3_CUDA(launch_row_plan(keys, w.seg_start, w.n_seg, L->offs, d, dv, w.seg_row0, w.seg_unit0,
                          w.seg_cost0, n_rows, max_rows, w.st, s));
  SegRowsArgs sr{};
  sr.sorted_keys = keys;
  sr.seg_start = w.seg_start;
  sr.n_seg = w.n_seg;
  sr.offs = L->offs;
  sr.seg_row0 = w.seg_row0;
  sr.seg_unit0 = w.seg_unit0;
  sr.seg_cost0 = w.seg_cost0;
  sr.x_sorted = w.x_sorted;
  sr.da_sorted = w.da16;
  sr.p_buf = w.p_buf;
  sr.ds_buf = w.ds_buf;
  sr.k_max = L->k_max;
  sr.d = d;
  sr.d_v = dv;
  sr.row_index = row_index;
  sr.dK_rows = dK_rows;
  sr.dV_rows = dV_rows;
  sr.max_rows = max_rows;
  sr.st = w.st;
  L3_CUDA(launch_seg_rows(sr, s));
  return L3_OK;
}

l3_status l3_stage_rows(const l3_layer* L, const int32_t* ids, int64_t T, void* K_stage,
                        void* V_stage, int64_t max_rows, int32_t* offs_stage, int32_t* ids_stage,
                        int32_t* n_rows, l3_layer* staged, void* ws, size_t ws_bytes,
                        l3_stream_t stream) {
  l3_status e = check_layer_args(L);
  if (e != L3_OK) return e;
  if (T < 1 || T >= (int64_t(1) << 31) || !ids || !K_stage || !V_stage || !offs_stage ||
      !ids_stage || !n_rows || !staged || !ws)
    return L3_ERR_INVALID_ARG;
  // the staged layer has vocabulary T and max_rows rows
  if (max_rows < T || max_rows > T * int64_t(L->k_max) || max_rows >= (int64_t(1) << 31))
    return L3_ERR_INVALID_ARG;
  if (ws_bytes < l3_workspace_size(L, T, L3_PASS_STAGE)) return L3_ERR_WORKSPACE;
  // the tables may be pinned host memory (read through its device-mapped address) or
  // device memory
  const void* src[2] = {L->K, L->V};
  const void* dev_src[2] = {nullptr, nullptr};
  for (int k = 0; k < 2; ++k) {
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, src[k]) != cudaSuccess) {
      (void)cudaGetLastError();
      return L3_ERR_INVALID_ARG;
    }
    if (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged)
      dev_src[k] = src[k];
    else if (at.type == cudaMemoryTypeHost && at.devicePointer)
      dev_src[k] = at.devicePointer;
    else
      return L3_ERR_INVALID_ARG;  // pageable host memory: the device cannot read it
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  Carve c(ws);
  DevStatus* st = c.take<DevStatus>(1);
  void* route_scratch = c.raw(route_scratch_bytes(T));
  int32_t* seg_start = c.take<int32_t>(size_t(T) + 1);
  int32_t* n_seg = c.take<int32_t>(1);
  int32_t* seg_row0 = c.take<int32_t>(size_t(T) + 1);
  int32_t* seg_unit0 = c.take<int32_t>(size_t(T) + 1);
  int64_t* seg_cost0 = c.take<int64_t>(size_t(T) + 1);
  L3_CUDA(cudaMemsetAsync(st, 0, sizeof(DevStatus), s));
  const uint64_t* keys = nullptr;
  L3_CUDA(launch_route(ids, T, L->vocab, route_scratch, RouteOut{nullptr, seg_start, nullptr, n_seg},
                       st, s, &keys));
  L3_CUDA(launch_row_plan(keys, seg_start, n_seg, L->offs, int(L->d), int(L->d_v), seg_row0,
                          seg_unit0, seg_cost0, n_rows, max_rows, st, s));
  const size_t es = L->dtype == L3_BF16 ? 2 : 4;
  StageArgs sa{};
  sa.sorted_keys = keys;
  sa.seg_start = seg_start;
  sa.n_seg = n_seg;
  sa.offs = L->offs;
  sa.seg_row0 = seg_row0;
  sa.n_rows = n_rows;
  sa.K_host = dev_src[0];
  sa.V_host = dev_src[1];
  sa.k_row_bytes = L->d * int64_t(es);
  sa.v_row_bytes = L->d_v * int64_t(es);
  sa.K_st = K_stage;
  sa.V_st = V_stage;
  sa.max_rows = max_rows;
  sa.offs_st = offs_stage;
  sa.ids_st = ids_stage;
  sa.T = T;
  sa.st = st;
  L3_CUDA(launch_stage_rows(sa, s));
  *staged = *L;
  staged->vocab = T;
  staged->v = max_rows;
  staged->offs = offs_stage;
  staged->K = K_stage;
  staged->V = V_stage;
  return L3_OK;
}

l3_status l3_get_error(void* ws, l3_stream_t stream) {
  if (!ws) return L3_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  DevStatus h{};
  L3_CUDA(cudaStreamSynchronize(s));
  L3_CUDA(cudaMemcpy(&h, ws, sizeof(h), cudaMemcpyDeviceToHost));
  L3_CUDA(cudaMemset(ws, 0, sizeof(h)));
  if (h.token_range) return L3_ERR_TOKEN_RANGE;
  if (h.layer_bad) return L3_ERR_LAYER;
  if (h.timeout) return L3_ERR_TIMEOUT;
  if (h.capacity) return L3_ERR_WORKSPACE;
  return L3_OK;
}

const char* l3_status_string(l3_status st) {
  switch (st) {
    case L3_OK: return "L3_OK";
    case L3_ERR_INVALID_ARG: return "L3_ERR_INVALID_ARG";
    case L3_ERR_INFEASIBLE: return "L3_ERR_INFEASIBLE";
    case L3_ERR_UNSUPPORTED: return "L3_ERR_UNSUPPORTED";
    case L3_ERR_WORKSPACE: return "L3_ERR_WORKSPACE";
    case L3_ERR_TOKEN_RANGE: return "L3_ERR_TOKEN_RANGE";
    case L3_ERR_CUDA: return "L3_ERR_CUDA";
    case L3_ERR_LAYER: return "L3_ERR_LAYER";
    case L3_ERR_TIMEOUT: return "L3_ERR_TIMEOUT";
  }
  return "L3_ERR_UNKNOWN";
}

l3_status l3_selftest_wait_timeout(void* ws, size_t ws_bytes, int64_t limit_ns,
                                   l3_stream_t stream) {
  if (!ws || ws_bytes < 256 || limit_ns < 1000 || limit_ns > 10000000000LL)
    return L3_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  L3_CUDA(cudaMemsetAsync(ws, 0, sizeof(DevStatus), s));
  L3_CUDA(launch_wait_selftest(static_cast<DevStatus*>(ws), uint64_t(limit_ns), s));
  return L3_OK;
}

uint64_t l3_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int32_t l3_abi_version(void) { return L3_ABI_VERSION; }

}  // extern "C"
