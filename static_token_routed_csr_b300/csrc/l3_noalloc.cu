// l3_route_noalloc: the batch sort of l3_route for callers that cannot hand the library
// any device memory of their own.
//
// Some callers have no way to allocate device memory when they need this call: a plugin
// running inside a host program that owns every device allocation and offers no
// allocation hook, or a latency-critical loop that must not enter an allocator (which
// can block, synchronise or fail at that moment). l3_route needs a workspace from its
// caller; this variant instead keeps its scratch (the sort keys and the status words) in
// one fixed array in device memory that the library itself declares. Each GPU that loads
// the library holds that array (about 1 MiB) until the process exits.
//
// The device address of the array is looked up once per device, by the first call made
// while that device is current (cudaGetSymbolAddress); that first call should therefore
// come before any stream capture. All calls share the one array, and it keeps whatever
// the last call left there: this code clears the status words at the start of every call,
// and two calls whose work overlaps on the GPU (different streams, no ordering between
// them) race on the array and may corrupt each other's results.
#include <mutex>

#include "l3_internal.h"

namespace l3 {
namespace {

constexpr int64_t kNoAllocMaxT = 65536;
constexpr size_t kStatusBytes = 256;
constexpr size_t kScratchBytes = 2 * size_t(kNoAllocMaxT) * sizeof(uint64_t);  // ping-pong keys

static __device__ __align__(256) unsigned char g_noalloc_scratch[kStatusBytes + kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Looks up (once per device) where the array lives on the current device.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return cudaSuccess;
}

// A token id outside [0, vocab) was seen: report it through n_seg = -1.
__global__ void fold_status_kernel(const DevStatus* st, int32_t* n_seg) {
  if (threadIdx.x == 0 && st->token_range) *n_seg = -1;
}

}  // namespace
}  // namespace l3

using namespace l3;

extern "C" l3_status l3_route_noalloc(const l3_layer* L, const int32_t* ids, int64_t T,
                                      int32_t* perm, int32_t* seg_start, int32_t* seg_id,
                                      int32_t* n_seg, l3_stream_t stream) {
  if (!L || L->vocab < 1 || L->vocab >= (int64_t(1) << 31)) return L3_ERR_INVALID_ARG;
  if (T < 0 || !n_seg || (T > 0 && !ids)) return L3_ERR_INVALID_ARG;
  if (T > kNoAllocMaxT) return L3_ERR_WORKSPACE;
  void* base = nullptr;
  if (scratch_address(&base) != cudaSuccess) {
    (void)cudaGetLastError();
    return L3_ERR_CUDA;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  DevStatus* st = static_cast<DevStatus*>(base);
  void* keys = static_cast<unsigned char*>(base) + kStatusBytes;
  if (cudaMemsetAsync(st, 0, sizeof(DevStatus), s) != cudaSuccess) {
    (void)cudaGetLastError();
    return L3_ERR_CUDA;
  }
  const uint64_t* sorted = nullptr;
  if (launch_route(ids, T, L->vocab, keys, RouteOut{perm, seg_start, seg_id, n_seg}, st, s,
                   &sorted) != cudaSuccess) {
    (void)cudaGetLastError();
    return L3_ERR_CUDA;
  }
  fold_status_kernel<<<1, 32, 0, s>>>(st, n_seg);
  count_launch();
  if (cudaGetLastError() != cudaSuccess) return L3_ERR_CUDA;
  return L3_OK;
}
