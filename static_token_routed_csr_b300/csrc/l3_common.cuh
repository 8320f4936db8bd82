// Shared device-side definitions of the L³ library (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "l3.h"

namespace l3 {

// Status words at the start of every workspace. Kernels only ever OR bits into them;
// l3_get_error reads and clears them.
struct DevStatus {
  int32_t token_range;  // a token id outside [0, vocab)
  int32_t layer_bad;    // offsets table violates its contract
  int32_t timeout;      // a bounded wait gave up (bit pattern says where)
  int32_t capacity;     // an output held fewer rows than the batch touches
};

constexpr size_t kAlign = 256;

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ---- element access -----------------------------------------------------------------------

template <typename T>
struct Elem;

template <>
struct Elem<float> {
  static constexpr int kPer16B = 4;
  __device__ static inline void load16(const float* p, float* out) {
    float4 v = __ldg(reinterpret_cast<const float4*>(p));
    out[0] = v.x;
    out[1] = v.y;
    out[2] = v.z;
    out[3] = v.w;
  }
  __device__ static inline float to_f(float v) { return v; }
  __device__ static inline float from_f(float v) { return v; }
};

template <>
struct Elem<__nv_bfloat16> {
  static constexpr int kPer16B = 8;
  __device__ static inline void load16(const __nv_bfloat16* p, float* out) {
    uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      out[2 * j] = __uint_as_float(w[j] << 16);
      out[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
    }
  }
  __device__ static inline float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
  __device__ static inline __nv_bfloat16 from_f(float v) { return __float2bfloat16_rn(v); }
};

__device__ inline float ld_as_float(const float* p) { return __ldg(p); }
__device__ inline float ld_as_float(const __nv_bfloat16* p) { return __bfloat162float(*p); }

__device__ inline float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ---- programmatic dependent launch ------------------------------------------------------
// A kernel launched with launch_pdl may start while the previous kernel on the stream is
// still running: it must call grid_dep_wait() before its first access to global memory
// that the previous kernels write or read. grid_dep_release() lets the next kernel be
// scheduled (it then waits in its own grid_dep_wait()).
__device__ __forceinline__ void grid_dep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_dep_release() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

__device__ inline float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

}  // namespace l3
