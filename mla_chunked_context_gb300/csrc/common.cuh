// Small device helpers shared by the CUDA kernels of this library.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "../../include/mla_chunked_context.h"

namespace mla {

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) {
  return __bfloat162float(x);
}
__device__ __forceinline__ float to_f32(__half x) { return __half2float(x); }

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) {
  return x;
}
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}
template <>
__device__ __forceinline__ __half from_f32<__half>(float x) {
  return __float2half_rn(x);
}

__device__ __forceinline__ bool is_neg_inf(float x) {
  return x == -__int_as_float(0x7f800000);
}

__device__ __forceinline__ float neg_inf() { return -__int_as_float(0x7f800000); }

// Index of the sequence that owns position `x`: the largest i in [0, n) with
// loc[i] <= x, for a non-decreasing loc[0..n].
__device__ __forceinline__ int find_seq(const int32_t *loc, int n, int x) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(loc + mid) <= x)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

// Kernels this library has enqueued since it was loaded (every launcher
// calls launch_status() once, right after its launch).
inline std::atomic<unsigned long long> g_kernel_launches{0};

inline int launch_status() {
  g_kernel_launches.fetch_add(1, std::memory_order_relaxed);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

inline int elem_bytes(int32_t dtype) { return dtype == MLA_DTYPE_F32 ? 4 : 2; }

// storage types of the inputs and of the final output
inline bool valid_dtype(int32_t dtype) {
  return dtype == MLA_DTYPE_BF16 || dtype == MLA_DTYPE_F32;
}
// storage types of the up-projected K/V workspace
inline bool valid_kv_dtype(int32_t dtype) {
  return dtype == MLA_DTYPE_BF16 || dtype == MLA_DTYPE_F32 || dtype == MLA_DTYPE_F16;
}

// Scratch of the key-split attention: `slots` partials of [H][128][Dv] f32
// (O) and [H][128] f32 (LSE); a launch splits its longest (sequence, query
// tile) units over their keys until it has about `target_ctas` CTAs.
struct SplitScratch {
  float *o = nullptr, *lse = nullptr;
  int slots = 0, target_ctas = 0;
};

inline int num_sms() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

}  // namespace mla
