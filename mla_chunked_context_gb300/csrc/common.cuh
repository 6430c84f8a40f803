// Small device helpers shared by the CUDA kernels of this library.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <vector>

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

// Smallest magnitude that rounds to infinity in fp16 (round to nearest even:
// the largest finite value is 65504, the midpoint to 2^16 is 65520).
constexpr float kF16Overflow = 65520.f;
template <typename T>
__host__ __device__ constexpr bool is_bf16() {
  return false;
}
template <>
__host__ __device__ constexpr bool is_bf16<__nv_bfloat16>() {
  return true;
}

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

// Per-launch timing of one host thread, between mla_profile_begin() and
// mla_profile_end(): every launcher calls launch_begin(s) right before its
// launch and launch_status(s, name) right after it; while profiling is on
// these record a CUDA event on the launching stream on either side of the
// kernel, tagged with the step of the method the caller is in (ProfRole).
// Off (the default), launch_begin does nothing.  Events come from a pool
// that lives as long as the thread.
struct ProfRecord {
  const char *name, *role;
  cudaStream_t stream;
  cudaEvent_t start, stop;
};
struct ProfState {
  bool on = false;
  const char *role = "";
  cudaEvent_t pending = nullptr;  // start event of the launch being enqueued
  std::vector<ProfRecord> recs;
  std::vector<cudaEvent_t> pool;  // recorded-and-read events, for reuse
  cudaEvent_t take() {
    if (!pool.empty()) {
      cudaEvent_t e = pool.back();
      pool.pop_back();
      return e;
    }
    cudaEvent_t e = nullptr;
    return cudaEventCreate(&e) == cudaSuccess ? e : nullptr;
  }
};
inline thread_local ProfState g_prof;

// Tags the launches enqueued while it lives with a step of the method.
struct ProfRole {
  const char *saved;
  explicit ProfRole(const char *role) : saved(g_prof.role) { g_prof.role = role; }
  ~ProfRole() { g_prof.role = saved; }
};

inline void launch_begin(cudaStream_t s) {
  if (!g_prof.on) return;
  cudaEvent_t e = g_prof.take();
  if (e && cudaEventRecord(e, s) == cudaSuccess) g_prof.pending = e;
}

inline int launch_status(cudaStream_t s, const char *name) {
  g_kernel_launches.fetch_add(1, std::memory_order_relaxed);
  const cudaError_t err = cudaGetLastError();
  if (g_prof.on && g_prof.pending) {
    cudaEvent_t e = g_prof.take();
    if (e && cudaEventRecord(e, s) == cudaSuccess)
      g_prof.recs.push_back({name, g_prof.role, s, g_prof.pending, e});
    g_prof.pending = nullptr;
  }
  return err == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
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

// The keys a context attention launch appends to each sequence's context
// keys: the sequence's own new tokens (rows q_loc[i] .. q_loc[i+1] of kv
// [T, H, 256] fp16 and latent [T, latent_ld] bf16, k_pe at column 512),
// attended causally.
struct NewKeySource {
  const void *kv = nullptr, *latent = nullptr;
  int64_t latent_ld = 0;
};

inline int num_sms() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

}  // namespace mla
