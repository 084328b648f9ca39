// Device helpers shared by the kernels: positions, the permitted key
// interval, element loads and warp reductions.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math_constants.h>
#include <stdint.h>

#include "cpattn.h"

namespace cpattn {

constexpr unsigned kFullMask = 0xffffffffu;

// Logical global position of row t held in physical order: physical chunk c
// holds logical chunk map[c] ("Context parallel attention: exchange keys and
// merge softmax globally", para 5: keep logical order and physical chunk).
__device__ __forceinline__ int64_t logical_pos(const int32_t* map, int32_t chunk_len, int64_t t) {
  if (map == nullptr) return t;
  int64_t c = t / chunk_len;
  return (int64_t)__ldg(map + c) * chunk_len + (t - c * chunk_len);
}

__device__ __forceinline__ int64_t query_pos(const cpattn_attn_args& a, int64_t t) {
  return a.causal_offset + logical_pos(a.q_chunk_map, a.chunk_len, t);
}

// The keys a query may attend to form one interval of logical positions:
// its own packed sequence [cu[s], cu[s+1]) ("... merge softmax globally",
// para 2), cut at qpos when causal (para 1).  Empty when lo > hi.
struct KeyInterval {
  int64_t lo, hi;
};

__device__ __forceinline__ KeyInterval allowed_interval(const cpattn_attn_args& a, int64_t qpos) {
  KeyInterval r;
  if (a.cu_seqlens != nullptr) {
    const int32_t* cu = a.cu_seqlens;
    const int n = a.num_seqs;
    const int64_t first = __ldg(cu), last = __ldg(cu + n);
    if (qpos < first || qpos >= last) return KeyInterval{1, 0};
    int s0 = 0, s1 = n;  // cu[s0] <= qpos < cu[s1] for a well-formed cu
    while (s1 - s0 > 1) {
      int mid = (s0 + s1) >> 1;
      if (__ldg(cu + mid) <= qpos) s0 = mid; else s1 = mid;
    }
    r.lo = __ldg(cu + s0);
    r.hi = (int64_t)__ldg(cu + s0 + 1) - 1;
  } else {
    r.lo = 0;
    r.hi = INT64_MAX / 4;
  }
  if (a.causal && r.hi > qpos) r.hi = qpos;
  return r;
}

template <typename T> __device__ __forceinline__ float to_f32(T x);
template <> __device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// 8 consecutive elements (16 bytes for bf16, 32 for fp32) as floats.
__device__ __forceinline__ void load8(const __nv_bfloat16* p, float* f) {
  uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 t = __bfloat1622float2(h[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}
__device__ __forceinline__ void load8(const float* p, float* f) {
  float4 a = __ldg(reinterpret_cast<const float4*>(p));
  float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
  f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(kFullMask, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(kFullMask, x, o);
  return x;
}
__device__ __forceinline__ double warp_sum_f64(double x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(kFullMask, x, o);
  return x;
}

// Limit of every bounded wait of a call: wait_limit_ns, or 2 s when 0.
__device__ __forceinline__ uint64_t wait_limit(const cpattn_attn_args& a) {
  return a.wait_limit_ns > 0 ? (uint64_t)a.wait_limit_ns : 2000000000ull;
}

// First device-side error wins; the caller zeroes the word before the call.
__device__ __forceinline__ void report_status(int32_t* status, int32_t code) {
  if (status != nullptr) atomicCAS(status, 0, code);
}

}  // namespace cpattn
