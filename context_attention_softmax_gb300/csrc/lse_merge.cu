// Merge of finalised per-chunk results (O_c, LSE_c) into the global result.
//
// "Context parallel attention: exchange keys and merge softmax globally",
// para 3: rescale every chunk to the larger maximum, add, divide at the end.
// In LSE form a finalised chunk (O_c, LSE_c) is its summary up to a common
// factor (l_c = exp(LSE_c - m_c), z_c = l_c O_c), so the merge reads
//   L = max_c LSE_c,  w_c = exp(LSE_c - L),  O = sum w_c O_c / sum w_c,
//   LSE = L + ln sum w_c.
// Para 4: a neutral chunk has LSE_c = -inf and weight 0 (never -inf - -inf);
// all chunks neutral gives O = 0, LSE = -inf.
//
// Memory-bound: each (row, head) reads n_parts * (Dv + 1) floats once and
// writes Dv outputs.  One warp per (row, head); lanes own 4 consecutive
// channels per step so each part is read with 16-byte coalesced loads.
#include "common.cuh"
#include "internal.h"

namespace cpattn {
namespace {

constexpr int kWarps = 8;
constexpr int kMaxUnrolled = 8;   // parts merged with all loads in flight

__device__ __forceinline__ uint32_t pack_bf16_rn(float lo, float hi) {
  __nv_bfloat162 t = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&t);
}

template <typename TO>
__device__ __forceinline__ void store4(TO* p, float4 v);
template <>
__device__ __forceinline__ void store4<float>(float* p, float4 v) {
  *reinterpret_cast<float4*>(p) = v;
}
template <>
__device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16* p, float4 v) {
  __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
  __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t*>(&a);
  u.y = *reinterpret_cast<uint32_t*>(&b);
  *reinterpret_cast<uint2*>(p) = u;
}

// Four consecutive channels of a part (fp32, or bf16 widened).
__device__ __forceinline__ float4 load4(const float* p) { return __ldg(reinterpret_cast<const float4*>(p)); }
__device__ __forceinline__ float4 load4(const __nv_bfloat16* p) {
  const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
  return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                     __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
}

template <typename TO, typename TP>
__global__ void __launch_bounds__(kWarps * 32)
lse_merge_kernel(int n_parts, const TP* __restrict__ part_o, const float* __restrict__ part_lse,
                 int64_t rows, int H, int Dv, TO* __restrict__ o, int64_t ost, int64_t osh,
                 float* __restrict__ lse) {
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
  if (row >= rows) return;
  const int64_t t = row / H;
  const int h = (int)(row - t * H);

  if (n_parts <= kMaxUnrolled && Dv == 128) {
    // every part's LSE, then every part's 4 channels of this lane, in flight together
    float lc[kMaxUnrolled];
#pragma unroll
    for (int c = 0; c < kMaxUnrolled; ++c)
      lc[c] = c < n_parts ? __ldg(part_lse + (int64_t)c * rows + row) : -CUDART_INF_F;
    float L = lc[0];
#pragma unroll
    for (int c = 1; c < kMaxUnrolled; ++c) L = fmaxf(L, lc[c]);
    TO* orow = o + t * ost + h * osh + lane * 4;
    if (L == -CUDART_INF_F) {
      store4<TO>(orow, make_float4(0.f, 0.f, 0.f, 0.f));
      if (lane == 0 && lse != nullptr) lse[row] = -CUDART_INF_F;
      return;
    }
    float4 x[kMaxUnrolled];
    float w[kMaxUnrolled];
#pragma unroll
    for (int c = 0; c < kMaxUnrolled; ++c) {
      w[c] = (lc[c] == -CUDART_INF_F) ? 0.f : expf(lc[c] - L);
      x[c] = w[c] != 0.f ? load4(part_o + ((int64_t)c * rows + row) * Dv + lane * 4)
                         : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float wsum = 0.f;
#pragma unroll
    for (int c = 0; c < kMaxUnrolled; ++c) {
      if (w[c] == 0.f) continue;
      wsum += w[c];
      acc.x = fmaf(w[c], x[c].x, acc.x);
      acc.y = fmaf(w[c], x[c].y, acc.y);
      acc.z = fmaf(w[c], x[c].z, acc.z);
      acc.w = fmaf(w[c], x[c].w, acc.w);
    }
    const float inv = 1.f / wsum;
    store4<TO>(orow, make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv));
    if (lane == 0 && lse != nullptr) lse[row] = L + logf(wsum);
    return;
  }

  float L = -CUDART_INF_F;
  for (int c = lane; c < n_parts; c += 32) L = fmaxf(L, __ldg(part_lse + (int64_t)c * rows + row));
  L = warp_max(L);

  TO* orow = o + t * ost + h * osh;
  if (L == -CUDART_INF_F) {
    for (int d = lane * 4; d < Dv; d += 128) store4<TO>(orow + d, make_float4(0.f, 0.f, 0.f, 0.f));
    if (lane == 0 && lse != nullptr) lse[row] = -CUDART_INF_F;
    return;
  }
  float W = 0.f;
  for (int d0 = 0; d0 < Dv; d0 += 128) {
    const int d = d0 + lane * 4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float wsum = 0.f;
    for (int c = 0; c < n_parts; ++c) {
      const float lc = __ldg(part_lse + (int64_t)c * rows + row);
      const float w = (lc == -CUDART_INF_F) ? 0.f : expf(lc - L);
      wsum += w;
      if (w != 0.f && d < Dv) {
        const float4 x = load4(part_o + ((int64_t)c * rows + row) * Dv + d);
        acc.x = fmaf(w, x.x, acc.x);
        acc.y = fmaf(w, x.y, acc.y);
        acc.z = fmaf(w, x.z, acc.z);
        acc.w = fmaf(w, x.w, acc.w);
      }
    }
    W = wsum;
    if (d < Dv) {
      const float inv = 1.f / wsum;
      store4<TO>(orow + d, make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv));
    }
  }
  if (lane == 0 && lse != nullptr) lse[row] = L + logf(W);
}

// Up to four parts of 128 channels: a half-warp merges one row, each lane
// eight channels, with every LSE and every part's channels of the row in
// flight at once (neutral parts, of weight 0, may hold anything and are
// skipped).  Few registers, so many rows per SM are in flight.
struct Ch8 {
  float v[8];
};
__device__ __forceinline__ Ch8 load8(const float* p) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(p));
  const float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
  return Ch8{{a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w}};
}
__device__ __forceinline__ Ch8 load8(const __nv_bfloat16* p) {
  const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
  return Ch8{{__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
              __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u),
              __uint_as_float(u.z << 16), __uint_as_float(u.z & 0xffff0000u),
              __uint_as_float(u.w << 16), __uint_as_float(u.w & 0xffff0000u)}};
}
__device__ __forceinline__ void store8(float* p, const float (&v)[8]) {
  reinterpret_cast<float4*>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
  reinterpret_cast<float4*>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
}
__device__ __forceinline__ void store8(__nv_bfloat16* p, const float (&v)[8]) {
  uint4 u;
  u.x = pack_bf16_rn(v[0], v[1]);
  u.y = pack_bf16_rn(v[2], v[3]);
  u.z = pack_bf16_rn(v[4], v[5]);
  u.w = pack_bf16_rn(v[6], v[7]);
  *reinterpret_cast<uint4*>(p) = u;
}

template <typename TO, typename TP>
__global__ void __launch_bounds__(kWarps * 32)
lse_merge4_kernel(int n_parts, const TP* __restrict__ part_o, const float* __restrict__ part_lse,
                  int64_t rows, int H, TO* __restrict__ o, int64_t ost, int64_t osh,
                  float* __restrict__ lse) {
  constexpr int Dv = 128;
  const int l16 = threadIdx.x & 15;
  const int64_t row = (int64_t)blockIdx.x * (kWarps * 2) + (threadIdx.x >> 4);
  if (row >= rows) return;
  float lc[4];
  Ch8 x[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) lc[c] = c < n_parts ? __ldg(part_lse + (int64_t)c * rows + row) : -CUDART_INF_F;
#pragma unroll
  for (int c = 0; c < 4; ++c)
    if (c < n_parts) x[c] = load8(part_o + ((int64_t)c * rows + row) * Dv + l16 * 8);
  const int64_t t = row / H;
  const int h = (int)(row - t * H);
  TO* orow = o + t * ost + h * osh + l16 * 8;
  const float L = fmaxf(fmaxf(lc[0], lc[1]), fmaxf(lc[2], lc[3]));
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  if (L == -CUDART_INF_F) {
    store8(orow, acc);
    if (l16 == 0 && lse != nullptr) lse[row] = -CUDART_INF_F;
    return;
  }
  float wsum = 0.f;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const float w = (lc[c] == -CUDART_INF_F) ? 0.f : expf(lc[c] - L);
    if (w == 0.f) continue;
    wsum += w;
#pragma unroll
    for (int j = 0; j < 8; ++j) acc[j] = fmaf(w, x[c].v[j], acc[j]);
  }
  const float inv = 1.f / wsum;
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j] *= inv;
  store8(orow, acc);
  if (l16 == 0 && lse != nullptr) lse[row] = L + logf(wsum);
}

}  // namespace

template <typename TP>
cudaError_t launch_merge(int32_t n_parts, const TP* part_o, const float* part_lse, int32_t Tq,
                         int32_t H, int32_t Dv, void* o, int32_t o_dtype, int64_t o_stride_t,
                         int64_t o_stride_h, float* lse, cudaStream_t stream) {
  const int64_t rows = (int64_t)Tq * H;
  if (rows == 0) return cudaSuccess;
  if (n_parts <= 4 && Dv == 128) {
    const unsigned blocks4 = (unsigned)((rows + kWarps * 2 - 1) / (kWarps * 2));
    if (o_dtype == CPATTN_BF16)
      lse_merge4_kernel<__nv_bfloat16, TP><<<blocks4, kWarps * 32, 0, stream>>>(
          n_parts, part_o, part_lse, rows, H, reinterpret_cast<__nv_bfloat16*>(o), o_stride_t,
          o_stride_h, lse);
    else
      lse_merge4_kernel<float, TP><<<blocks4, kWarps * 32, 0, stream>>>(
          n_parts, part_o, part_lse, rows, H, reinterpret_cast<float*>(o), o_stride_t, o_stride_h,
          lse);
    return cudaGetLastError();
  }
  const unsigned blocks = (unsigned)((rows + kWarps - 1) / kWarps);
  if (o_dtype == CPATTN_BF16)
    lse_merge_kernel<__nv_bfloat16, TP><<<blocks, kWarps * 32, 0, stream>>>(
        n_parts, part_o, part_lse, rows, H, Dv, reinterpret_cast<__nv_bfloat16*>(o), o_stride_t,
        o_stride_h, lse);
  else
    lse_merge_kernel<float, TP><<<blocks, kWarps * 32, 0, stream>>>(
        n_parts, part_o, part_lse, rows, H, Dv, reinterpret_cast<float*>(o), o_stride_t,
        o_stride_h, lse);
  return cudaGetLastError();
}

cudaError_t launch_lse_merge(int32_t n_parts, const float* part_o, const float* part_lse,
                             int32_t Tq, int32_t H, int32_t Dv, void* o, int32_t o_dtype,
                             int64_t o_stride_t, int64_t o_stride_h, float* lse,
                             cudaStream_t stream) {
  return launch_merge(n_parts, part_o, part_lse, Tq, H, Dv, o, o_dtype, o_stride_t, o_stride_h, lse,
                      stream);
}

cudaError_t launch_lse_merge_bf16parts(int32_t n_parts, const __nv_bfloat16* part_o,
                                       const float* part_lse, int32_t Tq, int32_t H, int32_t Dv,
                                       void* o, int32_t o_dtype, int64_t o_stride_t,
                                       int64_t o_stride_h, float* lse, cudaStream_t stream) {
  return launch_merge(n_parts, part_o, part_lse, Tq, H, Dv, o, o_dtype, o_stride_t, o_stride_h, lse,
                      stream);
}

}  // namespace cpattn
