// MoBA block gate: per (query, head), pick the top-k key blocks by the gate
// <q, mean of the block's keys> among blocks that end before the query's own
// block, and always add the own block ("Question on Implementing Context
// Parallelism with MoBA Efficient Attention": gating scores Q x K^T select
// the top-k KV blocks; pooling by the block mean, ties to the lower block).
//
// The selection must equal the one made by exact (float64) gates.  Two
// kernels:
//  1. block_mean_kernel - one pass over K.  Each column of a block is summed
//     in fp32 with Neumaier compensation; the (sum, compensation) pair is
//     widened to fp64 before the division by B, so the mean is accurate to
//     far below fp32 rounding.  Both the fp64 mean and its fp32 rounding are
//     kept in the workspace (the only scratch memory of this path).
//  2. gate_select_kernel - fp32 gates from the fp32 means, each with a
//     rigorous error bound e_b = 2 (D + 8) 2^-24 sum_d |q_d| |mu_d|, which
//     covers the fp32 dot product, the rounding of the mean and the rounding
//     of the bound itself.  With T = k-th largest lower bound g_b - e_b, the
//     set U = {b : g_b + e_b >= T} certainly contains the exact top-k and
//     everything outside it is certainly out.  |U| == k decides the
//     selection; otherwise the members of U are re-ranked by fp64 gates
//     from the fp64 means (ties to the lower block).
#include "common.cuh"
#include "internal.h"

namespace cpattn {
namespace {

constexpr int kGateWarps = 4;
constexpr int kQueriesPerWarp = 8;
constexpr int kMaxTopk = 64;

template <typename T>
__global__ void block_mean_kernel(const T* __restrict__ k, int64_t kst, int64_t ksh, int Hkv,
                                  int D, int B, double* __restrict__ mu64,
                                  float* __restrict__ mu32) {
  const int b = blockIdx.x;
  const int g = blockIdx.y;
  for (int d = threadIdx.x; d < D; d += blockDim.x) {
    const T* col = k + (int64_t)b * B * kst + g * ksh + d;
    float s = 0.f, c = 0.f;
    for (int t = 0; t < B; ++t) {
      const float x = to_f32(col[(int64_t)t * kst]);
      const float y = s + x;
      if (fabsf(s) >= fabsf(x)) c += (s - y) + x; else c += (x - y) + s;
      s = y;
    }
    const double mean = ((double)s + (double)c) / (double)B;
    const int64_t o = ((int64_t)b * Hkv + g) * D + d;
    mu64[o] = mean;
    mu32[o] = (float)mean;
  }
}

// Strict order used for every ranking: larger value first, then lower block.
__device__ __forceinline__ bool before(float v1, int b1, float v2, int b2) {
  return v1 > v2 || (v1 == v2 && b1 < b2);
}
__device__ __forceinline__ bool before64(double v1, int b1, double v2, int b2) {
  return v1 > v2 || (v1 == v2 && b1 < b2);
}

template <typename T>
__global__ void __launch_bounds__(kGateWarps * 32)
gate_select_kernel(const cpattn_attn_args a, int B, int n_blocks, int topk,
                   const double* __restrict__ mu64, const float* __restrict__ mu32,
                   int32_t* __restrict__ sel) {
  extern __shared__ __align__(16) unsigned char gate_smem[];
  const int D = a.Dqk;
  const int ld = D + 1;                                         // padded row: no bank conflicts
  double* g64_s = reinterpret_cast<double*>(gate_smem);         // [warps][n_blocks]
  float* mu_s = reinterpret_cast<float*>(g64_s + kGateWarps * n_blocks);  // [n_blocks][D+1]
  float* q_s = mu_s + (size_t)n_blocks * ld;                    // [warps][D]
  float* g_s = q_s + kGateWarps * D;                            // [warps][n_blocks]
  float* e_s = g_s + kGateWarps * n_blocks;                     // [warps][n_blocks]
  __shared__ int chosen_s[kGateWarps][kMaxTopk + 1];

  const int h = blockIdx.y;
  const int gkv = h / (a.Hq / a.Hkv);
  for (int idx = threadIdx.x; idx < n_blocks * D; idx += blockDim.x) {
    const int b = idx / D, d = idx - b * D;
    mu_s[b * ld + d] = mu32[((int64_t)b * a.Hkv + gkv) * D + d];
  }
  __syncthreads();

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float* q = q_s + warp * D;
  float* gw = g_s + warp * n_blocks;
  float* ew = e_s + warp * n_blocks;
  double* g64 = g64_s + warp * n_blocks;
  int* chosen = chosen_s[warp];
  const float gamma = 2.f * (float)(D + 8) * 5.9604645e-8f;  // 2 (D + 8) 2^-24

  for (int qi = 0; qi < kQueriesPerWarp; ++qi) {
    const int i = (blockIdx.x * kGateWarps + warp) * kQueriesPerWarp + qi;
    if (i >= a.Tq) break;
    const T* qrow = reinterpret_cast<const T*>(a.q) + (int64_t)i * a.q_stride_t + (int64_t)h * a.q_stride_h;
    for (int d = lane; d < D; d += 32) q[d] = to_f32(qrow[d]);
    __syncwarp();
    const int64_t own = query_pos(a, i) / B;
    const int n_cand = (int)min((int64_t)n_blocks, own);
    int n_chosen = 0;

    if (n_cand <= topk) {
      for (int b = lane; b < n_cand; b += 32) chosen[b] = b;
      n_chosen = max(n_cand, 0);
    } else {
      for (int b = lane; b < n_cand; b += 32) {
        const float* mu = mu_s + b * ld;
        float acc = 0.f, mag = 0.f;
        for (int d = 0; d < D; ++d) {
          acc = fmaf(q[d], mu[d], acc);
          mag = fmaf(fabsf(q[d]), fabsf(mu[d]), mag);
        }
        gw[b] = acc;
        ew[b] = gamma * mag + 1e-30f;
      }
      __syncwarp();
      // T: the topk-th largest lower bound.
      float pv = CUDART_INF_F;
      int pb = -1;
      for (int r = 0; r < topk; ++r) {
        float bv = -CUDART_INF_F;
        int bb = 0x7fffffff;
        for (int b = lane; b < n_cand; b += 32) {
          const float lo = gw[b] - ew[b];
          if (before(pv, pb, lo, b) && before(lo, b, bv, bb)) { bv = lo; bb = b; }
        }
        for (int o = 16; o > 0; o >>= 1) {
          const float ov = __shfl_xor_sync(kFullMask, bv, o);
          const int ob = __shfl_xor_sync(kFullMask, bb, o);
          if (before(ov, ob, bv, bb)) { bv = ov; bb = ob; }
        }
        pv = bv;
        pb = bb;
      }
      const float T_lo = pv;
      int n_u = 0;
      for (int b = lane; b < n_cand; b += 32) n_u += (gw[b] + ew[b] >= T_lo) ? 1 : 0;
      for (int o = 16; o > 0; o >>= 1) n_u += __shfl_xor_sync(kFullMask, n_u, o);

      if (n_u == topk) {
        // U is exactly the selection; compact it in block order.
        int base = 0;
        for (int b0 = 0; b0 < n_cand; b0 += 32) {
          const int b = b0 + lane;
          const bool in = b < n_cand && gw[b] + ew[b] >= T_lo;
          const unsigned m = __ballot_sync(kFullMask, in);
          if (in) chosen[base + __popc(m & ((1u << lane) - 1))] = b;
          base += __popc(m);
        }
        n_chosen = topk;
      } else {
        // Re-rank the uncertain set by fp64 gates (members only).
        for (int b = 0; b < n_cand; ++b) {
          if (!(gw[b] + ew[b] >= T_lo)) continue;
          const double* mu = mu64 + ((int64_t)b * a.Hkv + gkv) * D;
          double acc = 0.0;
          for (int d = lane; d < D; d += 32) acc = fma((double)q[d], mu[d], acc);
          acc = warp_sum_f64(acc);
          if (lane == 0) g64[b] = acc;
        }
        __syncwarp();
        double pv64 = CUDART_INF;
        pb = -1;
        for (int r = 0; r < topk; ++r) {
          double bv = -CUDART_INF;
          int bb = 0x7fffffff;
          for (int b = lane; b < n_cand; b += 32) {
            if (!(gw[b] + ew[b] >= T_lo)) continue;
            const double gv = g64[b];
            if (before64(pv64, pb, gv, b) && before64(gv, b, bv, bb)) { bv = gv; bb = b; }
          }
          for (int o = 16; o > 0; o >>= 1) {
            const double ov = __shfl_xor_sync(kFullMask, bv, o);
            const int ob = __shfl_xor_sync(kFullMask, bb, o);
            if (before64(ov, ob, bv, bb)) { bv = ov; bb = ob; }
          }
          if (bb == 0x7fffffff) break;  // fewer members than topk (only with NaN gates)
          if (lane == 0) chosen[r] = bb;
          n_chosen = r + 1;
          pv64 = bv;
          pb = bb;
        }
      }
    }
    __syncwarp();
    if (lane == 0) {
      // ascending order; every chosen block is below the own block
      for (int x = 1; x < n_chosen; ++x) {
        const int v = chosen[x];
        int y = x - 1;
        while (y >= 0 && chosen[y] > v) { chosen[y + 1] = chosen[y]; --y; }
        chosen[y + 1] = v;
      }
      int32_t* out = sel + ((int64_t)i * a.Hq + h) * (topk + 1);
      for (int x = 0; x < n_chosen; ++x) out[x] = chosen[x];
      out[n_chosen] = (int32_t)own;
      for (int x = n_chosen + 1; x <= topk; ++x) out[x] = -1;
    }
    __syncwarp();
  }
}

template <typename T>
cudaError_t launch_gate_t(const cpattn_attn_args& a, int B, int topk, int32_t* sel, void* ws,
                          cudaStream_t stream) {
  const int n_blocks = a.Tk / B;
  const int D = a.Dqk;
  const size_t n_mu = (size_t)n_blocks * a.Hkv * D;
  double* mu64 = reinterpret_cast<double*>(ws);
  float* mu32 = reinterpret_cast<float*>(mu64 + n_mu);
  if (n_blocks > 0) {
    block_mean_kernel<T><<<dim3(n_blocks, a.Hkv), min(D, 256), 0, stream>>>(
        reinterpret_cast<const T*>(a.k), a.k_stride_t, a.k_stride_h, a.Hkv, D, B, mu64, mu32);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  const size_t smem = block_gate_smem(n_blocks, D);
  auto kern = gate_select_kernel<T>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int q_per_cta = kGateWarps * kQueriesPerWarp;
  dim3 grid((a.Tq + q_per_cta - 1) / q_per_cta, a.Hq);
  kern<<<grid, kGateWarps * 32, smem, stream>>>(a, B, n_blocks, topk, mu64, mu32, sel);
  return cudaGetLastError();
}

}  // namespace

size_t block_gate_smem(int n_blocks, int D) {
  return (size_t)kGateWarps * n_blocks * sizeof(double) + (size_t)n_blocks * (D + 1) * 4 +
         (size_t)kGateWarps * D * 4 + (size_t)kGateWarps * n_blocks * 8;
}

size_t block_gate_workspace(const cpattn_attn_args& a, int32_t block_size) {
  const size_t n_blocks = block_size > 0 ? (size_t)(a.Tk / block_size) : 0;
  return n_blocks * a.Hkv * a.Dqk * (sizeof(double) + sizeof(float));
}

cudaError_t launch_block_gate(const cpattn_attn_args& a, int32_t block_size, int32_t topk,
                              int32_t* sel, void* workspace, cudaStream_t stream) {
  if ((int64_t)a.Tq * a.Hq == 0) return cudaSuccess;
  if (a.dtype == CPATTN_BF16)
    return launch_gate_t<__nv_bfloat16>(a, block_size, topk, sel, workspace, stream);
  return launch_gate_t<float>(a, block_size, topk, sel, workspace, stream);
}

}  // namespace cpattn
