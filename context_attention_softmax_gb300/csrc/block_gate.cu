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
//  2. gate_select_kernel - fp32 gates from the fp32 means (a register-tiled
//     product per head), each with a rigorous error bound
//     e_b = 2 (D + 8) 2^-24 ||q||_2 ||mu_b||_2 >= 2 (D + 8) 2^-24 sum_d |q_d||mu_d|,
//     which covers the fp32 dot product, the rounding of the mean and the
//     rounding of the bound itself.  With T = k-th largest lower bound g_b - e_b, the
//     set U = {b : g_b + e_b >= T} certainly contains the exact top-k and
//     everything outside it is certainly out.  |U| == k decides the
//     selection; otherwise the members of U are re-ranked by fp64 gates
//     from the fp64 means (ties to the lower block).
#include "common.cuh"
#include "internal.h"

namespace cpattn {
namespace {

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

// The same means, faster: 256 threads per (block, KV head) = column quads
// x row groups.  A warp reads 32 consecutive column quads of one row (one
// 256-byte run for bf16 at D = 128), four rows in flight per thread; each
// thread keeps a compensated sum per column of its rows, and the row groups'
// (sum, compensation) pairs are added in fp64, which loses nothing against
// the single compensated sum above.  CTAs of neighbouring indices take the
// KV heads of one block, so together they read whole rows of K.  Needs
// D % 4 == 0 and D <= 1024.
template <typename T>
__device__ __forceinline__ float4 load_quad(const T* p);
template <>
__device__ __forceinline__ float4 load_quad<__nv_bfloat16>(const __nv_bfloat16* p) {
  const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
  return make_float4(__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xffff0000u),
                     __uint_as_float(u.y << 16), __uint_as_float(u.y & 0xffff0000u));
}
template <>
__device__ __forceinline__ float4 load_quad<float>(const float* p) {
  return __ldg(reinterpret_cast<const float4*>(p));
}

__device__ __forceinline__ void neumaier(float& s, float& c, float x) {
  const float y = s + x;
  if (fabsf(s) >= fabsf(x)) c += (s - y) + x; else c += (x - y) + s;
  s = y;
}

constexpr int kMeanThreads = 256;

template <typename T>
__global__ void __launch_bounds__(kMeanThreads)
block_mean2_kernel(const T* __restrict__ k, int64_t kst, int64_t ksh, int Hkv, int D, int B,
                   double* __restrict__ mu64, float* __restrict__ mu32) {
  __shared__ double part[kMeanThreads * 4];
  const int g = blockIdx.x, b = blockIdx.y;   // the heads of one block run side by side
  const int P = D / 4, R = kMeanThreads / P;
  const int pi = threadIdx.x % P, gi = threadIdx.x / P;
  float s[4] = {0.f, 0.f, 0.f, 0.f}, c[4] = {0.f, 0.f, 0.f, 0.f};
  if (gi < R) {
    const T* col = k + (int64_t)b * B * kst + (int64_t)g * ksh + 4 * pi;
    int t = gi;
    for (; t + 3 * R < B; t += 4 * R) {
      float4 x[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) x[i] = load_quad<T>(col + (int64_t)(t + i * R) * kst);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        neumaier(s[0], c[0], x[i].x);
        neumaier(s[1], c[1], x[i].y);
        neumaier(s[2], c[2], x[i].z);
        neumaier(s[3], c[3], x[i].w);
      }
    }
    for (; t < B; t += R) {
      const float4 x = load_quad<T>(col + (int64_t)t * kst);
      neumaier(s[0], c[0], x.x);
      neumaier(s[1], c[1], x.y);
      neumaier(s[2], c[2], x.z);
      neumaier(s[3], c[3], x.w);
    }
  }
#pragma unroll
  for (int j = 0; j < 4; ++j) part[4 * threadIdx.x + j] = (double)s[j] + (double)c[j];
  __syncthreads();
  for (int e = threadIdx.x; e < D; e += kMeanThreads) {
    const int q = e / 4, j = e % 4;
    double tot = 0.0;
    for (int r = 0; r < R; ++r) tot += part[4 * (r * P + q) + j];
    const int64_t o = ((int64_t)b * Hkv + g) * D + e;
    const double m = tot / (double)B;
    mu64[o] = m;
    mu32[o] = (float)m;
  }
}

// Strict order used for every ranking: larger value first, then lower block.
__device__ __forceinline__ bool before(float v1, int b1, float v2, int b2) {
  return v1 > v2 || (v1 == v2 && b1 < b2);
}
__device__ __forceinline__ bool before64(double v1, int b1, double v2, int b2) {
  return v1 > v2 || (v1 == v2 && b1 < b2);
}

// Gates of 64 queries x all candidate blocks of one head, as a register-tiled
// fp32 product: 256 threads, each a 4-query x 4-block tile per 64-block
// chunk, both operands staged transposed in shared memory (about 100 KiB, so
// two CTAs share an SM).  The error bound
// uses norms: sum_d |q_d||mu_d| <= ||q||_2 ||mu||_2, so
//   e_b = 2 (D + 8) 2^-24 ||q||_2 ||mu_b||_2
// bounds |fp32 gate - exact gate| (dot product, rounding of the mean and of
// the norms included).  Selection then as described at the top of the file.
constexpr int kGQ = 64;          // queries per CTA
constexpr int kGB = 64;          // blocks per chunk
constexpr int kGThreads = 256;
constexpr int kQPad = kGQ + 4;   // shared row strides (floats), 16-byte aligned
constexpr int kBPad = kGB + 4;

__host__ __device__ constexpr size_t gate_smem_floats(int n_blocks, int D) {
  return (size_t)D * kQPad + (size_t)D * kBPad + (size_t)kGQ * (n_blocks + 1) + kGQ + n_blocks;
}

template <typename T>
__global__ void __launch_bounds__(kGThreads, 2)
gate_select_kernel(const cpattn_attn_args a, int B, int n_blocks, int topk,
                   const double* __restrict__ mu64, const float* __restrict__ mu32,
                   int32_t* __restrict__ sel) {
  extern __shared__ __align__(16) float gsm[];
  const int D = a.Dqk;
  float* q_s = gsm;                              // [D][kQPad]   q^T of the 64 queries
  float* m_s = q_s + (size_t)D * kQPad;          // [D][kBPad]   mu^T of one chunk
  float* g_s = m_s + (size_t)D * kBPad;          // [kGQ][n_blocks + 1] gates
  float* qn_s = g_s + (size_t)kGQ * (n_blocks + 1);  // [kGQ]  ||q||
  float* mn_s = qn_s + kGQ;                      // [n_blocks] ||mu||
  __shared__ int chosen_s[kGThreads / 32][kMaxTopk + 1];
  const int gld = n_blocks + 1;

  const int h = blockIdx.y;
  const int gkv = h / (a.Hq / a.Hkv);
  const int q0 = blockIdx.x * kGQ;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // q^T (fp32, exact from bf16) and ||q||
  for (int idx = tid; idx < kGQ * D; idx += kGThreads) {
    const int i = idx / D, d = idx - i * D;
    float v = 0.f;
    if (q0 + i < a.Tq)
      v = to_f32(reinterpret_cast<const T*>(a.q)[(int64_t)(q0 + i) * a.q_stride_t +
                                                   (int64_t)h * a.q_stride_h + d]);
    q_s[d * kQPad + i] = v;
  }
  __syncthreads();
  if (tid < kGQ) {
    float ss = 0.f;
    for (int d = 0; d < D; ++d) ss = fmaf(q_s[d * kQPad + tid], q_s[d * kQPad + tid], ss);
    qn_s[tid] = sqrtf(ss);
  }

  const int tq = tid >> 4, tb = tid & 15;   // 4 queries x 4 blocks per thread
  for (int c0 = 0; c0 < n_blocks; c0 += kGB) {
    const int nb = min(kGB, n_blocks - c0);
    __syncthreads();
    for (int idx = tid; idx < kGB * D; idx += kGThreads) {
      const int b = idx / D, d = idx - b * D;
      m_s[d * kBPad + b] = b < nb ? mu32[((int64_t)(c0 + b) * a.Hkv + gkv) * D + d] : 0.f;
    }
    __syncthreads();
    if (tid < nb) {
      float ss = 0.f;
      for (int d = 0; d < D; ++d) ss = fmaf(m_s[d * kBPad + tid], m_s[d * kBPad + tid], ss);
      mn_s[c0 + tid] = sqrtf(ss);
    }
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
#pragma unroll 4
    for (int d = 0; d < D; ++d) {
      const float4 qv = *reinterpret_cast<const float4*>(q_s + d * kQPad + 4 * tq);
      const float4 mv = *reinterpret_cast<const float4*>(m_s + d * kBPad + 4 * tb);
      const float qa[4] = {qv.x, qv.y, qv.z, qv.w};
      const float ma[4] = {mv.x, mv.y, mv.z, mv.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(qa[i], ma[j], acc[i][j]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (4 * tb + j < nb) g_s[(4 * tq + i) * gld + c0 + 4 * tb + j] = acc[i][j];
  }
  __syncthreads();

  // selection: warp w takes queries w, w + 8, ...
  int* chosen = chosen_s[warp];
  const float gamma = 2.f * (float)(D + 8) * 5.9604645e-8f * 1.01f;   // 2 (D + 8) 2^-24, padded
  for (int i = warp; i < kGQ; i += kGThreads / 32) {
    const int qi = q0 + i;
    if (qi >= a.Tq) break;
    const float* gw = g_s + i * gld;
    const float qn = qn_s[i];
    const int64_t own = query_pos(a, qi) / B;
    const int n_cand = (int)min((int64_t)n_blocks, own);
    int n_chosen = 0;
    auto err = [&](int b) { return gamma * qn * mn_s[b] + 1e-30f; };
    if (n_cand <= topk) {
      for (int b = lane; b < n_cand; b += 32) chosen[b] = b;
      n_chosen = max(n_cand, 0);
    } else {
      // T: the topk-th largest lower bound
      float pv = CUDART_INF_F;
      int pb = -1;
      for (int r = 0; r < topk; ++r) {
        float bv = -CUDART_INF_F;
        int bb = 0x7fffffff;
        for (int b = lane; b < n_cand; b += 32) {
          const float lo = gw[b] - err(b);
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
      for (int b = lane; b < n_cand; b += 32) n_u += (gw[b] + err(b) >= T_lo) ? 1 : 0;
      for (int o = 16; o > 0; o >>= 1) n_u += __shfl_xor_sync(kFullMask, n_u, o);
      if (n_u == topk) {
        int base = 0;
        for (int b0 = 0; b0 < n_cand; b0 += 32) {
          const int b = b0 + lane;
          const bool in = b < n_cand && gw[b] + err(b) >= T_lo;
          const unsigned m = __ballot_sync(kFullMask, in);
          if (in) chosen[base + __popc(m & ((1u << lane) - 1))] = b;
          base += __popc(m);
        }
        n_chosen = topk;
      } else {
        // re-rank the uncertain set by fp64 gates (q exact from its input type)
        const T* qrow = reinterpret_cast<const T*>(a.q) + (int64_t)qi * a.q_stride_t +
                        (int64_t)h * a.q_stride_h;
        double pv64 = CUDART_INF;
        pb = -1;
        for (int r = 0; r < topk; ++r) {
          double bv = -CUDART_INF;
          int bb = 0x7fffffff;
          for (int b = 0; b < n_cand; ++b) {
            if (!(gw[b] + err(b) >= T_lo)) continue;
            const double* mu = mu64 + ((int64_t)b * a.Hkv + gkv) * D;
            double acc = 0.0;
            for (int d = lane; d < D; d += 32) acc = fma((double)to_f32(qrow[d]), mu[d], acc);
            acc = warp_sum_f64(acc);
            if (before64(pv64, pb, acc, b) && before64(acc, b, bv, bb)) { bv = acc; bb = b; }
          }
          if (bb == 0x7fffffff) break;   // fewer members than topk (only with NaN gates)
          if (lane == 0) chosen[r] = bb;
          n_chosen = r + 1;
          pv64 = bv;
          pb = bb;
        }
      }
    }
    __syncwarp();
    if (lane == 0) {
      for (int x = 1; x < n_chosen; ++x) {
        const int v = chosen[x];
        int y = x - 1;
        while (y >= 0 && chosen[y] > v) { chosen[y + 1] = chosen[y]; --y; }
        chosen[y + 1] = v;
      }
      int32_t* out = sel + ((int64_t)qi * a.Hq + h) * (topk + 1);
      for (int x = 0; x < n_chosen; ++x) out[x] = chosen[x];
      out[n_chosen] = (int32_t)own;
      for (int x = n_chosen + 1; x <= topk; ++x) out[x] = -1;
    }
    __syncwarp();
  }
}

template <typename T>
cudaError_t launch_gate_t(const cpattn_attn_args& a, int B, int topk, int32_t* sel, void* ws,
                          size_t ws_bytes, cudaStream_t stream) {
  const int n_blocks = a.Tk / B;
  const int D = a.Dqk;
  const size_t n_mu = (size_t)n_blocks * a.Hkv * D;
  double* mu64 = reinterpret_cast<double*>(ws);
  float* mu32 = reinterpret_cast<float*>(mu64 + n_mu);
  if (n_blocks > 0) {
    const bool quads_ok = D % 4 == 0 && D / 4 <= kMeanThreads && a.k_stride_t % 4 == 0 &&
                          a.k_stride_h % 4 == 0 && reinterpret_cast<uintptr_t>(a.k) % (4 * sizeof(T)) == 0;
    if (quads_ok)
      block_mean2_kernel<T><<<dim3(a.Hkv, n_blocks), kMeanThreads, 0, stream>>>(
          reinterpret_cast<const T*>(a.k), a.k_stride_t, a.k_stride_h, a.Hkv, D, B, mu64, mu32);
    else
      block_mean_kernel<T><<<dim3(n_blocks, a.Hkv), min(D, 256), 0, stream>>>(
          reinterpret_cast<const T*>(a.k), a.k_stride_t, a.k_stride_h, a.Hkv, D, B, mu64, mu32);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (n_blocks > 0 && gate_tc_supported(a, B, topk) && ws_bytes >= block_gate_workspace(a, B)) {
    bool launched = false;
    cudaError_t e = launch_gate_tc(a, B, topk, sel, mu64, mu32, mu32 + n_mu, stream, &launched);
    if (e != cudaSuccess || launched) return e;
  }
  const size_t smem = block_gate_smem(n_blocks, D);
  auto kern = gate_select_kernel<T>;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid((a.Tq + kGQ - 1) / kGQ, a.Hq);
  kern<<<grid, kGThreads, smem, stream>>>(a, B, n_blocks, topk, mu64, mu32, sel);
  return cudaGetLastError();
}

}  // namespace

size_t block_gate_smem(int n_blocks, int D) { return gate_smem_floats(n_blocks, D) * sizeof(float); }

size_t block_gate_workspace_min(const cpattn_attn_args& a, int32_t block_size) {
  const size_t n_blocks = block_size > 0 ? (size_t)(a.Tk / block_size) : 0;
  return n_blocks * a.Hkv * a.Dqk * (sizeof(double) + sizeof(float));
}

size_t block_gate_workspace(const cpattn_attn_args& a, int32_t block_size) {
  size_t n = block_gate_workspace_min(a, block_size);
  if (block_size > 0 && gate_tc_supported(a, block_size, 0)) n += gate_tc_parts_bytes(a, block_size);
  return n;
}

cudaError_t launch_block_gate(const cpattn_attn_args& a, int32_t block_size, int32_t topk,
                              int32_t* sel, void* workspace, size_t workspace_bytes,
                              cudaStream_t stream) {
  if ((int64_t)a.Tq * a.Hq == 0) return cudaSuccess;
  if (a.dtype == CPATTN_BF16)
    return launch_gate_t<__nv_bfloat16>(a, block_size, topk, sel, workspace, workspace_bytes, stream);
  return launch_gate_t<float>(a, block_size, topk, sel, workspace, workspace_bytes, stream);
}

}  // namespace cpattn
