// General attention kernel: one warp per (query row, head), fp32 arithmetic.
//
// This is the kernel for fp32 inputs and for shapes the tensor-core kernels
// do not take, and the sparse kernel for per-head key lists.  For each row it
// walks the selected keys in groups of 32 (one key per lane), keeps the
// running summary (m, l, z) of "Context parallel attention: exchange keys and
// merge softmax globally" para 3 - m and l warp-uniform, z split over lanes
// by value channel - and rescales to the larger max as each group arrives.
// With partial output it closes a summary at every KV-chunk boundary, writes
// it finalised, and merges it into the running total the same way.
//
// Key selection modes:
//   dense  - every permitted key.  The permitted keys of a query are one
//            interval of logical positions (own sequence, cut at qpos when
//            causal), so each physical chunk contributes one contiguous run
//            of rows and no per-key mask is needed.
//   tokens - the keys named by the query's index list (logical positions,
//            "[Feature-request] Context Parallel support for DSAttention",
//            allgather CP mode), each re-checked against the interval.
//   blocks - the key blocks named by the index list (MoBA top-k blocks),
//            each block cut to the interval.
#include <cuda_bf16.h>

#include "common.cuh"
#include "internal.h"

namespace cpattn {
namespace {

constexpr int kWarps = 4;

struct RowParams {
  cpattn_attn_args a;
  SparseArgs sp;
  int32_t n_parts;       // summaries per row (1 when no partials are written)
  int32_t part_len;      // physical rows per partial chunk
};

template <int VPL>
struct Summary {
  float m, l;
  float z[VPL];
  __device__ __forceinline__ void reset() {
    m = -CUDART_INF_F;
    l = 0.f;
#pragma unroll
    for (int r = 0; r < VPL; ++r) z[r] = 0.f;
  }
};

template <typename T>
__device__ __forceinline__ float dot_row(const float* qs, const T* krow, int D) {
  float acc = 0.f;
  for (int d = 0; d < D; d += 8) {
    float kf[8];
    load8(krow + d, kf);
#pragma unroll
    for (int e = 0; e < 8; ++e) acc = fmaf(qs[d + e], kf[e], acc);
  }
  return acc;
}

// Fold one group of up to 32 keys (one physical row per lane, -1 = none)
// into the running summary: rescale to the larger max, then add.
template <typename T, int VPL>
__device__ __forceinline__ void fold_group(Summary<VPL>& st, const float* qs, const T* kb,
                                           const T* vb, int64_t kst, int64_t vst, int Dqk,
                                           int Dv, float scale, int64_t j, int lane) {
  float s = -CUDART_INF_F;
  if (j >= 0) s = scale * dot_row(qs, kb + j * kst, Dqk);
  const float mt = warp_max(s);
  if (mt == -CUDART_INF_F) return;
  const float m_new = fmaxf(st.m, mt);
  const float alpha = (st.m == -CUDART_INF_F) ? 0.f : expf(st.m - m_new);
  const float p = (j >= 0) ? expf(s - m_new) : 0.f;
  st.l = st.l * alpha + warp_sum(p);
  st.m = m_new;
#pragma unroll
  for (int r = 0; r < VPL; ++r) st.z[r] *= alpha;
  unsigned live = __ballot_sync(kFullMask, j >= 0);
  while (live) {
    const int t = __ffs(live) - 1;
    live &= live - 1;
    const float pt = __shfl_sync(kFullMask, p, t);
    const long long jt = __shfl_sync(kFullMask, (long long)j, t);
    const T* vrow = vb + jt * vst;
#pragma unroll
    for (int r = 0; r < VPL; ++r) {
      const int d = lane + 32 * r;
      if (d < Dv) st.z[r] = fmaf(pt, to_f32(vrow[d]), st.z[r]);
    }
  }
}

// Merge summary b into a (para 3), never evaluating -inf - (-inf) (para 4).
template <int VPL>
__device__ __forceinline__ void merge_into(Summary<VPL>& a, const Summary<VPL>& b) {
  const float m = fmaxf(a.m, b.m);
  if (m == -CUDART_INF_F) return;
  const float wa = (a.m == -CUDART_INF_F) ? 0.f : expf(a.m - m);
  const float wb = (b.m == -CUDART_INF_F) ? 0.f : expf(b.m - m);
  a.l = wa * a.l + wb * b.l;
#pragma unroll
  for (int r = 0; r < VPL; ++r) a.z[r] = wa * a.z[r] + wb * b.z[r];
  a.m = m;
}

// Divide at the end: O = z / l, LSE = m + ln l; no key -> (0, -inf).
template <typename TO, int VPL>
__device__ __forceinline__ void write_final(const Summary<VPL>& st, TO* orow, float* lse_out,
                                            int Dv, int lane) {
  const bool live = st.l > 0.f;
  const float inv = live ? 1.f / st.l : 0.f;
#pragma unroll
  for (int r = 0; r < VPL; ++r) {
    const int d = lane + 32 * r;
    if (d < Dv) orow[d] = from_f32<TO>(live ? st.z[r] * inv : 0.f);
  }
  if (lane == 0 && lse_out != nullptr) *lse_out = live ? st.m + logf(st.l) : -CUDART_INF_F;
}

template <typename T, int VPL, int MODE, bool PARTIALS>
__global__ void __launch_bounds__(kWarps * 32)
rowwise_attn_kernel(const RowParams p) {
  extern __shared__ float smem[];
  const cpattn_attn_args& a = p.a;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int Dqk = a.Dqk, Dv = a.Dv;
  float* qs = smem + warp * Dqk;
  int* inv = reinterpret_cast<int*>(smem + kWarps * Dqk);

  // Inverse chunk map (logical chunk -> physical chunk) for index lookups.
  const bool use_inv = (MODE != kDense) && a.kv_chunk_map != nullptr;
  if (use_inv) {
    for (int c = threadIdx.x; c < a.n_kv_chunks; c += blockDim.x) inv[c] = -1;
    __syncthreads();
    for (int c = threadIdx.x; c < a.n_kv_chunks; c += blockDim.x) {
      const int lc = __ldg(a.kv_chunk_map + c);
      if (lc >= 0 && lc < a.n_kv_chunks) inv[lc] = c;
    }
    __syncthreads();
  }

  const int64_t row = (int64_t)blockIdx.x * kWarps + warp;
  if (row >= (int64_t)a.Tq * a.Hq) return;
  const int i = (int)(row / a.Hq);
  const int h = (int)(row - (int64_t)i * a.Hq);
  const int g = h / (a.Hq / a.Hkv);

  const T* qrow = reinterpret_cast<const T*>(a.q) + i * a.q_stride_t + h * a.q_stride_h;
  for (int d = lane; d < Dqk; d += 32) qs[d] = to_f32(qrow[d]);
  __syncwarp();

  const T* kb = reinterpret_cast<const T*>(a.k) + g * a.k_stride_h;
  const T* vb = reinterpret_cast<const T*>(a.v) + g * a.v_stride_h;
  const int64_t qpos = query_pos(a, i);
  const KeyInterval iv = allowed_interval(a, qpos);
  const int64_t Tk = a.Tk;

  Summary<VPL> tot;
  tot.reset();

  if (MODE == kDense) {
    const int64_t L = a.kv_chunk_map ? a.chunk_len : (Tk > 0 ? Tk : 1);
    for (int pc = 0; pc < p.n_parts; ++pc) {
      Summary<VPL> cur;
      cur.reset();
      Summary<VPL>& st = PARTIALS ? cur : tot;
      const int64_t r0 = (int64_t)pc * p.part_len;
      const int64_t r1 = min(r0 + (int64_t)p.part_len, Tk);
      for (int64_t c = r0 / L; c * L < r1 && iv.lo <= iv.hi; ++c) {
        const int64_t P0 = max(c * L, r0), P1 = min((c + 1) * L, r1);  // physical [P0, P1)
        const int64_t lbase = logical_pos(a.kv_chunk_map, a.chunk_len, P0);
        const int64_t x0 = max(lbase, iv.lo), x1 = min(lbase + (P1 - P0) - 1, iv.hi);
        for (int64_t j0 = x0; j0 <= x1; j0 += 32) {
          const int64_t jl = j0 + lane;
          const int64_t j = (jl <= x1) ? P0 + (jl - lbase) : -1;
          fold_group<T, VPL>(st, qs, kb, vb, a.k_stride_t, a.v_stride_t, Dqk, Dv, a.scale, j, lane);
        }
      }
      if (PARTIALS) {
        const int64_t off = ((int64_t)pc * a.Tq + i) * a.Hq + h;
        write_final<float, VPL>(cur, a.partial_o + off * Dv, a.partial_lse + off, Dv, lane);
        merge_into(tot, cur);
      }
    }
  } else {
    const int32_t* idx = p.sp.indices +
        ((int64_t)i * p.sp.index_heads + (p.sp.index_heads == 1 ? 0 : h)) * p.sp.topk;
    const int64_t L = a.chunk_len;
    auto physical = [&](int64_t jl) -> int64_t {
      if (!use_inv) return jl;
      const int pc = inv[jl / L];
      return pc < 0 ? -1 : (int64_t)pc * L + (jl % L);
    };
    if (MODE == kTokens) {
      for (int t0 = 0; t0 < p.sp.topk; t0 += 32) {
        const int t = t0 + lane;
        int64_t j = -1;
        if (t < p.sp.topk) {
          const int64_t e = __ldg(idx + t);
          if (e < -1 || e >= Tk) {
            report_status(a.dev_status, CPATTN_ERR_BAD_INDEX);
          } else if (e >= 0 && e >= iv.lo && e <= iv.hi) {
            j = physical(e);
          }
        }
        fold_group<T, VPL>(tot, qs, kb, vb, a.k_stride_t, a.v_stride_t, Dqk, Dv, a.scale, j, lane);
      }
    } else {
      const int64_t B = p.sp.block_size;
      for (int t = 0; t < p.sp.topk; ++t) {
        const int64_t e = __ldg(idx + t);
        if (e == -1) continue;
        if (e < -1 || e * B >= Tk) {
          if (lane == 0) report_status(a.dev_status, CPATTN_ERR_BAD_INDEX);
          continue;
        }
        const int64_t x0 = max(e * B, iv.lo), x1 = min(min(e * B + B, Tk) - 1, iv.hi);
        for (int64_t j0 = x0; j0 <= x1; j0 += 32) {
          const int64_t jl = j0 + lane;
          const int64_t j = (jl <= x1) ? physical(jl) : -1;
          fold_group<T, VPL>(tot, qs, kb, vb, a.k_stride_t, a.v_stride_t, Dqk, Dv, a.scale, j, lane);
        }
      }
    }
  }

  if (a.o == nullptr) return;   // partial summaries only (kv_chunk_len > 0)
  T* orow = reinterpret_cast<T*>(a.o) + i * a.o_stride_t + h * a.o_stride_h;
  write_final<T, VPL>(tot, orow, a.lse ? a.lse + row : nullptr, Dv, lane);
}

template <typename T, int VPL, int MODE, bool PARTIALS>
cudaError_t launch_t(const RowParams& p, cudaStream_t stream) {
  const int64_t rows = (int64_t)p.a.Tq * p.a.Hq;
  const int64_t blocks = (rows + kWarps - 1) / kWarps;
  size_t smem = (size_t)kWarps * p.a.Dqk * sizeof(float);
  if (MODE != kDense && p.a.kv_chunk_map) smem += (size_t)p.a.n_kv_chunks * sizeof(int);
  auto kern = rowwise_attn_kernel<T, VPL, MODE, PARTIALS>;
  if (smem > 48 * 1024) {
    cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), (int)smem);
    if (e != cudaSuccess) return e;
  }
  kern<<<(unsigned)blocks, kWarps * 32, smem, stream>>>(p);
  return cudaGetLastError();
}

template <typename T, int VPL>
cudaError_t launch_mode(const RowParams& p, KeyMode mode, cudaStream_t s) {
  if (mode == kTokens) return launch_t<T, VPL, kTokens, false>(p, s);
  if (mode == kBlocks) return launch_t<T, VPL, kBlocks, false>(p, s);
  if (p.a.kv_chunk_len > 0) return launch_t<T, VPL, kDense, true>(p, s);
  return launch_t<T, VPL, kDense, false>(p, s);
}

template <typename T>
cudaError_t launch_dtype(const RowParams& p, KeyMode mode, cudaStream_t s) {
  const int Dv = p.a.Dv;
  if (Dv <= 64) return launch_mode<T, 2>(p, mode, s);
  if (Dv <= 128) return launch_mode<T, 4>(p, mode, s);
  if (Dv <= 256) return launch_mode<T, 8>(p, mode, s);
  return launch_mode<T, 16>(p, mode, s);
}

}  // namespace

cudaError_t launch_rowwise(const cpattn_attn_args& a, KeyMode mode, const SparseArgs& sp,
                           cudaStream_t stream) {
  if ((int64_t)a.Tq * a.Hq == 0) return cudaSuccess;
  RowParams p;
  p.a = a;
  p.sp = sp;
  if (mode == kDense && a.kv_chunk_len > 0) {
    p.part_len = a.kv_chunk_len;
    p.n_parts = (int32_t)((a.Tk + a.kv_chunk_len - 1) / a.kv_chunk_len);  // 0 when Tk == 0
  } else {
    p.part_len = a.Tk > 0 ? a.Tk : 1;
    p.n_parts = 1;
  }
  if (a.dtype == CPATTN_BF16) return launch_dtype<__nv_bfloat16>(p, mode, stream);
  return launch_dtype<float>(p, mode, stream);
}

}  // namespace cpattn
