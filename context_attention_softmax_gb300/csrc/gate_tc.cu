// MoBA block gate on the tensor cores (bf16 queries, d = 128, at most 128
// key blocks, top-k <= 8).
//
// "MoBA: Mixture of Block Attention for Long-Context LLMs" (para 1 of the
// CP summary): a query scores every key block by its dot product with the
// block's mean key and keeps the top-k.  The selection has to equal the one
// made with float64 means and float64 dot products, so the gates here are
// computed to a certified error bound and only near-ties are re-ranked in
// float64, exactly as the SIMT gate does; what changes is how the gates are
// computed.
//
// Each fp32 block mean mu (rounded from the float64 mean) is split into
// three bf16 terms hi + mid + lo (each the bf16 rounding of what is left),
// which reproduce mu to 2^-24 relative.  q is bf16, so every product q_d *
// term is exact in fp32, and one K = 3 * 128 MMA [q q q] . [hi mid lo]^T
// accumulates the gate in fp32 in the tensor core.  Whatever order and
// rounding the accumulator uses, each of the 24 K = 16 steps adds at most
// 17 terms and rounds relative to 2^-23 of the running magnitude, so
//   |gate - q . mu64| <= e = (3 D + 32) 2^-22 ||q||_2 ||mu||_2 * 1.02
// (the slack also covers the mean's and the split's rounding and the fp32
// norms).  One thread per query row then takes T = the k-th largest lower
// bound g_b - e_b; U = {b : g_b + e_b >= T} contains the exact top-k; if
// |U| == k it is the answer, otherwise U is re-ranked with float64 gates
// (ties to the lower block).
//
// Roles (320 threads): warp 0 TMA (the three mean terms of the current KV
// group once, query tiles double-buffered), warp 1 MMA issuer + TMEM owner
// (two accumulators of N columns), warps 2-5 and 6-9 selection of the even
// and odd tiles (row = TMEM lane).
// Persistent CTAs take contiguous ranges of (head, query tile) items in
// head-major order, so a CTA reloads the means only when the KV group
// changes.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"
#include "sm100.cuh"

namespace cpattn {
namespace {

using namespace sm100;

constexpr int GD = 128;                       // head dim
constexpr int GM = 128;                       // queries per tile (MMA rows)
constexpr int kGateMaxBlocks = 128;
constexpr int kGateMaxTopk = 8;
constexpr int kGateThreads = 320;
constexpr uint32_t kQBox = GM * 128;          // one 64-channel box of a query tile: 16 KiB
constexpr uint32_t kMuBoxMax = kGateMaxBlocks * 128;   // one 64-channel box of a mean term

struct GateTcParams {
  cpattn_attn_args a;
  int B;                 // block size
  int n_blocks;
  int npad;              // MMA N: n_blocks rounded up to 16
  int topk;
  int n_qtiles;
  int n_items;           // Hq * n_qtiles
  const double* mu64;    // [n_blocks][Hkv][D]
  const float* mnorm;    // [Hkv][n_blocks] ||mu||_2 (fp32)
  int32_t* sel;
};

struct GateSmem {
  uint8_t mu[3][2][kMuBoxMax];     // mean terms, two 64-channel boxes each (SW128, K-major)
  uint8_t q[2][2][kQBox];          // query tiles, double-buffered
  float mnorm[2][kGateMaxBlocks];  // ||mu_b||_2 of each selection group's current KV group
  uint64_t mu_full, mu_empty;
  uint64_t q_full[2], q_empty[2];
  uint64_t acc_full[2], acc_free[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};
constexpr size_t kGateSmemBytes = sizeof(GateSmem) + 1024;
static_assert(kGateSmemBytes <= 232448, "shared memory budget");

// Mean terms for the MMA: [Hkv][n_blocks][3 * D] bf16, term t in channels
// [t*D, (t+1)*D): hi = bf16(mu), mid = bf16(mu - hi), lo = bf16(mu - hi - mid);
// and ||mu||_2 in fp32 per (KV head, block).  One warp per mean, 4 channels
// per lane.
__global__ void gate_split_kernel(const float* __restrict__ mu32, int n_blocks, int Hkv,
                                  __nv_bfloat16* __restrict__ parts, float* __restrict__ mnorm) {
  const int lane = threadIdx.x & 31;
  const int64_t n_rows = (int64_t)n_blocks * Hkv;
  for (int64_t row = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5; row < n_rows;
       row += ((int64_t)gridDim.x * blockDim.x) >> 5) {
    const int g = (int)(row % Hkv), b = (int)(row / Hkv);
    const float4 m4 = *reinterpret_cast<const float4*>(mu32 + row * GD + 4 * lane);
    const float m[4] = {m4.x, m4.y, m4.z, m4.w};
    __nv_bfloat16* out = parts + ((int64_t)g * n_blocks + b) * (3 * GD) + 4 * lane;
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const __nv_bfloat16 hi = __float2bfloat16_rn(m[j]);
      const float r1 = m[j] - __bfloat162float(hi);
      const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
      const float r2 = r1 - __bfloat162float(mid);
      out[j] = hi;
      out[GD + j] = mid;
      out[2 * GD + j] = __float2bfloat16_rn(r2);
      ss = fmaf(m[j], m[j], ss);
    }
    ss = warp_sum(ss);
    if (lane == 0) mnorm[(int64_t)g * n_blocks + b] = sqrtf(ss);
  }
}

// Strict ranking order: larger value first, then lower block (branch-free).
__device__ __forceinline__ bool ahead64(double v1, int b1, double v2, int b2) {
  return (v1 > v2) | ((v1 == v2) & (b1 < b2));
}

// The k-th largest of the lower bounds of blocks 0 .. n_cand-1 held in TMEM
// (row = lane, 128 columns from acc): each value passes down a chain of
// KMAX slots kept in descending order by max / min exchanges, so the slots
// end holding the KMAX largest values with multiplicity.  NaN never enters
// (fmaxf / fminf drop it), as NaN gates are never selected.
template <int KMAX>
__device__ __forceinline__ float kth_lower(uint32_t acc, int k, int n_cand) {
  float tv[KMAX];
#pragma unroll
  for (int t = 0; t < KMAX; ++t) tv[t] = -CUDART_INF_F;
#pragma unroll 1
  for (int c = 0; c < 4; ++c) {
    uint32_t rr[32];
    tmem_ld32(acc + 32 * c, rr);
    tmem_wait_ld();
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      float v = (32 * c + j < n_cand) ? __uint_as_float(rr[j]) : -CUDART_INF_F;
#pragma unroll
      for (int t = 0; t < KMAX; ++t) {
        const float hi = fmaxf(tv[t], v);
        v = fminf(tv[t], v);
        tv[t] = hi;
      }
    }
  }
  float T = tv[0];
#pragma unroll
  for (int t = 1; t < KMAX; ++t) T = (t == k - 1) ? tv[t] : T;
  return T;
}

__global__ void __launch_bounds__(kGateThreads, 1)
gate_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_mu,
               const GateTcParams p) {
  extern __shared__ uint8_t smem_raw[];
  GateSmem& s = *reinterpret_cast<GateSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const cpattn_attn_args& a = p.a;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int group = a.Hq / a.Hkv;
  const int i0 = (int)((int64_t)blockIdx.x * p.n_items / gridDim.x);
  const int i1 = (int)((int64_t)(blockIdx.x + 1) * p.n_items / gridDim.x);
  volatile int* abort_flag = &s.abort;
  const uint64_t lim = wait_limit(a);

  if (threadIdx.x == 0) {
    mbar_init(&s.mu_full, 1);
    mbar_init(&s.mu_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.q_full[i], 1);
      mbar_init(&s.q_empty[i], 128);   // the selection group reads ||q|| from the tile
      mbar_init(&s.acc_full[i], 1);
      mbar_init(&s.acc_free[i], 128);
    }
    mbar_init(&s.drain, 1);
    s.abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_mu);
  }
  if (warp == 1) {
    tmem_alloc(&s.tmem_base, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s.tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int cur_g = -1, n_mu = 0, ti = 0;
      const uint32_t mu_bytes = 6u * 128u * (uint32_t)p.npad;
      for (int it = i0; it < i1; ++it, ++ti) {
        const int h = it / p.n_qtiles, qt = it - h * p.n_qtiles, g = h / group;
        if (g != cur_g) {
          // the previous group's means stay until every MMA reading them is done
          if (n_mu > 0 && !mbar_wait(&s.mu_empty, (n_mu - 1) & 1, abort_flag, lim)) break;
          mbar_arrive_expect_tx(&s.mu_full, mu_bytes);
          for (int t = 0; t < 3; ++t)
            for (int kb = 0; kb < 2; ++kb)
              tma_load_3d(s.mu[t][kb], &tm_mu, &s.mu_full, t * GD + kb * 64, 0, g);
          cur_g = g;
          ++n_mu;
        }
        const int st = ti & 1;
        if (!mbar_wait(&s.q_empty[st], ((ti >> 1) & 1) ^ 1, abort_flag, lim)) break;
        mbar_arrive_expect_tx(&s.q_full[st], 2 * kQBox);
        tma_load_3d(s.q[st][0], &tm_q, &s.q_full[st], 0, h, qt * GM);
        tma_load_3d(s.q[st][1], &tm_q, &s.q_full[st], 64, h, qt * GM);
      }
      if (*abort_flag) {   // let copies in flight land before the CTA exits
        int no_abort = 0;
        if (n_mu > 0) mbar_wait(&s.mu_full, (n_mu - 1) & 1, &no_abort, 200000000ull);
        for (int j = max(0, ti - 2); j < ti; ++j)
          mbar_wait(&s.q_full[j & 1], (j >> 1) & 1, &no_abort, 200000000ull);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the issue loop, converged, and one elected lane
    // issues each MMA group (waits made warp-uniform).
    {
      auto wait_w = [&](uint64_t* bar, uint32_t ph) {
        return __all_sync(kFullMask, mbar_wait(bar, ph, abort_flag, lim));
      };
      const uint32_t idesc = idesc_bf16_f32(GM, p.npad, 0, 0);
      uint32_t mlo[3][2], qlo[2][2];
      for (int t = 0; t < 3; ++t)
        for (int kb = 0; kb < 2; ++kb) mlo[t][kb] = desc_lo(smem_u32(s.mu[t][kb]), 16);
      for (int st = 0; st < 2; ++st)
        for (int kb = 0; kb < 2; ++kb) qlo[st][kb] = desc_lo(smem_u32(s.q[st][kb]), 16);
      int cur_g = -1, n_mu = 0, ti = 0;
      bool ok = true;
      for (int it = i0; it < i1 && ok; ++it, ++ti) {
        const int h = it / p.n_qtiles, g = h / group;
        if (g != cur_g) {
          if (!wait_w(&s.mu_full, n_mu & 1)) { ok = false; break; }
          cur_g = g;
          ++n_mu;
        }
        const int st = ti & 1;
        if (!wait_w(&s.q_full[st], (ti >> 1) & 1) ||
            !wait_w(&s.acc_free[st], ((ti >> 1) & 1) ^ 1)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(st * 128);
        // K = 3 x 128: the same query tile against each mean term
#pragma unroll
        for (int t = 0; t < 3; ++t)
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            umma_ss_lo<true>(d, qlo[st][kk >> 2] + (kk & 3) * 2, mlo[t][kk >> 2] + (kk & 3) * 2, idesc,
                       (t | kk) != 0);
        umma_commit<true>(&s.acc_full[st]);
        const bool last_of_group = it + 1 >= i1 || (it + 1) / p.n_qtiles / group != g;
        if (last_of_group) umma_commit<true>(&s.mu_empty);
      }
      umma_commit<true>(&s.drain);
      int no_abort = 0;
      mbar_wait(&s.drain, 0, &no_abort, 1000000000ull);
    }
  } else {
    // ------------------------------------------------------------ selection
    const int grp = (warp - 2) >> 2;     // even or odd tiles, accumulator grp
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;   // query row of the tile = TMEM lane
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const float gamma = (float)(3 * GD + 32) * 2.3841858e-7f * 1.02f;   // (3D + 32) 2^-22, padded
    const int k = p.topk;
    float* mnorm = s.mnorm[grp];
    int cur_g = -1, ti = grp;
    bool ok = true;
    for (int it = i0 + grp; it < i1; it += 2, ti += 2) {
      const int h = it / p.n_qtiles, qt = it - h * p.n_qtiles, g = h / group;
      if (g != cur_g) {   // ||mu_b|| of the new KV group into shared memory
        named_bar_sync(1 + grp, 128);
        for (int b = r; b < p.n_blocks; b += 128) mnorm[b] = p.mnorm[(int64_t)g * p.n_blocks + b];
        named_bar_sync(1 + grp, 128);
        cur_g = g;
      }
      const int st = ti & 1;
      ok = ok && __all_sync(kFullMask, mbar_wait(&s.acc_full[st], (ti >> 1) & 1, abort_flag, lim));
      const int64_t qi = (int64_t)qt * GM + r;
      const bool valid = ok && qi < a.Tq;
      // ||q||^2 of this row from the staged query tile (the MMA that read it
      // is complete: acc_full); the tile is released for the tile after next
      // once the whole group has read it.  Row r of a 64-channel box sits at
      // r * 128 bytes, its 16-byte piece c at ((c ^ (r % 8)) * 16).
      float qss = 0.f;
      if (ok) {
        tc_fence_after();
#pragma unroll
        for (int kb = 0; kb < 2; ++kb) {
          const uint8_t* rowp = s.q[st][kb] + r * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint4 w = *reinterpret_cast<const uint4*>(rowp + ((c ^ (r & 7)) << 4));
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const float lo = __uint_as_float(ws[j] << 16), hi = __uint_as_float(ws[j] & 0xffff0000u);
              qss = fmaf(lo, lo, fmaf(hi, hi, qss));
            }
          }
        }
        mbar_arrive(&s.q_empty[st]);
      }
      if (!valid) qss = 0.f;
      const float ge = gamma * sqrtf(qss);
      const int64_t own = valid ? query_pos(a, qi) / p.B : 0;
      const int n_cand = (int)max((int64_t)0, min((int64_t)p.n_blocks, own));
      // The gates stay in TMEM (row = lane) and are read 32 columns at a
      // time; every loop over them is unrolled and branch-free.  U is kept as
      // a 128-bit mask.
      const uint32_t acc = tmem + lane_base + (uint32_t)(st * 128);
      uint32_t um[4] = {0u, 0u, 0u, 0u};
      bool rerank = false;
      const bool select = __any_sync(kFullMask, valid && n_cand > k);
      if (ok && select) {
        tc_fence_after();
        // lower bounds g_b - e_b written back in place; upper bounds are taken
        // as lower + 2 e_b, which rounding leaves above g_b + e_b by far less
        // than the bound's padding
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t rr[32];
          tmem_ld32(acc + 32 * c, rr);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j)
            rr[j] = __float_as_uint(__uint_as_float(rr[j]) - ge * mnorm[32 * c + j]);
          tmem_st32(acc + 32 * c, rr);
        }
        tmem_wait_st();
        // T: the k-th largest lower bound (with multiplicity), from one pass
        // keeping the k largest in a max/min exchange chain
        const float pv = k <= 4 ? kth_lower<4>(acc, k, n_cand) : kth_lower<kGateMaxTopk>(acc, k, n_cand);
        int n_u = 0;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t rr[32];
          tmem_ld32(acc + 32 * c, rr);
          tmem_wait_ld();
          uint32_t m = 0u;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int b = 32 * c + j;
            m |= (uint32_t)((b < n_cand) & (__uint_as_float(rr[j]) + 2.f * ge * mnorm[b] >= pv)) << j;
          }
          um[c] = m;
          n_u += __popc(m);
        }
        rerank = valid && n_cand > k && n_u != k;
      }
      tc_fence_before();
      mbar_arrive(&s.acc_free[st]);   // the accumulator is free for the tile after next
      if (valid && !rerank) {
        int32_t* out = p.sel + (qi * a.Hq + h) * (k + 1);
        int n = 0;
        if (n_cand <= k) {
          for (; n < n_cand; ++n) out[n] = n;
        } else {
          for (int w = 0; w < 4; ++w)
            for (uint32_t m = um[w]; m != 0u; m &= m - 1u) out[n++] = 32 * w + __ffs(m) - 1;
        }
        out[n] = (int32_t)own;
        for (int x = n + 1; x <= k; ++x) out[x] = -1;
      }
      // Rows whose uncertain set is not exactly k: float64 gates from the
      // float64 means for the members of U, one row at a time by the whole
      // warp (4 channels per lane), ties to the lower block.
      for (unsigned need = __ballot_sync(kFullMask, rerank); need != 0u; need &= need - 1u) {
        const int L = __ffs(need) - 1;
        const int64_t qL = __shfl_sync(kFullMask, qi, L);
        const int64_t ownL = __shfl_sync(kFullMask, own, L);
        uint32_t mL[4];
#pragma unroll
        for (int w = 0; w < 4; ++w) mL[w] = __shfl_sync(kFullMask, um[w], L);
        const __nv_bfloat16* qr = reinterpret_cast<const __nv_bfloat16*>(a.q) + qL * a.q_stride_t +
                                  (int64_t)h * a.q_stride_h + 4 * lane;
        const uint2 qw = *reinterpret_cast<const uint2*>(qr);
        const double q0 = __uint_as_float(qw.x << 16), q1 = __uint_as_float(qw.x & 0xffff0000u);
        const double q2 = __uint_as_float(qw.y << 16), q3 = __uint_as_float(qw.y & 0xffff0000u);
        double tv[kGateMaxTopk];
        int tb[kGateMaxTopk];
        int n_top = 0;
#pragma unroll
        for (int j = 0; j < kGateMaxTopk; ++j) { tv[j] = -CUDART_INF; tb[j] = 0x7fffffff; }
        // The members of U, four at a time: their float64 means are loaded
        // and their gates reduced together, so the loads' latency overlaps;
        // then each is inserted into the ranked list in ascending block order.
        int w = 0;
        uint32_t mcur = mL[0];
        while (true) {
          int bs[4];
          int nb = 0;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            while (mcur == 0u && w < 3) {
              ++w;
              mcur = w == 1 ? mL[1] : (w == 2 ? mL[2] : mL[3]);
            }
            if (mcur != 0u) {
              bs[i] = 32 * w + __ffs(mcur) - 1;
              mcur &= mcur - 1u;
              ++nb;
            } else {
              bs[i] = -1;
            }
          }
          if (nb == 0) break;
          double vs[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int b = bs[i] >= 0 ? bs[i] : 0;
            const double* mu = p.mu64 + ((int64_t)b * a.Hkv + g) * GD + 4 * lane;
            const double2 u0 = *reinterpret_cast<const double2*>(mu);
            const double2 u1 = *reinterpret_cast<const double2*>(mu + 2);
            vs[i] = fma(q3, u1.y, fma(q2, u1.x, fma(q1, u0.y, q0 * u0.x)));
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
            for (int i = 0; i < 4; ++i) vs[i] += __shfl_xor_sync(kFullMask, vs[i], o);
          }
          for (int i = 0; i < nb; ++i) {
            double v = vs[0];
            int vb = bs[0];
#pragma unroll
            for (int x = 1; x < 4; ++x)
              if (x == i) { v = vs[x]; vb = bs[x]; }
            bool placed = false;   // insert (v, vb) into the ranked list of the best k
#pragma unroll
            for (int j = 0; j < kGateMaxTopk; ++j) {
              const bool here = (j < k) & !placed & ((j >= n_top) | ahead64(v, vb, tv[j], tb[j]));
              const double ov = tv[j];
              const int ob = tb[j];
              tv[j] = here ? v : ov;
              tb[j] = here ? vb : ob;
              v = here ? ov : v;
              vb = here ? ob : vb;
              placed = placed | (here & (j >= n_top));
            }
            n_top = min(n_top + 1, k);
          }
        }
        if (lane == L) {
          int ch[kGateMaxTopk];
          int n = 0;
          for (int j = 0; j < n_top; ++j) {
            if (tb[j] == 0x7fffffff) break;   // NaN gates: fewer than k members
            int y = n - 1;                   // ascending block order
            while (y >= 0 && ch[y] > tb[j]) { ch[y + 1] = ch[y]; --y; }
            ch[y + 1] = tb[j];
            ++n;
          }
          int32_t* out = p.sel + (qL * a.Hq + h) * (k + 1);
          for (int x = 0; x < n; ++x) out[x] = ch[x];
          out[n] = (int32_t)ownL;
          for (int x = n + 1; x <= k; ++x) out[x] = -1;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 256);
  if (threadIdx.x == 0 && s.abort) report_status(a.dev_status, CPATTN_ERR_TIMEOUT);
}

bool gate_map(CUtensorMap* m, const void* base, const cuuint64_t (&dims)[3],
              const cuuint64_t (&strides)[2], const cuuint32_t (&box)[3]) {
  const uint64_t d[3] = {dims[0], dims[1], dims[2]};
  const uint64_t s[2] = {strides[0], strides[1]};
  const uint32_t b[3] = {box[0], box[1], box[2]};
  return encode_bf16_3d(m, base, d, s, b);
}

}  // namespace

bool gate_tc_supported(const cpattn_attn_args& a, int32_t block_size, int32_t topk) {
  if (a.dtype != CPATTN_BF16 || a.Dqk != GD || block_size < 1 || topk < 0 || topk > kGateMaxTopk)
    return false;
  const int n_blocks = a.Tk / block_size;
  return n_blocks >= 1 && n_blocks <= kGateMaxBlocks && a.Tq > 0 && a.q_stride_h > 0;
}

// bf16 mean terms [Hkv][n_blocks][3 D], then the norms [Hkv][n_blocks] fp32.
size_t gate_tc_parts_bytes(const cpattn_attn_args& a, int32_t block_size) {
  const size_t rows = (size_t)(a.Tk / block_size) * a.Hkv;
  return rows * 3 * GD * sizeof(__nv_bfloat16) + (rows * sizeof(float) + 15) / 16 * 16;
}

cudaError_t launch_gate_tc(const cpattn_attn_args& a, int32_t block_size, int32_t topk, int32_t* sel,
                           const double* mu64, const float* mu32, void* parts, cudaStream_t stream,
                           bool* launched) {
  *launched = false;
  const int n_blocks = a.Tk / block_size;
  const int npad = (n_blocks + 15) / 16 * 16;
  CUtensorMap tq, tmu;
  const cuuint64_t qd[3] = {(cuuint64_t)GD, (cuuint64_t)a.Hq, (cuuint64_t)a.Tq};
  const cuuint64_t qs[2] = {(cuuint64_t)a.q_stride_h * 2, (cuuint64_t)a.q_stride_t * 2};
  const cuuint32_t qb[3] = {64, 1, (cuuint32_t)GM};
  const cuuint64_t md[3] = {(cuuint64_t)(3 * GD), (cuuint64_t)n_blocks, (cuuint64_t)a.Hkv};
  const cuuint64_t ms[2] = {(cuuint64_t)(3 * GD * 2), (cuuint64_t)n_blocks * 3 * GD * 2};
  const cuuint32_t mb[3] = {64, (cuuint32_t)npad, 1};
  if (!gate_map(&tq, a.q, qd, qs, qb) || !gate_map(&tmu, parts, md, ms, mb)) return cudaSuccess;
  const int64_t rows = (int64_t)n_blocks * a.Hkv;
  float* mnorm = reinterpret_cast<float*>(static_cast<__nv_bfloat16*>(parts) + rows * 3 * GD);
  const int64_t nb8 = (rows + 7) / 8;   // 8 warps per 256-thread block
  gate_split_kernel<<<(int)(nb8 < 4096 ? nb8 : 4096), 256, 0, stream>>>(
      mu32, n_blocks, a.Hkv, static_cast<__nv_bfloat16*>(parts), mnorm);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  GateTcParams p;
  p.a = a;
  p.B = block_size;
  p.n_blocks = n_blocks;
  p.npad = npad;
  p.topk = topk;
  p.n_qtiles = (a.Tq + GM - 1) / GM;
  p.n_items = a.Hq * p.n_qtiles;
  p.mu64 = mu64;
  p.mnorm = mnorm;
  p.sel = sel;
  const int n_sm = device_sm_count();
  e = ensure_smem_attr(reinterpret_cast<const void*>(gate_tc_kernel), (int)kGateSmemBytes);
  if (e != cudaSuccess) return e;
  const int grid = p.n_items < n_sm ? p.n_items : n_sm;
  gate_tc_kernel<<<grid, kGateThreads, kGateSmemBytes, stream>>>(tq, tmu, p);
  *launched = true;
  return cudaGetLastError();
}

}  // namespace cpattn
