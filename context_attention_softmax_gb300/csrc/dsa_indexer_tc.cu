// DSA indexer scores on the tensor cores.
//
// "[1/2] Enable DSA CP, THD with absorbed MLA - #3674" (sequence diagram:
// QK scores -> top-k) with the workload's indexer rule
//   score(i, j) = sum_h w_h * max(0, <qI[i, h], kI[j]>)
// (fp32 qI [Tq, H, 128], kI [Tk, 128], w [H]).  The selection
// (idx_select_kernel) certifies the exact top-k from any scores S with
// |S - score| <= c * a_i * ||kI_j||, a_i = sum_h |w_h| ||qI[i, h]||, so this
// path only has to compute S quickly and state its c:
//   * every fp32 value x is split into bf16 x1 = bf16(x) and
//     x2 = bf16(x - x1) (x - x1 is exact in fp32; |x - x1 - x2| <= 2^-16 |x|),
//     and <q, k> is taken as q1.k1 + q1.k2 + q2.k1: one bf16 GEMM with
//     K = 3 * 128 ([q1 q1 q2] against [k1 k2 k1]), every product exact,
//     accumulated in fp32 in the tensor core;
//   * leaving out q2.k2 and the split residues costs at most
//     3.02 * 2^-16 sum_d |q_d k_d|; the accumulation, whatever its order and
//     rounding (each of the 24 K = 16 steps adds at most 17 terms and rounds
//     relative to 2^-23 of the running magnitude), at most
//     (3 D + 32) 2^-22 * 1.02 sum_d |q_d k_d|; and sum_d |q_d k_d| <=
//     ||q|| ||k||;
//   * relu is 1-Lipschitz, and the weighted sum over the H heads rounds at
//     most (H + 2) 2^-24 of sum_h |w_h| |T_h|;
// so c = ((3 D + 32) 2^-22 * 1.02 + 3.02 * 2^-16 + (H + 2) 2^-24) * 1.02,
// about 18 times the bound of the fp32 SIMT scores: the band the selection
// re-ranks in float64 widens accordingly.
//
// GEMM rows are (query, head) pairs, row = query * H + head, so a 128-row
// tile holds 128 / H queries with their heads in consecutive TMEM lanes;
// columns are keys, 128 per tile.  The epilogue applies relu and the head
// weight per lane and sums the H lanes of a query by a transpose-reduce of
// shuffles (each lane ends with 32 / H consecutive keys of every 32), then
// stores row-contiguous pieces of the query's score row.  Tiles whose
// queries permit no key of the tile are skipped: the selection never reads
// those scores.
//
// Roles (256 threads): warp 0 TMA producer, warp 1 MMA issuer (converged,
// one elected lane) and TMEM owner (two accumulators), warps 4-7 epilogue.
// Persistent CTAs take tiles in a fixed stride, key tiles fastest, so the
// CTAs running at one time share their query rows in L2.  Every wait is
// bounded; on expiry the CTA drains its copies and MMAs in flight, frees
// TMEM and reports CPATTN_ERR_TIMEOUT in dev_status.
#include <climits>

#include "common.cuh"
#include "internal.h"
#include "sm100.cuh"

namespace cpattn {
namespace {

using namespace sm100;

constexpr int TD = 128;                      // head dim of the indexer
constexpr int TM = 128, TN = 128, TK = 64;   // tile rows, key columns, K per stage
constexpr int kStages = 6;
constexpr int kThreads = 256;
constexpr int kSplitCols = 2 * TD;           // [x1 | x2] per row, bf16
constexpr uint32_t kBox = TM * TK * 2;       // 16 KiB per operand per stage
// K steps of a tile: (A column, B column) of [q1 q1 q2] . [k1 k2 k1]
__constant__ int2 kSteps[6] = {{0, 0}, {64, 64}, {0, 128}, {64, 192}, {128, 0}, {192, 64}};

struct TcIdxParams {
  cpattn_attn_args a;
  const float* w;
  float* S;
  int64_t ldS;
  const int64_t* mt_lo;   // per row tile: the smallest and largest permitted key
  const int64_t* mt_hi;
  int m_tiles, n_tiles;
  int64_t n_total;
};

struct TcIdxSmem {
  uint8_t a[kStages][kBox];
  uint8_t b[kStages][kBox];
  uint64_t full[kStages], empty[kStages];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};
constexpr size_t kTcIdxSmemBytes = sizeof(TcIdxSmem) + 1024;

__device__ __forceinline__ bool tile_live(const TcIdxParams& p, int64_t t, int& mt, int& nt) {
  mt = (int)(t / p.n_tiles);
  nt = (int)(t - (int64_t)mt * p.n_tiles);
  const int64_t lo = p.mt_lo[mt], hi = p.mt_hi[mt], k0 = (int64_t)nt * TN;
  return lo <= hi && k0 <= hi && k0 + TN - 1 >= lo;
}

// x -> [bf16(x) | bf16(x - bf16(x))] for every row of qI (row = query * H +
// head) and of kI.
__global__ void idx_split_kernel(const cpattn_attn_args a, __nv_bfloat16* __restrict__ qs,
                                 __nv_bfloat16* __restrict__ ks) {
  const int64_t nq = (int64_t)a.Tq * a.Hq * (TD / 4), nk = (int64_t)a.Tk * (TD / 4);
  const float* qI = reinterpret_cast<const float*>(a.q);
  const float* kI = reinterpret_cast<const float*>(a.k);
  for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < nq + nk;
       e += (int64_t)gridDim.x * blockDim.x) {
    const bool is_q = e < nq;
    const int64_t f = is_q ? e : e - nq;
    const int64_t row = f / (TD / 4);
    const int d = (int)(f - row * (TD / 4)) * 4;
    float4 x;
    if (is_q) {
      const int64_t i = row / a.Hq, h = row - i * a.Hq;
      x = *reinterpret_cast<const float4*>(qI + i * a.q_stride_t + h * a.q_stride_h + d);
    } else {
      x = *reinterpret_cast<const float4*>(kI + row * a.k_stride_t + d);
    }
    const float v[4] = {x.x, x.y, x.z, x.w};
    uint32_t hw[2], lw[2];
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const __nv_bfloat16 h0 = __float2bfloat16_rn(v[2 * c]), h1 = __float2bfloat16_rn(v[2 * c + 1]);
      const __nv_bfloat16 l0 = __float2bfloat16_rn(v[2 * c] - __bfloat162float(h0));
      const __nv_bfloat16 l1 = __float2bfloat16_rn(v[2 * c + 1] - __bfloat162float(h1));
      __nv_bfloat162 hp = __halves2bfloat162(h0, h1), lp = __halves2bfloat162(l0, l1);
      hw[c] = *reinterpret_cast<uint32_t*>(&hp);
      lw[c] = *reinterpret_cast<uint32_t*>(&lp);
    }
    __nv_bfloat16* dst = (is_q ? qs : ks) + row * kSplitCols + d;
    *reinterpret_cast<uint2*>(dst) = make_uint2(hw[0], hw[1]);
    *reinterpret_cast<uint2*>(dst + TD) = make_uint2(lw[0], lw[1]);
  }
}

// Per row tile (128 / H queries): the smallest lower and largest upper end of
// the permitted key intervals of its queries (lo > hi when none permits any).
__global__ void idx_tile_iv_kernel(const cpattn_attn_args a, int m_tiles, int64_t* __restrict__ mt_lo,
                                   int64_t* __restrict__ mt_hi) {
  const int mt = (int)((blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (mt >= m_tiles) return;
  const int nq = TM / a.Hq;
  long long lo = LLONG_MAX, hi = LLONG_MIN;
  for (int t = lane; t < nq; t += 32) {
    const int64_t i = (int64_t)mt * nq + t;
    if (i >= a.Tq) break;
    const KeyInterval iv = allowed_interval(a, query_pos(a, i));
    const int64_t l = max(iv.lo, (int64_t)0), h = min(iv.hi, (int64_t)a.Tk - 1);
    if (l <= h) {
      lo = min(lo, (long long)l);
      hi = max(hi, (long long)h);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    lo = min(lo, __shfl_xor_sync(kFullMask, lo, o));
    hi = max(hi, __shfl_xor_sync(kFullMask, hi, o));
  }
  if (lane == 0) {
    mt_lo[mt] = lo;
    mt_hi[mt] = hi;
  }
}

template <int H>
__global__ void __launch_bounds__(kThreads, 1)
idx_score_tc_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                    const TcIdxParams p) {
  extern __shared__ uint8_t smem_raw[];
  TcIdxSmem& s = *reinterpret_cast<TcIdxSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
  const cpattn_attn_args& a = p.a;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = &s.abort;
  const uint64_t lim = wait_limit(a);

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&s.full[i], 1);
      mbar_init(&s.empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.acc_full[i], 1);
      mbar_init(&s.acc_empty[i], 128);
    }
    mbar_init(&s.drain, 1);
    s.abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_a);
    tma_prefetch_desc(&tm_b);
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
      int it = 0;   // stage fills issued
      bool ok = true;
      for (int64_t t = blockIdx.x; t < p.n_total && ok; t += gridDim.x) {
        int mt, nt;
        if (!tile_live(p, t, mt, nt)) continue;
        for (int ks = 0; ks < 6; ++ks, ++it) {
          const int st = it % kStages;
          if (!mbar_wait(&s.empty[st], ((it / kStages) & 1) ^ 1, abort_flag, lim)) { ok = false; break; }
          mbar_arrive_expect_tx(&s.full[st], 2 * kBox);
          const int2 c = kSteps[ks];
          tma_load_3d(s.a[st], &tm_a, &s.full[st], c.x, 0, mt * TM);
          tma_load_3d(s.b[st], &tm_b, &s.full[st], c.y, 0, nt * TN);
        }
      }
      if (!ok || *abort_flag) {   // let the copies in flight land before the CTA exits
        // fill j was issued only after fill j - kStages had been consumed
        int no_abort = 0;
        for (int j = max(0, it - kStages); j < it; ++j)
          mbar_wait(&s.full[j % kStages], (j / kStages) & 1, &no_abort, 200000000ull);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the issue loop, converged, and one elected lane
    // issues each MMA (waits made warp-uniform).
    auto wait_w = [&](uint64_t* bar, uint32_t ph) {
      return __all_sync(kFullMask, mbar_wait(bar, ph, abort_flag, lim));
    };
    const uint32_t idesc = idesc_bf16_f32(TM, TN, 0, 0);   // both operands K-major
    int it = 0, ti = 0;
    bool ok = true;
    for (int64_t t = blockIdx.x; t < p.n_total && ok; t += gridDim.x) {
      int mt, nt;
      if (!tile_live(p, t, mt, nt)) continue;
      const int buf = ti & 1;
      if (!wait_w(&s.acc_empty[buf], ((ti >> 1) & 1) ^ 1)) { ok = false; break; }
      tc_fence_after();
      const uint32_t d = tmem + (uint32_t)(buf * TN);
      for (int ks = 0; ks < 6; ++ks, ++it) {
        const int st = it % kStages;
        if (!wait_w(&s.full[st], (it / kStages) & 1)) { ok = false; break; }
        tc_fence_after();
        const uint32_t a_lo = desc_lo(smem_u32(s.a[st]), 16), b_lo = desc_lo(smem_u32(s.b[st]), 16);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          umma_ss_lo<true>(d, a_lo + 2 * k, b_lo + 2 * k, idesc, (ks > 0 || k > 0) ? 1u : 0u);
        umma_commit<true>(&s.empty[st]);
      }
      if (ok) umma_commit<true>(&s.acc_full[buf]);
      ++ti;
    }
    umma_commit<true>(&s.drain);
    int no_abort = 0;
    mbar_wait(&s.drain, 0, &no_abort, 1000000000ull);
  } else if (warp >= 4) {
    // ------------------------------------------------------------ epilogue
    constexpr int kPer = 32 / H;   // keys of every 32 that a lane ends with
    const int r = (warp - 4) * 32 + lane;   // TMEM lane = (query, head) row of the tile
    const uint32_t lane_base = (uint32_t)((warp - 4) * 32) << 16;
    const int hl = r % H;
    const float wh = p.w[hl];
    int ti = 0;
    for (int64_t t = blockIdx.x; t < p.n_total; t += gridDim.x) {
      int mt, nt;
      if (!tile_live(p, t, mt, nt)) continue;
      const int buf = ti & 1;
      const bool ok = __all_sync(kFullMask, mbar_wait(&s.acc_full[buf], (ti >> 1) & 1, abort_flag, lim));
      if (!ok) break;
      tc_fence_after();
      const int64_t i = (int64_t)mt * (TM / H) + r / H;   // query of this row
      float* srow = p.S + i * p.ldS + (int64_t)nt * TN + kPer * hl;
#pragma unroll 1
      for (int c4 = 0; c4 < TN / 32; ++c4) {
        uint32_t acc[32];
        tmem_ld32(tmem + lane_base + (uint32_t)(buf * TN + c4 * 32), acc);
        tmem_wait_ld();
        float v[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) v[k] = wh * fmaxf(__uint_as_float(acc[k]), 0.f);
        // transpose-reduce over the H lanes of the query: at the step with
        // partner distance b the lane keeps the half of its values that its
        // bit b selects and adds the partner's copy of that half
#pragma unroll
        for (int b = H / 2, hs = 16; b >= 1; b >>= 1, hs >>= 1) {
          const bool upper = (lane & b) != 0;
#pragma unroll
          for (int k = 0; k < hs; ++k) {
            const float send = upper ? v[k] : v[hs + k];
            const float keep = upper ? v[hs + k] : v[k];
            v[k] = keep + __shfl_xor_sync(kFullMask, send, b);
          }
        }
        if (i < a.Tq) {
          float* dst = srow + c4 * 32;
          const int64_t col = (int64_t)nt * TN + c4 * 32 + kPer * hl;
          if constexpr (kPer >= 4) {
#pragma unroll
            for (int k = 0; k < kPer; k += 4)
              if (col + k < p.ldS)
                *reinterpret_cast<float4*>(dst + k) = make_float4(v[k], v[k + 1], v[k + 2], v[k + 3]);
          } else {
#pragma unroll
            for (int k = 0; k < kPer; ++k)
              if (col + k < p.ldS) dst[k] = v[k];
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&s.acc_empty[buf]);
      ++ti;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 256);
  if (threadIdx.x == 0 && s.abort) report_status(a.dev_status, CPATTN_ERR_TIMEOUT);
}

template <int H>
cudaError_t launch_score_tc(const CUtensorMap& ta, const CUtensorMap& tb, const TcIdxParams& p,
                            cudaStream_t stream) {
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(idx_score_tc_kernel<H>),
                                   (int)kTcIdxSmemBytes);
  if (e != cudaSuccess) return e;
  const int n_sm = device_sm_count();
  const int64_t grid = p.n_total < n_sm ? p.n_total : n_sm;
  idx_score_tc_kernel<H><<<(unsigned)grid, kThreads, kTcIdxSmemBytes, stream>>>(ta, tb, p);
  return cudaGetLastError();
}

}  // namespace

bool dsa_indexer_tc_supported(const cpattn_attn_args& a) {
  const int H = a.Hq;
  return a.Dqk == TD && a.Tk > 0 && a.Tq > 0 && H >= 1 && H <= 32 && (H & (H - 1)) == 0 &&
         a.q_stride_h % 4 == 0 && a.q_stride_t % 4 == 0 && a.k_stride_t % 4 == 0 &&
         (reinterpret_cast<uintptr_t>(a.q) & 15) == 0 && (reinterpret_cast<uintptr_t>(a.k) & 15) == 0;
}

size_t dsa_indexer_tc_workspace(const cpattn_attn_args& a) {
  const int64_t rows = (int64_t)a.Tq * a.Hq;
  const int64_t m_tiles = (rows + TM - 1) / TM;
  size_t b = (size_t)rows * kSplitCols * 2;
  b = (b + 255) & ~size_t(255);
  b += (size_t)a.Tk * kSplitCols * 2;
  b = (b + 255) & ~size_t(255);
  b += (size_t)m_tiles * 16 + 256;
  return b;
}

float dsa_indexer_tc_bound(const cpattn_attn_args& a) {
  const double u22 = 2.384185791015625e-07, u16 = 1.52587890625e-05, u24 = 5.9604644775390625e-08;
  return (float)(((3.0 * TD + 32.0) * u22 * 1.02 + 3.02 * u16 + (a.Hq + 2.0) * u24) * 1.02);
}

cudaError_t launch_dsa_indexer_scores_tc(const cpattn_attn_args& a, const float* w, float* S,
                                         int64_t ldS, void* tc_ws, cudaStream_t stream) {
  const int64_t rows = (int64_t)a.Tq * a.Hq;
  const int m_tiles = (int)((rows + TM - 1) / TM), n_tiles = (int)((a.Tk + TN - 1) / TN);
  char* p = static_cast<char*>(tc_ws);
  __nv_bfloat16* qs = reinterpret_cast<__nv_bfloat16*>(p);
  size_t off = ((size_t)rows * kSplitCols * 2 + 255) & ~size_t(255);
  __nv_bfloat16* ks = reinterpret_cast<__nv_bfloat16*>(p + off);
  off = (off + (size_t)a.Tk * kSplitCols * 2 + 255) & ~size_t(255);
  int64_t* mt_lo = reinterpret_cast<int64_t*>(p + off);
  int64_t* mt_hi = mt_lo + m_tiles;

  const int64_t n_vec = (rows + a.Tk) * (TD / 4);
  const int n_sm = device_sm_count();
  const int64_t g1 = min((n_vec + 255) / 256, (int64_t)n_sm * 8);
  idx_split_kernel<<<(unsigned)g1, 256, 0, stream>>>(a, qs, ks);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  idx_tile_iv_kernel<<<(unsigned)((m_tiles * 32 + 255) / 256), 256, 0, stream>>>(a, m_tiles, mt_lo, mt_hi);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  CUtensorMap ta, tb;
  const uint64_t da[3] = {(uint64_t)kSplitCols, 1, (uint64_t)rows};
  const uint64_t db[3] = {(uint64_t)kSplitCols, 1, (uint64_t)a.Tk};
  const uint64_t st[2] = {(uint64_t)kSplitCols * 2, (uint64_t)kSplitCols * 2};
  const uint32_t box[3] = {TK, 1, TM};
  if (!encode_bf16_3d(&ta, qs, da, st, box) || !encode_bf16_3d(&tb, ks, db, st, box))
    return cudaErrorInvalidValue;
  TcIdxParams prm;
  prm.a = a;
  prm.w = w;
  prm.S = S;
  prm.ldS = ldS;
  prm.mt_lo = mt_lo;
  prm.mt_hi = mt_hi;
  prm.m_tiles = m_tiles;
  prm.n_tiles = n_tiles;
  prm.n_total = (int64_t)m_tiles * n_tiles;
  switch (a.Hq) {
    case 1: return launch_score_tc<1>(ta, tb, prm, stream);
    case 2: return launch_score_tc<2>(ta, tb, prm, stream);
    case 4: return launch_score_tc<4>(ta, tb, prm, stream);
    case 8: return launch_score_tc<8>(ta, tb, prm, stream);
    case 16: return launch_score_tc<16>(ta, tb, prm, stream);
    case 32: return launch_score_tc<32>(ta, tb, prm, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace cpattn
