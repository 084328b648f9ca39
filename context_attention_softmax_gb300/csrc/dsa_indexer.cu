// DSA indexer: the top-k keys of every query by the indexer score.
//
// "[1/2] Enable DSA CP, THD with absorbed MLA - #3674", sequence diagram:
// the index mask and the varlen bounds, then the indexer's QK scores, then
// top-k, then the sparse gather; "[Feature-request] Context Parallel support
// for DSAttention": the indices are global key positions.  The score (this
// library's reading of the indexer) is
//
//   score(i, j) = sum_h w_h * max(0, <qI[i, h], kI[j]>)
//
// over the keys the layout permits (one interval of logical positions per
// query: the causal prefix inside the query's packed sequence).  The k
// largest scores win, equal scores going to the lower key; the row is
// written ascending, padded with -1.  The selection must equal the one made
// with float64 scores, so:
//
//  1. idx_norm_kernel: ||kI_j|| and a_i = sum_h |w_h| ||qI_ih||, in float64
//     and rounded up to fp32.
//  2. idx_score_kernel: the fp32 scores of 128 queries x 128 keys per CTA
//     (register-tiled: 8 x 8 per thread; the next d-chunk's loads in flight
//     while the current one is multiplied), every dot product accumulated by
//     fma over d in order, then relu, then fma over the heads in order.  So
//       |S_ij - score_ij| <= (D + H) 2^-24 (1 + tiny) ||kI_j|| a_i,
//     and e_ij = c ||kI_j|| a_i with c = (D + H + 4) 2^-24 * 1.02 bounds it.
//  3. idx_select_kernel, one row per CTA pass: with L = S - e and U = S + e
//     (directed rounding), T = the k-th largest L and U* = the (k+1)-th
//     largest U (radix selects on the fp32 bit patterns).  Keys with
//     L > U* are certainly in the top k, keys with U < T certainly out; the
//     keys in between (the band, usually a handful) are scored again in
//     float64 and the best k - |in| of them join, ties to the lower key.
#include "common.cuh"
#include "internal.h"
#include "sm100.cuh"

namespace cpattn {
namespace {

constexpr int kTQ = 128, kTK = 128, kTD = 16;    // score tile: queries x keys x d-chunk
constexpr int kScoreThreads = 256;
constexpr int kSelThreads = 512;
constexpr int kBins = 2048;                      // radix-select digits of 11, 11, 10 bits

__host__ __device__ constexpr int64_t round_up4(int64_t x) { return (x + 3) & ~int64_t(3); }

// fp32 <-> unsigned keys in the order of the values (+0 above -0 is harmless
// here: both map next to each other and no selection depends on the sign of 0).
__device__ __forceinline__ uint32_t ord32(float x) {
  const uint32_t u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ uint64_t ord64(double x) {
  const uint64_t u = (uint64_t)__double_as_longlong(x);
  return (u & 0x8000000000000000ull) ? ~u : (u | 0x8000000000000000ull);
}

// ---------------------------------------------------------------- norms
__global__ void idx_norm_kernel(const cpattn_attn_args a, const float* __restrict__ w,
                                float* __restrict__ kn, float* __restrict__ qa) {
  const int warp = (int)((blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  const int D = a.Dqk, H = a.Hq;
  const float* kI = reinterpret_cast<const float*>(a.k);
  const float* qI = reinterpret_cast<const float*>(a.q);
  if (warp < a.Tk) {
    double ss = 0.0;
    for (int d = lane; d < D; d += 32) {
      const double x = kI[(int64_t)warp * a.k_stride_t + d];
      ss += x * x;
    }
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(kFullMask, ss, o);
    if (lane == 0) kn[warp] = __double2float_ru(sqrt(ss) * (1.0 + 1e-15));
  } else if (warp < a.Tk + a.Tq) {
    const int64_t i = warp - a.Tk;
    double acc = 0.0;
    for (int h = 0; h < H; ++h) {
      double ss = 0.0;
      for (int d = lane; d < D; d += 32) {
        const double x = qI[i * a.q_stride_t + (int64_t)h * a.q_stride_h + d];
        ss += x * x;
      }
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(kFullMask, ss, o);
      acc += fabs((double)w[h]) * sqrt(ss);
    }
    if (lane == 0) qa[i] = __double2float_ru(acc * (1.0 + 1e-15));
  }
}

// ---------------------------------------------------------------- scores
// Thread (ty, tx) of 16 x 16 owns query rows ty*4 + {0..3}, 64 + ty*4 + {0..3}
// and key columns tx*4 + {0..3}, 64 + tx*4 + {0..3} of the 128 x 128 tile.
struct ScoreSmem {
  float a[2][kTD][kTQ + 4];   // qI chunks, d-major, double-buffered
  float b[2][kTD][kTK + 4];   // kI chunks, d-major
  long long lo, hi;           // permitted key range of the tile's query rows
};

__global__ void __launch_bounds__(kScoreThreads)
idx_score_kernel(const cpattn_attn_args a, const float* __restrict__ w, float* __restrict__ S,
                 int64_t ldS) {
  __shared__ ScoreSmem s;
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  const int q0 = blockIdx.y * kTQ, k0 = blockIdx.x * kTK;
  const int D = a.Dqk, H = a.Hq;
  const float* qI = reinterpret_cast<const float*>(a.q);
  const float* kI = reinterpret_cast<const float*>(a.k);
  if (tid == 0) {
    s.lo = LLONG_MAX;
    s.hi = LLONG_MIN;
  }
  __syncthreads();
  if (tid < kTQ && q0 + tid < a.Tq) {
    const KeyInterval iv = allowed_interval(a, query_pos(a, q0 + tid));
    if (iv.lo <= iv.hi) {
      atomicMin(&s.lo, (long long)iv.lo);
      atomicMax(&s.hi, (long long)iv.hi);
    }
  }
  __syncthreads();
  if (s.lo > s.hi || s.hi < k0 || s.lo > k0 + kTK - 1) return;   // no permitted key in the tile

  // chunk c = (head c / nd, d-chunk c % nd); the next chunk's global loads
  // are in flight while the current one is multiplied
  const int nd = (D + kTD - 1) / kTD, nc = H * nd;
  float4 ra[2], rb[2];
  auto load = [&](int c) {
    const int h = c / nd, d0 = (c - h * nd) * kTD;
#pragma unroll
    for (int t = 0; t < 2; ++t) {   // 512 float4 of each operand, two per thread
      const int idx = tid + kScoreThreads * t, r = idx >> 2, c4 = idx & 3;
      const int d = d0 + 4 * c4;
      ra[t] = make_float4(0.f, 0.f, 0.f, 0.f);
      rb[t] = ra[t];
      if (q0 + r < a.Tq && d < D)
        ra[t] = *reinterpret_cast<const float4*>(qI + (int64_t)(q0 + r) * a.q_stride_t +
                                                 (int64_t)h * a.q_stride_h + d);
      if (k0 + r < a.Tk && d < D)
        rb[t] = *reinterpret_cast<const float4*>(kI + (int64_t)(k0 + r) * a.k_stride_t + d);
    }
  };
  auto store = [&](int buf) {
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const int idx = tid + kScoreThreads * t, r = idx >> 2, c4 = idx & 3;
      s.a[buf][4 * c4 + 0][r] = ra[t].x; s.a[buf][4 * c4 + 1][r] = ra[t].y;
      s.a[buf][4 * c4 + 2][r] = ra[t].z; s.a[buf][4 * c4 + 3][r] = ra[t].w;
      s.b[buf][4 * c4 + 0][r] = rb[t].x; s.b[buf][4 * c4 + 1][r] = rb[t].y;
      s.b[buf][4 * c4 + 2][r] = rb[t].z; s.b[buf][4 * c4 + 3][r] = rb[t].w;
    }
  };

  // acc2[i][jp] holds the dots of row i with columns 2 jp and 2 jp + 1 as a
  // packed pair: one f32x2 fma does both (each lane an ordinary fp32 fma,
  // so every dot still accumulates over d in order).
  float sc[8][8];
  uint64_t acc2[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
#pragma unroll
    for (int j = 0; j < 8; ++j) sc[i][j] = 0.f;
#pragma unroll
    for (int jp = 0; jp < 4; ++jp) acc2[i][jp] = 0ull;
  }
  load(0);
  for (int c = 0; c < nc; ++c) {
    const int buf = c & 1;
    store(buf);
    __syncthreads();
    if (c + 1 < nc) load(c + 1);
#pragma unroll
    for (int d = 0; d < kTD; ++d) {   // d ascending: every dot accumulates in order
      const float4 a0 = *reinterpret_cast<const float4*>(&s.a[buf][d][ty * 4]);
      const float4 a1 = *reinterpret_cast<const float4*>(&s.a[buf][d][64 + ty * 4]);
      const float4 b0 = *reinterpret_cast<const float4*>(&s.b[buf][d][tx * 4]);
      const float4 b1 = *reinterpret_cast<const float4*>(&s.b[buf][d][64 + tx * 4]);
      const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const uint64_t bp[4] = {sm100::f2_pack(b0.x, b0.y), sm100::f2_pack(b0.z, b0.w),
                              sm100::f2_pack(b1.x, b1.y), sm100::f2_pack(b1.z, b1.w)};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint64_t ai = sm100::f2_pack(av[i], av[i]);
#pragma unroll
        for (int jp = 0; jp < 4; ++jp) acc2[i][jp] = sm100::f2_fma(ai, bp[jp], acc2[i][jp]);
      }
    }
    if ((c + 1) % nd == 0) {   // a head's dots are complete: relu, weight, add
      const float wh = w[c / nd];
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int jp = 0; jp < 4; ++jp) {
          float d0, d1;
          sm100::f2_unpack(acc2[i][jp], d0, d1);
          sc[i][2 * jp] = fmaf(wh, fmaxf(d0, 0.f), sc[i][2 * jp]);
          sc[i][2 * jp + 1] = fmaf(wh, fmaxf(d1, 0.f), sc[i][2 * jp + 1]);
          acc2[i][jp] = 0ull;
        }
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int row = q0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + (i - 4));
    if (row >= a.Tq) continue;
    float* srow = S + (int64_t)row * ldS + k0;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int col = half * 64 + tx * 4;
      if (k0 + col < ldS)
        *reinterpret_cast<float4*>(srow + col) =
            make_float4(sc[i][4 * half], sc[i][4 * half + 1], sc[i][4 * half + 2], sc[i][4 * half + 3]);
    }
  }
}

// ---------------------------------------------------------------- selection
// Block-wide helpers for 512 threads (16 warps).
struct SelSmem {
  uint32_t hist[kBins];
  uint32_t hist2[kBins];           // the second histogram of select32_pair
  int wsum[kSelThreads / 32];
  int found_digit, found_above;
  int n_in, n_band;
};

// Exclusive prefix sum of v over the block's threads (thread order); also
// returns the block total.  Uses sm.wsum; two barriers.
__device__ __forceinline__ int block_excl_scan(int v, SelSmem& sm, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(kFullMask, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sm.wsum[warp] = x;
  __syncthreads();
  int before = 0;
  total = 0;
  for (int w2 = 0; w2 < kSelThreads / 32; ++w2) {
    const int t = sm.wsum[w2];
    if (w2 < warp) before += t;
    total += t;
  }
  __syncthreads();
  return before + x - v;
}

// The digit holding the kk-th largest key of a histogram of kBins bins, and
// the number of keys in higher digits.  Thread t owns bins 4t .. 4t + 3.
__device__ __forceinline__ void find_digit(SelSmem& sm, int kk, const uint32_t* hist) {
  const int t = threadIdx.x;
  const int c0 = hist[4 * t], c1 = hist[4 * t + 1], c2 = hist[4 * t + 2], c3 = hist[4 * t + 3];
  const int local = c0 + c1 + c2 + c3;
  // suffix sum over threads above t: reverse the order and scan
  const int lane = t & 31, warp = t >> 5;
  int x = local;   // inclusive suffix within the warp (lanes lane .. 31)
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_down_sync(kFullMask, x, o);
    if (lane + o < 32) x += y;
  }
  if (lane == 0) sm.wsum[warp] = x;
  __syncthreads();
  int above = x - local;
  for (int w2 = warp + 1; w2 < kSelThreads / 32; ++w2) above += sm.wsum[w2];
  const int cs[4] = {c0, c1, c2, c3};
  int cum = above;
#pragma unroll
  for (int b = 3; b >= 0; --b) {
    if (cum < kk && cum + cs[b] >= kk) {
      sm.found_digit = 4 * t + b;
      sm.found_above = cum;
    }
    cum += cs[b];
  }
  __syncthreads();
}

// Selections over j in [lo, hi] of 32-bit keys take three radix passes of 11,
// 11 and 10 bits.  Two of them run at once: the kk1-th largest of key1 and
// the kk2-th largest (with multiplicity) of key2, every pass reading each j
// once and filling both histograms.
template <typename KeyFn1, typename KeyFn2>
__device__ void select32_pair(SelSmem& sm, int64_t lo, int64_t hi, int kk1, KeyFn1 key1, int kk2,
                              KeyFn2 key2, uint32_t& out1, uint32_t& out2) {
  uint32_t p1 = 0u, p2 = 0u, pmask = 0u;
  const int shifts[3] = {21, 10, 0}, widths[3] = {11, 11, 10};
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = shifts[pass];
    const uint32_t dmask = (1u << widths[pass]) - 1u;
    for (int b = threadIdx.x; b < kBins; b += kSelThreads) {
      sm.hist[b] = 0u;
      sm.hist2[b] = 0u;
    }
    __syncthreads();
    for (int64_t j = lo + threadIdx.x; j <= hi; j += kSelThreads) {
      const uint32_t x1 = key1(j), x2 = key2(j);
      if ((x1 & pmask) == p1) atomicAdd(&sm.hist[(x1 >> shift) & dmask], 1u);
      if ((x2 & pmask) == p2) atomicAdd(&sm.hist2[(x2 >> shift) & dmask], 1u);
    }
    __syncthreads();
    find_digit(sm, kk1, sm.hist);
    const int d1 = sm.found_digit, a1 = sm.found_above;
    __syncthreads();   // every thread has read the first result
    find_digit(sm, kk2, sm.hist2);
    kk1 -= a1;
    p1 |= (uint32_t)d1 << shift;
    kk2 -= sm.found_above;
    p2 |= (uint32_t)sm.found_digit << shift;
    pmask |= dmask << shift;
    __syncthreads();
  }
  out1 = p1;
  out2 = p2;
}

// The same for 64-bit keys of the band members bk[0 .. n): eight 8-bit passes.
__device__ uint64_t select64(SelSmem& sm, const uint64_t* bk, int n, int kk) {
  uint64_t prefix = 0ull, pmask = 0ull;
  for (int pass = 0; pass < 8; ++pass) {
    const int shift = 56 - 8 * pass;
    for (int b = threadIdx.x; b < kBins; b += kSelThreads) sm.hist[b] = 0u;
    __syncthreads();
    for (int m = threadIdx.x; m < n; m += kSelThreads) {
      const uint64_t x = bk[m];
      if ((x & pmask) == prefix) atomicAdd(&sm.hist[(x >> shift) & 0xffu], 1u);
    }
    __syncthreads();
    find_digit(sm, kk, sm.hist);
    kk -= sm.found_above;
    prefix |= (uint64_t)sm.found_digit << shift;
    pmask |= 0xffull << shift;
    __syncthreads();
  }
  return prefix;
}

// Float64 score of key j for query i by one warp: dots over d in lane order
// then a fixed butterfly, relu, weighted sum over the heads in order.
__device__ double exact_score(const cpattn_attn_args& a, const float* w, int64_t i, int64_t j) {
  const int lane = threadIdx.x & 31;
  const float* qI = reinterpret_cast<const float*>(a.q) + i * a.q_stride_t;
  const float* kI = reinterpret_cast<const float*>(a.k) + j * a.k_stride_t;
  double sc = 0.0;
  for (int h = 0; h < a.Hq; ++h) {
    double part = 0.0;
    for (int d = lane; d < a.Dqk; d += 32)
      part = fma((double)qI[(int64_t)h * a.q_stride_h + d], (double)kI[d], part);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(kFullMask, part, o);
    sc = fma((double)w[h], fmax(part, 0.0), sc);
  }
  return sc;
}

// fp32 score of key j for query i by one thread, in the arithmetic the SIMT
// score kernel uses (fma over d in order, relu, fma over the heads in
// order), so that its error is within (D + H + 4) 2^-24 a_i ||kI_j||.  Rows
// are read as float4 (the tensor-core path, its only user, requires rows
// aligned to 16 bytes and D a multiple of 4).
__device__ float fp32_score(const cpattn_attn_args& a, const float* w, int64_t i, int64_t j) {
  const float* qI = reinterpret_cast<const float*>(a.q) + i * a.q_stride_t;
  const float4* k4 = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(a.k) + j * a.k_stride_t);
  float sc = 0.f;
  for (int h = 0; h < a.Hq; ++h) {
    const float4* q4 = reinterpret_cast<const float4*>(qI + (int64_t)h * a.q_stride_h);
    float acc = 0.f;
#pragma unroll 8
    for (int d4 = 0; d4 < a.Dqk / 4; ++d4) {
      const float4 q = __ldg(q4 + d4), k = __ldg(k4 + d4);
      acc = fmaf(q.x, k.x, acc);
      acc = fmaf(q.y, k.y, acc);
      acc = fmaf(q.z, k.z, acc);
      acc = fmaf(q.w, k.w, acc);
    }
    sc = fmaf(w[h], fmaxf(acc, 0.f), sc);
  }
  return sc;
}

struct SelParams {
  cpattn_attn_args a;
  const float* w;
  int topk;
  const float* S;
  int64_t ldS;
  const float* kn;
  const float* qa;
  float c;                 // bound factor of the scores S
  float c2;                // > 0: S came from the tensor cores; bound factor of fp32_score
  int32_t* band_idx;       // per CTA: Tk entries
  uint64_t* band_key;      // per CTA: Tk entries (ordered float64 bits)
  int32_t* out;            // [Tq, topk]
  int words;               // bitmap words: ceil(Tk / 32)
};

__global__ void __launch_bounds__(kSelThreads) idx_select_kernel(const SelParams p) {
  __shared__ SelSmem sm;
  extern __shared__ uint32_t bits[];            // [words] selected, then [words] equal-at-cut
  uint32_t* sel = bits;
  uint32_t* eq = bits + p.words;
  const cpattn_attn_args& a = p.a;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int32_t* bidx = p.band_idx + (int64_t)blockIdx.x * a.Tk;
  uint64_t* bkey = p.band_key + (int64_t)blockIdx.x * a.Tk;
  for (int64_t i = blockIdx.x; i < a.Tq; i += gridDim.x) {
    int32_t* orow = p.out + i * p.topk;
    const KeyInterval iv = allowed_interval(a, query_pos(a, i));
    const int64_t lo = max(iv.lo, (int64_t)0), hi = min(iv.hi, (int64_t)a.Tk - 1);
    const int64_t n = hi >= lo ? hi - lo + 1 : 0;
    if (n <= p.topk) {   // every permitted key, ascending, then -1
      for (int t = tid; t < p.topk; t += kSelThreads) orow[t] = t < n ? (int32_t)(lo + t) : -1;
      continue;
    }
    const float* srow = p.S + i * p.ldS;
    const float es = __fmul_ru(p.c, p.qa[i]);
    auto lkey = [&](int64_t j) {
      return ord32(__fsub_rd(srow[j], __fmul_ru(es, p.kn[j])));
    };
    auto ukey = [&](int64_t j) {
      return ord32(__fadd_ru(srow[j], __fmul_ru(es, p.kn[j])));
    };
    // T: the k-th largest lower bound; U*: the (k+1)-th largest upper bound
    uint32_t T, Us;
    select32_pair(sm, lo, hi, p.topk, lkey, p.topk + 1, ukey, T, Us);
    const int nw = (int)((n + 31) >> 5);
    for (int x = tid; x < nw; x += kSelThreads) { sel[x] = 0u; eq[x] = 0u; }
    if (tid == 0) { sm.n_in = 0; sm.n_band = 0; }
    __syncthreads();
    // certainly in (L > U*): selected; the band (U >= T, L <= U*): to rank
    int my_in = 0;
    for (int64_t j = lo + tid; j <= hi; j += kSelThreads) {
      const uint32_t l = lkey(j), u = ukey(j);
      if (l > Us) {
        atomicOr(&sel[(j - lo) >> 5], 1u << ((j - lo) & 31));
        ++my_in;
      } else if (u >= T) {
        const int m = atomicAdd(&sm.n_band, 1);
        bidx[m] = (int32_t)j;
      }
    }
    atomicAdd(&sm.n_in, my_in);
    __syncthreads();
    int n_band = sm.n_band, need = p.topk - sm.n_in;
    if (p.c2 > 0.f && need > 0 && n_band > need) {
      // The scores S carry the wide tensor-core bound: narrow the band first
      // with fp32 scores of its members (fma over d in order, relu, fma over
      // the heads in order) and their own bound c2.  Within the band, a key
      // whose lower bound beats the (need+1)-th largest upper bound is in, a
      // key whose upper bound is below the need-th largest lower bound is
      // out; only the rest is ranked in float64.
      for (int m = tid; m < n_band; m += kSelThreads)
        bkey[m] = (uint64_t)__float_as_uint(fp32_score(a, p.w, i, bidx[m]));
      __syncthreads();
      const float es2 = __fmul_ru(p.c2, p.qa[i]);
      auto lkey2 = [&](int64_t m) {
        return ord32(__fsub_rd(__uint_as_float((uint32_t)bkey[m]), __fmul_ru(es2, p.kn[bidx[m]])));
      };
      auto ukey2 = [&](int64_t m) {
        return ord32(__fadd_ru(__uint_as_float((uint32_t)bkey[m]), __fmul_ru(es2, p.kn[bidx[m]])));
      };
      uint32_t T2, U2;
      select32_pair(sm, 0, n_band - 1, need, lkey2, need + 1, ukey2, T2, U2);
      // classify, compacting the undecided members to the front of the list
      // (a member is written at or before its own position, after every
      // member of its pass has been read)
      int n_keep = 0, my_in2 = 0;
      for (int base = 0; base < n_band; base += kSelThreads) {
        const int m = base + tid;
        bool keep = false;
        int32_t j = 0;
        if (m < n_band) {
          j = bidx[m];
          const uint32_t l = lkey2(m), u = ukey2(m);
          if (l > U2) {
            atomicOr(&sel[(j - lo) >> 5], 1u << ((j - lo) & 31));
            ++my_in2;
          } else if (u >= T2) {
            keep = true;
          }
        }
        int kept = 0;
        const int pos = block_excl_scan(keep ? 1 : 0, sm, kept);
        if (keep) bidx[n_keep + pos] = j;
        n_keep += kept;
        __syncthreads();
      }
      int in2 = 0;
      block_excl_scan(my_in2, sm, in2);
      need -= in2;
      n_band = n_keep;
    }
    if (need > 0) {
      // float64 scores of the band, one warp per member
      for (int m = warp; m < n_band; m += kSelThreads / 32) {
        const double v = exact_score(a, p.w, i, bidx[m]);
        if (lane == 0) bkey[m] = ord64(v);
      }
      __threadfence_block();
      __syncthreads();
      const uint64_t t64 = select64(sm, bkey, n_band, need);
      // above the cut: in; at the cut: the lowest keys fill what is left
      int my_gt = 0;
      for (int m = tid; m < n_band; m += kSelThreads) {
        const int64_t j = bidx[m];
        if (bkey[m] > t64) {
          atomicOr(&sel[(j - lo) >> 5], 1u << ((j - lo) & 31));
          ++my_gt;
        } else if (bkey[m] == t64) {
          atomicOr(&eq[(j - lo) >> 5], 1u << ((j - lo) & 31));
        }
      }
      int n_gt = 0;
      block_excl_scan(my_gt, sm, n_gt);
      const int take = need - n_gt;
      // the first `take` keys equal at the cut, in ascending key order
      const int per = (nw + kSelThreads - 1) / kSelThreads;
      const int w0 = tid * per, w1 = min(nw, w0 + per);
      int cnt = 0;
      for (int x = w0; x < w1; ++x) cnt += __popc(eq[x]);
      int total = 0;
      int pos = block_excl_scan(cnt, sm, total);
      for (int x = w0; x < w1 && pos < take; ++x) {
        uint32_t e = eq[x];
        while (e != 0u && pos < take) {
          const int b = __ffs(e) - 1;
          e &= e - 1u;
          atomicOr(&sel[x], 1u << b);
          ++pos;
        }
      }
      __syncthreads();
    }
    // write the selection in ascending key order (exactly topk keys)
    {
      const int per = (nw + kSelThreads - 1) / kSelThreads;
      const int w0 = tid * per, w1 = min(nw, w0 + per);
      int cnt = 0;
      for (int x = w0; x < w1; ++x) cnt += __popc(sel[x]);
      int total = 0;
      int pos = block_excl_scan(cnt, sm, total);
      for (int x = w0; x < w1; ++x) {
        uint32_t e = sel[x];
        while (e != 0u) {
          const int b = __ffs(e) - 1;
          e &= e - 1u;
          if (pos < p.topk) orow[pos] = (int32_t)(lo + 32 * (int64_t)x + b);
          ++pos;
        }
      }
      for (int t = total + tid; t < p.topk; t += kSelThreads) orow[t] = -1;   // not reached: total == topk
      __syncthreads();
    }
  }
}

}  // namespace

size_t dsa_indexer_workspace(const cpattn_attn_args& a, int grid) {
  const int64_t ldS = round_up4(a.Tk);
  size_t b = (size_t)a.Tq * ldS * 4;                   // scores
  b += (size_t)round_up4(a.Tk) * 4 + (size_t)round_up4(a.Tq) * 4;   // key norms, query weights
  b = (b + 255) & ~size_t(255);
  b += (size_t)grid * a.Tk * (4 + 8) + 256;            // band lists
  b = (b + 255) & ~size_t(255);
  if (dsa_indexer_tc_supported(a)) b += dsa_indexer_tc_workspace(a);   // split operands
  return b;
}

int dsa_indexer_grid(const cpattn_attn_args& a) {
  const int n_sm = device_sm_count();
  const int g = 2 * (n_sm > 0 ? n_sm : 1);
  return a.Tq < g ? (a.Tq > 0 ? a.Tq : 1) : g;
}

cudaError_t launch_dsa_indexer(const cpattn_attn_args& a, const float* w, int topk, int32_t* out,
                               void* ws, cudaStream_t stream) {
  if (a.Tq <= 0) return cudaSuccess;
  const int grid = dsa_indexer_grid(a);
  const int64_t ldS = round_up4(a.Tk);
  char* p = static_cast<char*>(ws);
  float* S = reinterpret_cast<float*>(p);
  float* kn = S + (size_t)a.Tq * ldS;
  float* qa = kn + round_up4(a.Tk);
  size_t off = ((size_t)a.Tq * ldS * 4 + (size_t)round_up4(a.Tk) * 4 + (size_t)round_up4(a.Tq) * 4 + 255) &
               ~size_t(255);
  int32_t* band_idx = reinterpret_cast<int32_t*>(p + off);
  uint64_t* band_key = reinterpret_cast<uint64_t*>(
      p + ((off + (size_t)grid * a.Tk * 4 + 7) & ~size_t(7)));
  const int64_t warps = (int64_t)a.Tk + a.Tq;
  idx_norm_kernel<<<(unsigned)((warps * 32 + 255) / 256), 256, 0, stream>>>(a, w, kn, qa);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // scores: on the tensor cores (split operands, wider certified bound) when
  // the shape allows, else the fp32 SIMT kernel
  const bool tc = dsa_indexer_tc_supported(a);
  if (tc) {
    size_t tc_off = ((off + (size_t)grid * a.Tk * (4 + 8) + 256) + 255) & ~size_t(255);
    e = launch_dsa_indexer_scores_tc(a, w, S, ldS, p + tc_off, stream);
    if (e != cudaSuccess) return e;
  } else if (a.Tk > 0) {
    const dim3 g2((unsigned)((a.Tk + kTK - 1) / kTK), (unsigned)((a.Tq + kTQ - 1) / kTQ));
    idx_score_kernel<<<g2, kScoreThreads, 0, stream>>>(a, w, S, ldS);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  SelParams sp;
  sp.a = a;
  sp.w = w;
  sp.topk = topk;
  sp.S = S;
  sp.ldS = ldS;
  sp.kn = kn;
  sp.qa = qa;
  const float c_simt = (float)((a.Dqk + a.Hq + 4) * 5.9604644775390625e-8 * 1.02);
  sp.c = tc ? dsa_indexer_tc_bound(a) : c_simt;
  sp.c2 = tc ? c_simt : 0.f;
  sp.band_idx = band_idx;
  sp.band_key = band_key;
  sp.out = out;
  sp.words = (a.Tk + 31) / 32;
  const size_t smem = (size_t)sp.words * 2 * 4;
  if (smem > 48 * 1024) {
    e = ensure_smem_attr(reinterpret_cast<const void*>(idx_select_kernel), (int)smem);
    if (e != cudaSuccess) return e;
  }
  idx_select_kernel<<<grid, kSelThreads, smem, stream>>>(sp);
  return cudaGetLastError();
}

}  // namespace cpattn
