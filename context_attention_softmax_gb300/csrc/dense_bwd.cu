// Backward of the dense CP-chunk attention on the tensor cores (bf16, d = 128).
//
// "Context parallel attention: exchange keys and merge softmax globally",
// para 2: backward must return each chunk's contributions to the owners of
// K and V - so dk and dv cover every gathered KV row, and each is what this
// chunk's queries add (summing over chunks is the caller's collective); para
// 4: the probabilities are rebuilt from the forward's saved statistics.
// With P[i, j] = exp(s_ij - LSE_i) on permitted pairs (0 elsewhere), g = dO
// and D_i = <g_i, o_i> (= sum_j P_ij dP_ij):
//   dv_j = sum_i P_ij g_i,   dP_ij = <g_i, v_j>,   dS_ij = P_ij (dP_ij - D_i),
//   dq_i = scale sum_j dS_ij k_j,   dk_j = scale sum_i dS_ij q_i,
// dk and dv of a KV head summed over its query heads (GQA).
//
// Three launches, no atomics (the results do not depend on scheduling):
//   bwd_iv_init_kernel, bwd_prep_kernel
//                    D_i and LSE_i in log2 units per (query, head), and the
//                    union of the permitted key intervals of every 128-query
//                    tile (one interval per query: own sequence, cut at qpos);
//   bwd_kernel       two kinds of CTA in one grid:
//     dk/dv CTAs     one per (128-key tile, KV head): for every query head
//                    of the group and every query tile whose interval meets
//                    the key tile,
//                      S^T = K Q^T, dP^T = V g^T      (TMEM, key row = lane)
//                      P^T, dS^T written as bf16 over S^T, dP^T
//                      dv += P^T g,  dk += dS^T Q      (A operand from TMEM)
//     dq CTAs        one per (128-query tile, query head): for every live
//                    key tile, S = Q K^T, dP = g V^T, dS over S, dq += dS K.
// TMA loads 128 x 128 tiles as two 64-column 128-byte-swizzled boxes; one
// tile serves as a K-major operand (the S and dP products) and as an
// MN-major one (the gradient products) without a copy.
//
// Every wait is bounded (wait_limit_ns, 2 s by default); on expiry a CTA
// drains its copies and MMAs in flight, frees TMEM and writes
// CPATTN_ERR_TIMEOUT to dev_status.
#include "dense_tc_common.cuh"

namespace cpattn {
namespace {

constexpr int kBwdThreads = 384;    // warp 0 TMA, 1 MMA, 3 tile list, 4-11 element work
// Element warps 4..11: warp w works on TMEM lanes 32 (w % 4) .. + 31 (its rows)
// and on columns [64 hc, 64 hc + 64) of them, hc = (w - 4) / 4, so each
// sub-partition runs two element warps.
constexpr int kElemThreads = 256;
constexpr int kMaxQTiles = 8192;    // Tq <= 1 Mi tokens on this path

struct BwdParams {
  cpattn_attn_args a;
  const __nv_bfloat16* g;           // dO [Tq, Hq, 128]
  int64_t g_st, g_sh;
  float* dq; int64_t dq_st, dq_sh;  // fp32 [Tq, Hq, 128]
  float* dk; int64_t dk_st, dk_sh;  // fp32 [Tk, Hkv, 128]
  float* dv; int64_t dv_st, dv_sh;  // fp32 [Tk, Hkv, 128]
  float* dvec;                      // [Tq, Hq]  D_i
  float* lse2;                      // [Tq, Hq]  LSE_i * log2(e)
  int2* qt_iv;                      // [n_qtiles] union of the tiles' key intervals (lo, hi)
  int n_qtiles, n_ktiles;
};

// ---------------------------------------------------------------- prep
// One warp per (query, head): D = <g, o> (4 channels per lane) and LSE in
// log2 units.  Warp 0 of every block also folds 32 queries' intervals into
// their tile's union.
__global__ void bwd_prep_kernel(const BwdParams p) {
  const cpattn_attn_args& a = p.a;
  const int lane = threadIdx.x & 31;
  const int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (row < (int64_t)a.Tq * a.Hq) {
    const int64_t t = row / a.Hq;
    const int h = (int)(row - t * a.Hq);
    const __nv_bfloat16* o = reinterpret_cast<const __nv_bfloat16*>(a.o) + t * a.o_stride_t +
                             (int64_t)h * a.o_stride_h + 4 * lane;
    const __nv_bfloat16* g = p.g + t * p.g_st + (int64_t)h * p.g_sh + 4 * lane;
    const uint2 ow = *reinterpret_cast<const uint2*>(o);
    const uint2 gw = *reinterpret_cast<const uint2*>(g);
    float d = __uint_as_float(ow.x << 16) * __uint_as_float(gw.x << 16);
    d = fmaf(__uint_as_float(ow.x & 0xffff0000u), __uint_as_float(gw.x & 0xffff0000u), d);
    d = fmaf(__uint_as_float(ow.y << 16), __uint_as_float(gw.y << 16), d);
    d = fmaf(__uint_as_float(ow.y & 0xffff0000u), __uint_as_float(gw.y & 0xffff0000u), d);
    d = warp_sum(d);
    if (lane == 0) {
      p.dvec[row] = d;
      const float l = a.lse[row];
      p.lse2[row] = l * 1.4426950408889634f;   // -inf stays -inf
    }
  }
  // tile intervals: thread i of the grid handles query i (heads share positions)
  const int64_t qi = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (qi < (int64_t)p.n_qtiles * BM) {
    long long lo = LLONG_MAX, hi = LLONG_MIN;
    if (qi < a.Tq) {
      const KeyInterval iv = allowed_interval(a, query_pos(a, qi));
      if (iv.lo <= iv.hi) { lo = iv.lo; hi = iv.hi; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      lo = min(lo, __shfl_xor_sync(kFullMask, lo, o));
      hi = max(hi, __shfl_xor_sync(kFullMask, hi, o));
    }
    if (lane == 0) {
      const int qt = (int)(qi / BM);
      const int lo32 = lo == LLONG_MAX ? INT_MAX : (int)min(lo, (long long)INT_MAX);
      const int hi32 = hi == LLONG_MIN ? INT_MIN : (int)min(hi, (long long)INT_MAX);
      atomicMin(&p.qt_iv[qt].x, lo32);
      atomicMax(&p.qt_iv[qt].y, hi32);
    }
  }
}

__global__ void bwd_iv_init_kernel(int2* iv, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) iv[i] = make_int2(INT_MAX, INT_MIN);
}

// Logical key range [first, last] of physical key tile kt (tiles never
// straddle a chunk of the map).
__device__ __forceinline__ void key_tile_range(const cpattn_attn_args& a, int kt, int64_t& first,
                                               int64_t& last) {
  const int64_t j0 = (int64_t)kt * BN;
  first = logical_pos(a.kv_chunk_map, a.chunk_len, j0);
  last = first + min((int64_t)BN, (int64_t)a.Tk - j0) - 1;
}

// ---------------------------------------------------------------- dk, dv
struct DkdvSmem {
  uint8_t k[kTileBytes];
  uint8_t v[kTileBytes];
  uint8_t q[2][kTileBytes];
  uint8_t g[2][kTileBytes];
  uint64_t kv_full, qg_full[2], qg_empty[2], s_full, p_full, acc_done, drain;
  uint32_t tmem_base;
  int abort;
  int n_live;
  int issued;                       // query-tile loads issued (for the drain on abort)
  int4 qinfo[8][BM / 2];            // per element warp: (lo, hi, lse2, D) of its 64 queries
  uint16_t live_qt[kMaxQTiles];
};
constexpr size_t kDkdvSmem = sizeof(DkdvSmem) + 1024;

constexpr uint32_t kColDP = 128, kColDV = 256, kColDK = 384;   // S or S^T at kColS = 0

// One CTA of the dk/dv work: key tile kt of KV head gkv, from CTA index bid.
__device__ __forceinline__ void dkdv_cta(const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                                         const CUtensorMap& tm_v, const CUtensorMap& tm_g,
                                         const BwdParams& p, int bid) {
  extern __shared__ uint8_t smem_raw[];
  DkdvSmem& s = *reinterpret_cast<DkdvSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const cpattn_attn_args& a = p.a;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Key tiles in ascending order, KV heads minor: under a causal mask the
  // early key tiles meet the most query tiles, so the heaviest CTAs are
  // launched first and the light ones fill in behind them.
  const int kt = bid / a.Hkv, gkv = bid % a.Hkv;
  const int group = a.Hq / a.Hkv;
  volatile int* abort_flag = &s.abort;
  const uint64_t lim = wait_limit(a);

  if (threadIdx.x == 0) {
    mbar_init(&s.kv_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.qg_full[i], 1);
      mbar_init(&s.qg_empty[i], 1);
    }
    mbar_init(&s.s_full, 1);
    mbar_init(&s.p_full, kElemThreads);
    mbar_init(&s.acc_done, 1);
    mbar_init(&s.drain, 1);
    s.abort = 0;
    s.issued = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_g);
  }
  if (warp == 1) {
    tmem_alloc(&s.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  int64_t kfirst, klast;
  key_tile_range(a, kt, kfirst, klast);
  if (warp == 3) {   // query tiles whose key intervals meet this key tile
    int base = 0;
    for (int t0 = 0; t0 < p.n_qtiles; t0 += 32) {
      const int t = t0 + lane;
      bool live = false;
      if (t < p.n_qtiles) {
        const int2 iv = p.qt_iv[t];
        live = iv.x <= iv.y && (int64_t)iv.x <= klast && (int64_t)iv.y >= kfirst;
      }
      const unsigned m = __ballot_sync(kFullMask, live);
      if (live) s.live_qt[base + __popc(m & ((1u << lane) - 1))] = (uint16_t)t;
      base += __popc(m);
    }
    if (lane == 0) s.n_live = base;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s.tmem_base;
  const int n_steps = s.n_live * group;   // step = (head of the group, live query tile), head-major

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && n_steps > 0) {
      mbar_arrive_expect_tx(&s.kv_full, 2 * kTileBytes);
      for (int x = 0; x < 2; ++x) {
        tma_load_3d(s.k + x * kHalf, &tm_k, &s.kv_full, 64 * x, gkv, kt * BN);
        tma_load_3d(s.v + x * kHalf, &tm_v, &s.kv_full, 64 * x, gkv, kt * BN);
      }
      int issued = 0;
      for (int it = 0; it < n_steps; ++it) {
        const int b = it & 1;
        if (!mbar_wait(&s.qg_empty[b], ((it >> 1) & 1) ^ 1, abort_flag, lim)) break;
        const int h = gkv * group + it / s.n_live, qt = s.live_qt[it % s.n_live];
        mbar_arrive_expect_tx(&s.qg_full[b], 2 * kTileBytes);
        for (int x = 0; x < 2; ++x) {
          tma_load_3d(s.q[b] + x * kHalf, &tm_q, &s.qg_full[b], 64 * x, h, qt * BM);
          tma_load_3d(s.g[b] + x * kHalf, &tm_g, &s.qg_full[b], 64 * x, h, qt * BM);
        }
        ++issued;
      }
      s.issued = issued;
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the issue loop, converged, and one elected lane
    // issues each MMA group (waits made warp-uniform).
    if (n_steps > 0) {
      auto wait_w = [&](uint64_t* bar, uint32_t ph) {
        return __all_sync(kFullMask, mbar_wait(bar, ph, abort_flag, lim));
      };
      const uint32_t idesc_kk = idesc_bf16_f32(BM, BN, 0, 0);
      const uint32_t idesc_mn = idesc_bf16_f32(BM, HD, 0, 1);
      const uint32_t k_lo = desc_lo(smem_u32(s.k), 16), v_lo = desc_lo(smem_u32(s.v), 16);
      bool ok = wait_w(&s.kv_full, 0);
      for (int it = 0; it < n_steps && ok; ++it) {
        const int b = it & 1;
        if (!wait_w(&s.qg_full[b], (it >> 1) & 1)) { ok = false; break; }
        tc_fence_after();
        const uint32_t q_lo = desc_lo(smem_u32(s.q[b]), 16), g_lo = desc_lo(smem_u32(s.g[b]), 16);
        umma8_ss_kmajor<true>(tmem + kColS, k_lo, q_lo, idesc_kk);    // S^T = K Q^T
        umma8_ss_kmajor<true>(tmem + kColDP, v_lo, g_lo, idesc_kk);   // dP^T = V g^T
        umma_commit<true>(&s.s_full);
        if (!wait_w(&s.p_full, it & 1)) { ok = false; break; }
        tc_fence_after();
        const uint32_t q_mn = desc_lo(smem_u32(s.q[b]), kHalf), g_mn = desc_lo(smem_u32(s.g[b]), kHalf);
        // P^T and dS^T of queries 0..63 sit at columns 0..31 of their
        // regions, those of queries 64..127 at columns 64..95 (one half per
        // element warpgroup); B rows 64.. start 4 K-steps (8 KiB) further on.
        if (it == 0) {
          umma4_ts_mn<0, true>(tmem + kColDV, tmem + kColS, g_mn, idesc_mn);          // dv  = P^T g
          umma4_ts_mn<0, true>(tmem + kColDK, tmem + kColDP, q_mn, idesc_mn);         // dk  = dS^T q
        } else {
          umma4_ts_mn<1, true>(tmem + kColDV, tmem + kColS, g_mn, idesc_mn);          // dv += P^T g
          umma4_ts_mn<1, true>(tmem + kColDK, tmem + kColDP, q_mn, idesc_mn);         // dk += dS^T q
        }
        umma4_ts_mn<1, true>(tmem + kColDV, tmem + kColS + 64, g_mn + 512, idesc_mn);
        umma4_ts_mn<1, true>(tmem + kColDK, tmem + kColDP + 64, q_mn + 512, idesc_mn);
        umma_commit<true>(&s.qg_empty[b]);
      }
      if (ok) umma_commit<true>(&s.acc_done);
      umma_commit<true>(&s.drain);
      int no_abort = 0;
      mbar_wait(&s.drain, 0, &no_abort, 1000000000ull);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ P^T, dS^T; epilogue
    const int ew = warp - 4, hc = ew >> 2;                // column half of this warp
    const int r = (ew & 3) * 32 + lane;                   // key row = TMEM lane
    const uint32_t lane_base = (uint32_t)((ew & 3) * 32) << 16;
    const int64_t jrow = (int64_t)kt * BN + r;
    const bool key_ok = jrow < a.Tk;
    const int kpos = key_ok ? (int)logical_pos(a.kv_chunk_map, a.chunk_len, jrow) : INT_MIN;
    const float sl2 = a.scale * 1.4426950408889634f;
    int4* qinfo = s.qinfo[ew];                            // this warp's own copy
    bool ok = true;
    for (int it = 0; it < n_steps; ++it) {
      const int h = gkv * group + it / s.n_live, qt = s.live_qt[it % s.n_live];
      // every warp stages the statistics of its 64 queries in its own copy
      // (lane l: queries 64 hc + l and 64 hc + l + 32), so no barrier spans warps
      __syncwarp();
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int c = lane + 32 * u;
        const int64_t qi = (int64_t)qt * BM + 64 * hc + c;
        int lo = INT_MAX, hi = INT_MIN;
        float l2 = -CUDART_INF_F, dd = 0.f;
        if (qi < a.Tq) {
          const KeyInterval iv = allowed_interval(a, query_pos(a, qi));
          if (iv.lo <= iv.hi) {
            lo = (int)iv.lo;
            hi = (int)min(iv.hi, (int64_t)INT_MAX);
          }
          l2 = p.lse2[qi * a.Hq + h];
          dd = p.dvec[qi * a.Hq + h];
        }
        if (!(l2 > -CUDART_INF_F)) { lo = INT_MAX; hi = INT_MIN; l2 = 0.f; }
        qinfo[c] = make_int4(lo, hi, __float_as_int(l2), __float_as_int(dd));
      }
      __syncwarp();
      ok = __all_sync(kFullMask, mbar_wait(&s.s_full, it & 1, abort_flag, lim));
      if (!ok) break;
      tc_fence_after();
#pragma unroll 1
      for (int c2 = 0; c2 < 2; ++c2) {
        const int c4 = 2 * hc + c2;                       // 32-column chunk of the row
        uint32_t sr[32], dr[32];
        tmem_ld32(tmem + lane_base + kColS + 32 * c4, sr);
        tmem_ld32(tmem + lane_base + kColDP + 32 * c4, dr);
        tmem_wait_ld();
        uint32_t pk[16], dk2[16];
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          float pp[2], ds[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int4 qc = qinfo[32 * c2 + c + e];
            const bool allowed = kpos >= qc.x && kpos <= qc.y;
            const float x = fmaf(__uint_as_float(sr[c + e]), sl2, -__int_as_float(qc.z));
            pp[e] = allowed ? ex2_approx(x) : 0.f;
            ds[e] = pp[e] * (__uint_as_float(dr[c + e]) - __int_as_float(qc.w));
          }
          pk[c >> 1] = pack_bf16(pp[0], pp[1]);
          dk2[c >> 1] = pack_bf16(ds[0], ds[1]);
        }
        // packed into this half's own columns, which it has already read:
        // queries 64 hc .. 64 hc + 63 at columns 64 hc .. 64 hc + 31
        tmem_st16(tmem + lane_base + kColS + 64 * hc + 16 * c2, pk);
        tmem_st16(tmem + lane_base + kColDP + 64 * hc + 16 * c2, dk2);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&s.p_full);
    }
    // epilogue: dv and scale * dk for this CTA's key rows (zero if no step);
    // this warp writes channels [64 hc, 64 hc + 64) of its rows
    const bool have = ok && n_steps > 0 &&
                      __all_sync(kFullMask, mbar_wait(&s.acc_done, 0, abort_flag, lim));
    if (have) tc_fence_after();
    // Stores go row-contiguously through a staging slice per warp in the
    // first query tile buffer, which no copy or MMA touches any more once
    // acc_done has completed; without it (abort or no step) rows are written
    // directly.
    float* dvrow = p.dv + jrow * p.dv_st + (int64_t)gkv * p.dv_sh;
    float* dkrow = p.dk + jrow * p.dk_st + (int64_t)gkv * p.dk_sh;
    float (*stage)[kStageStride] =
        reinterpret_cast<float (*)[kStageStride]>(s.q[0] + (size_t)(warp - 4) * kStageSliceBytes);
    const StagedRows tv = staged_rows(dvrow, key_ok), tk = staged_rows(dkrow, key_ok);
#pragma unroll 1
    for (int c2 = 0; c2 < 2; ++c2) {
      const int c4 = 2 * hc + c2;
      uint32_t vv[32], kk[32];
      if (have) {
        tmem_ld32(tmem + lane_base + kColDV + 32 * c4, vv);
        tmem_ld32(tmem + lane_base + kColDK + 32 * c4, kk);
        tmem_wait_ld();
        store_rows32(stage, tv, vv, 1.f, 32 * c4);
        store_rows32(stage, tk, kk, a.scale, 32 * c4);
      } else if (key_ok) {
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
          *reinterpret_cast<float4*>(dvrow + 32 * c4 + i) = make_float4(0.f, 0.f, 0.f, 0.f);
          *reinterpret_cast<float4*>(dkrow + 32 * c4 + i) = make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (s.abort && warp == 0 && lane == 0 && n_steps > 0) {
    // every role has stopped: let the copies still in flight land (at most
    // the last two query-tile loads; earlier ones were consumed)
    int no_abort = 0;
    mbar_wait(&s.kv_full, 0, &no_abort, 200000000ull);
    for (int j = max(0, s.issued - 2); j < s.issued; ++j)
      mbar_wait(&s.qg_full[j & 1], (j >> 1) & 1, &no_abort, 200000000ull);
  }
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
  if (threadIdx.x == 0 && s.abort) report_status(a.dev_status, CPATTN_ERR_TIMEOUT);
}

// ---------------------------------------------------------------- dq
struct DqSmem {
  uint8_t q[kTileBytes];
  uint8_t g[kTileBytes];
  uint8_t k[2][kTileBytes];
  uint8_t v[2][kTileBytes];
  uint64_t qg_full, kv_full[2], kv_empty[2], s_full, p_full, acc_done, drain;
  uint32_t tmem_base;
  int abort;
  int n_live;
  int issued;
  uint16_t live_kt[kMaxKTiles];
};
constexpr size_t kDqSmem = sizeof(DqSmem) + 1024;

constexpr uint32_t kColDQ = 256;

// One CTA of the dq work: query tile qt of query head h, from CTA index bid.
__device__ __forceinline__ void dq_cta(const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                                       const CUtensorMap& tm_v, const CUtensorMap& tm_g,
                                       const BwdParams& p, int bid) {
  extern __shared__ uint8_t smem_raw[];
  DqSmem& s = *reinterpret_cast<DqSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                         ~uintptr_t(1023));
  const cpattn_attn_args& a = p.a;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Query tiles in descending order, heads minor: later query tiles see the
  // most key tiles under a causal mask, so they are launched first.
  const int qt = p.n_qtiles - 1 - bid / a.Hq, h = bid % a.Hq;
  const int gkv = h / (a.Hq / a.Hkv);
  volatile int* abort_flag = &s.abort;
  const uint64_t lim = wait_limit(a);

  if (threadIdx.x == 0) {
    mbar_init(&s.qg_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.kv_full[i], 1);
      mbar_init(&s.kv_empty[i], 1);
    }
    mbar_init(&s.s_full, 1);
    mbar_init(&s.p_full, kElemThreads);
    mbar_init(&s.acc_done, 1);
    mbar_init(&s.drain, 1);
    s.abort = 0;
    s.issued = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_g);
  }
  if (warp == 1) {
    tmem_alloc(&s.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  if (warp == 3) {   // key tiles that meet the union of this query tile's intervals
    const int2 iv = p.qt_iv[qt];
    int base = 0;
    for (int t0 = 0; t0 < p.n_ktiles; t0 += 32) {
      const int t = t0 + lane;
      bool live = false;
      if (t < p.n_ktiles && iv.x <= iv.y) {
        int64_t f, l;
        key_tile_range(a, t, f, l);
        live = (int64_t)iv.x <= l && (int64_t)iv.y >= f;
      }
      const unsigned m = __ballot_sync(kFullMask, live);
      if (live) s.live_kt[base + __popc(m & ((1u << lane) - 1))] = (uint16_t)t;
      base += __popc(m);
    }
    if (lane == 0) s.n_live = base;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s.tmem_base;
  const int n_steps = s.n_live;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && n_steps > 0) {
      mbar_arrive_expect_tx(&s.qg_full, 2 * kTileBytes);
      for (int x = 0; x < 2; ++x) {
        tma_load_3d(s.q + x * kHalf, &tm_q, &s.qg_full, 64 * x, h, qt * BM);
        tma_load_3d(s.g + x * kHalf, &tm_g, &s.qg_full, 64 * x, h, qt * BM);
      }
      int issued = 0;
      for (int it = 0; it < n_steps; ++it) {
        const int b = it & 1;
        if (!mbar_wait(&s.kv_empty[b], ((it >> 1) & 1) ^ 1, abort_flag, lim)) break;
        const int kt = s.live_kt[it];
        mbar_arrive_expect_tx(&s.kv_full[b], 2 * kTileBytes);
        for (int x = 0; x < 2; ++x) {
          tma_load_3d(s.k[b] + x * kHalf, &tm_k, &s.kv_full[b], 64 * x, gkv, kt * BN);
          tma_load_3d(s.v[b] + x * kHalf, &tm_v, &s.kv_full[b], 64 * x, gkv, kt * BN);
        }
        ++issued;
      }
      s.issued = issued;
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the issue loop, converged, and one elected lane
    // issues each MMA group (waits made warp-uniform).
    if (n_steps > 0) {
      auto wait_w = [&](uint64_t* bar, uint32_t ph) {
        return __all_sync(kFullMask, mbar_wait(bar, ph, abort_flag, lim));
      };
      const uint32_t idesc_kk = idesc_bf16_f32(BM, BN, 0, 0);
      const uint32_t idesc_mn = idesc_bf16_f32(BM, HD, 0, 1);
      const uint32_t q_lo = desc_lo(smem_u32(s.q), 16), g_lo = desc_lo(smem_u32(s.g), 16);
      bool ok = wait_w(&s.qg_full, 0);
      for (int it = 0; it < n_steps && ok; ++it) {
        const int b = it & 1;
        if (!wait_w(&s.kv_full[b], (it >> 1) & 1)) { ok = false; break; }
        tc_fence_after();
        umma8_ss_kmajor<true>(tmem + kColS, q_lo, desc_lo(smem_u32(s.k[b]), 16), idesc_kk);    // S = Q K^T
        umma8_ss_kmajor<true>(tmem + kColDP, g_lo, desc_lo(smem_u32(s.v[b]), 16), idesc_kk);   // dP = g V^T
        umma_commit<true>(&s.s_full);
        if (!wait_w(&s.p_full, it & 1)) { ok = false; break; }
        tc_fence_after();
        const uint32_t k_mn = desc_lo(smem_u32(s.k[b]), kHalf);
        // dS of keys 0..63 at columns 0..31, of keys 64..127 at columns 64..95
        if (it == 0) umma4_ts_mn<0, true>(tmem + kColDQ, tmem + kColS, k_mn, idesc_mn);   // dq  = dS k
        else umma4_ts_mn<1, true>(tmem + kColDQ, tmem + kColS, k_mn, idesc_mn);           // dq += dS k
        umma4_ts_mn<1, true>(tmem + kColDQ, tmem + kColS + 64, k_mn + 512, idesc_mn);
        umma_commit<true>(&s.kv_empty[b]);
      }
      if (ok) umma_commit<true>(&s.acc_done);
      umma_commit<true>(&s.drain);
      int no_abort = 0;
      mbar_wait(&s.drain, 0, &no_abort, 1000000000ull);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ dS; epilogue
    const int ew = warp - 4, hc = ew >> 2;                // column half of this warp
    const int r = (ew & 3) * 32 + lane;                   // query row = TMEM lane
    const uint32_t lane_base = (uint32_t)((ew & 3) * 32) << 16;
    const int64_t qi = (int64_t)qt * BM + r;
    KeyInterval iv{1, 0};
    float l2 = -CUDART_INF_F, dd = 0.f;
    if (qi < a.Tq) {
      iv = allowed_interval(a, query_pos(a, qi));
      l2 = p.lse2[qi * a.Hq + h];
      dd = p.dvec[qi * a.Hq + h];
    }
    if (!(l2 > -CUDART_INF_F)) iv = KeyInterval{1, 0};
    const float sl2 = a.scale * 1.4426950408889634f;
    bool ok = true;
    for (int it = 0; it < n_steps; ++it) {
      const int kt = s.live_kt[it];
      int64_t kf, kl;
      key_tile_range(a, kt, kf, kl);
      int lo_c = 1, hi_c = 0;
      if (iv.lo <= iv.hi) {
        lo_c = (int)max((int64_t)0, min((int64_t)BN, iv.lo - kf));
        hi_c = (int)max((int64_t)-1, min(kl - kf, iv.hi - kf));
      }
      ok = __all_sync(kFullMask, mbar_wait(&s.s_full, it & 1, abort_flag, lim));
      if (!ok) break;
      tc_fence_after();
#pragma unroll 1
      for (int c2 = 0; c2 < 2; ++c2) {
        const int c4 = 2 * hc + c2;                       // 32-key chunk of the row
        uint32_t sr[32], dr[32];
        tmem_ld32(tmem + lane_base + kColS + 32 * c4, sr);
        tmem_ld32(tmem + lane_base + kColDP + 32 * c4, dr);
        tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          float ds[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int kc = 32 * c4 + c + e;
            const float pp = (kc >= lo_c && kc <= hi_c)
                                 ? ex2_approx(fmaf(__uint_as_float(sr[c + e]), sl2, -l2)) : 0.f;
            ds[e] = pp * (__uint_as_float(dr[c + e]) - dd);
          }
          pk[c >> 1] = pack_bf16(ds[0], ds[1]);
        }
        tmem_st16(tmem + lane_base + kColS + 64 * hc + 16 * c2, pk);   // own columns, already read
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&s.p_full);
    }
    const bool have = ok && n_steps > 0 &&
                      __all_sync(kFullMask, mbar_wait(&s.acc_done, 0, abort_flag, lim));
    if (have) tc_fence_after();
    // row-contiguous stores through a staging slice per warp in the first
    // key tile buffer (idle once acc_done has completed), as for dk and dv
    float* dqrow = p.dq + qi * p.dq_st + (int64_t)h * p.dq_sh;
    float (*stage)[kStageStride] =
        reinterpret_cast<float (*)[kStageStride]>(s.k[0] + (size_t)(warp - 4) * kStageSliceBytes);
    const StagedRows tq = staged_rows(dqrow, qi < a.Tq);
#pragma unroll 1
    for (int c2 = 0; c2 < 2; ++c2) {                      // channels [64 hc, 64 hc + 64)
      const int c4 = 2 * hc + c2;
      uint32_t qq[32];
      if (have) {
        tmem_ld32(tmem + lane_base + kColDQ + 32 * c4, qq);
        tmem_wait_ld();
        store_rows32(stage, tq, qq, a.scale, 32 * c4);
      } else if (qi < a.Tq) {
#pragma unroll
        for (int i = 0; i < 32; i += 4)
          *reinterpret_cast<float4*>(dqrow + 32 * c4 + i) = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (s.abort && warp == 0 && lane == 0 && n_steps > 0) {
    int no_abort = 0;
    mbar_wait(&s.qg_full, 0, &no_abort, 200000000ull);
    for (int j = max(0, s.issued - 2); j < s.issued; ++j)
      mbar_wait(&s.kv_full[j & 1], (j >> 1) & 1, &no_abort, 200000000ull);
  }
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
  if (threadIdx.x == 0 && s.abort) report_status(a.dev_status, CPATTN_ERR_TIMEOUT);
}

// dk/dv and dq in one launch: the two are independent, and each alone is
// 1.7 waves of CTAs on 152 SMs, so the dq CTAs (listed after the dk/dv
// ones, heaviest first in each part) fill the SMs that the dk/dv tail
// leaves idle.
constexpr size_t kBwdSmem = kDkdvSmem > kDqSmem ? kDkdvSmem : kDqSmem;

__global__ void __launch_bounds__(kBwdThreads, 1) bwd_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_g,
    const BwdParams p) {
  const int n_dkdv = p.n_ktiles * p.a.Hkv;
  if ((int)blockIdx.x < n_dkdv) dkdv_cta(tm_q, tm_k, tm_v, tm_g, p, (int)blockIdx.x);
  else dq_cta(tm_q, tm_k, tm_v, tm_g, p, (int)blockIdx.x - n_dkdv);
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace

bool dense_bwd_supported(const cpattn_attn_args& a) {
  if (a.dtype != CPATTN_BF16 || a.Dqk != HD || a.Dv != HD) return false;
  if (!(a.scale > 0.f)) return false;
  if ((a.q_chunk_map || a.kv_chunk_map) && a.chunk_len % BN != 0) return false;
  if ((a.Tk + BN - 1) / BN > kMaxKTiles || (a.Tq + BM - 1) / BM > kMaxQTiles) return false;
  if (a.q_stride_h <= 0 || a.k_stride_h <= 0 || a.v_stride_h <= 0) return false;
  // key positions and intervals are kept in 32 bits on this path
  if (a.causal_offset + (int64_t)a.Tq + (int64_t)a.Tk >= (int64_t)INT_MAX) return false;
  return true;
}

size_t dense_bwd_workspace(const cpattn_attn_args& a) {
  const size_t rows = (size_t)a.Tq * a.Hq;
  const size_t n_qt = (size_t)(a.Tq + BM - 1) / BM;
  return 2 * align256(rows * sizeof(float)) + align256(n_qt * sizeof(int2));
}

cudaError_t launch_dense_bwd(const cpattn_attn_args& a, const void* g, int64_t g_st, int64_t g_sh,
                             float* dq, int64_t dq_st, int64_t dq_sh, float* dk, int64_t dk_st,
                             int64_t dk_sh, float* dv, int64_t dv_st, int64_t dv_sh, void* ws,
                             cudaStream_t stream) {
  CUtensorMap tq, tk, tv, tg;
  if (!make_map(&tq, a.q, a.Tq, a.Hq, a.q_stride_t, a.q_stride_h) ||
      !make_map(&tk, a.k, a.Tk, a.Hkv, a.k_stride_t, a.k_stride_h) ||
      !make_map(&tv, a.v, a.Tk, a.Hkv, a.v_stride_t, a.v_stride_h) ||
      !make_map(&tg, g, a.Tq, a.Hq, g_st, g_sh))
    return cudaErrorInvalidValue;
  BwdParams p;
  p.a = a;
  p.g = static_cast<const __nv_bfloat16*>(g);
  p.g_st = g_st;
  p.g_sh = g_sh;
  p.dq = dq; p.dq_st = dq_st; p.dq_sh = dq_sh;
  p.dk = dk; p.dk_st = dk_st; p.dk_sh = dk_sh;
  p.dv = dv; p.dv_st = dv_st; p.dv_sh = dv_sh;
  p.n_qtiles = (a.Tq + BM - 1) / BM;
  p.n_ktiles = (a.Tk + BN - 1) / BN;
  char* w = static_cast<char*>(ws);
  const size_t rows = (size_t)a.Tq * a.Hq;
  p.dvec = reinterpret_cast<float*>(w);
  p.lse2 = reinterpret_cast<float*>(w + align256(rows * sizeof(float)));
  p.qt_iv = reinterpret_cast<int2*>(w + 2 * align256(rows * sizeof(float)));
  bwd_iv_init_kernel<<<(p.n_qtiles + 255) / 256, 256, 0, stream>>>(p.qt_iv, p.n_qtiles);
  const int64_t prep_threads = max((int64_t)rows * 32, (int64_t)p.n_qtiles * BM);
  bwd_prep_kernel<<<(unsigned)((prep_threads + 255) / 256), 256, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = ensure_smem_attr(reinterpret_cast<const void*>(bwd_kernel), (int)kBwdSmem);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)(p.n_ktiles * a.Hkv + p.n_qtiles * a.Hq);
  bwd_kernel<<<grid, kBwdThreads, kBwdSmem, stream>>>(tq, tk, tv, tg, p);
  return cudaGetLastError();
}

}  // namespace cpattn
