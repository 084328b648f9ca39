// Dense CP-chunk attention on the tensor cores with the KV work spread evenly
// over every SM.
//
// Same work units as dense_tc_kernel (two 128-row blocks that read one KV
// head), same roles, ping-pong and softmax.  What differs is the schedule:
// when there are fewer units than SMs, or their causal extents differ, one
// unit per CTA leaves SMs idle.  Here the live KV tiles of all units form
// one stream (unit by unit, tile by tile) and persistent CTA g takes stream
// positions [g*W/G, (g+1)*W/G).  A unit cut by a segment boundary is
// computed in pieces; each piece writes its running summary (m, l, z)
// ("Context parallel attention: exchange keys and merge softmax globally"
// para 3) to the workspace, and the CTA that finishes the unit's last piece
// merges the pieces by rescaling to the larger max and writes O and LSE.
//
// The stream needs every unit's live-tile count in every CTA.  A unit's
// permitted keys are one interval of logical positions, found from the
// intervals of its first and last valid rows (they are monotone in the
// query position: packed-sequence bounds and the causal cut both grow with
// it).  Without a KV chunk map its live tiles are one range of tiles; with
// one, a range inside every chunk whose logical keys meet the interval.  So
// each CTA derives all counts itself and no grid-wide step is needed.
//
// Pieces of a unit are counted on a per-(unit, block) word in the workspace whose high
// half carries a per-launch tag, so stale words from earlier launches read as
// zero and the workspace needs no clearing.
#include <atomic>

#include "dense_tc_common.cuh"

namespace cpattn {
namespace {

constexpr int kMaxUnits = 2048;
constexpr int kPartChunks = HD / 4 + 1;   // per row: 32 float4 of z, then (m in log2 units, l, 0, 0)
constexpr float kLn2 = 0.6931471805599453f;
// The producer and MMA loops here also walk the piece list: 72 registers for
// warpgroup 0 (128 * 72 + 256 * 216 = 64512 = 168 * 384).
constexpr uint32_t kBalRegsControl = 72;
static_assert(128 * kBalRegsControl + 256 * kRegsSoftmax <= 168 * kThreads, "register split");

struct BalParams {
  cpattn_attn_args a;
  int n_qtiles;
  int n_ktiles;
  int head_pairs;
  int n_units;
  float4* part;                    // [grid][2 slots][2 blocks][kPartChunks][128 rows]
  unsigned long long* pieces;      // [n_units] (tag << 32) | pieces finished
  unsigned tag;
};

struct BalSmem {
  uint8_t q[2][kTileBytes];
  uint8_t k[NS][kTileBytes];
  uint8_t v[NS][kTileBytes];
  uint64_t q_full, q_empty;
  uint64_t k_full[NS], k_empty[NS], v_full[NS], v_empty[NS];
  uint64_t s_full[2], p_full[2], o_ready[2], o_free[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int merge[2];                    // this CTA finishes block X of the current unit
  int scan[kThreads / 32];
  int pref[kMaxUnits + 1];         // exclusive prefix of live-tile counts; pref[n] = W
};

constexpr size_t kBalSmemBytes = sizeof(BalSmem) + 1024;
static_assert(kBalSmemBytes <= 232448, "shared memory budget");

// Permitted key positions [lo, hi] of the rows of the block starting at
// query row q0 (rows past Tq or outside every packed sequence have none).
// Rows of a block are consecutive logical positions (a block never straddles
// a query chunk), and both ends of a row's interval grow with its position,
// so the first and last valid rows give the block's bounds.
__device__ bool block_bounds(const cpattn_attn_args& a, int q0, int64_t& lo, int64_t& hi) {
  const int64_t t1 = min((int64_t)q0 + BM, (int64_t)a.Tq) - 1;
  if (t1 < q0) return false;
  int64_t qa = query_pos(a, q0), qb = query_pos(a, t1);
  if (a.cu_seqlens != nullptr) {
    qa = max(qa, (int64_t)__ldg(a.cu_seqlens));
    qb = min(qb, (int64_t)__ldg(a.cu_seqlens + a.num_seqs) - 1);
    if (qa > qb) return false;
  }
  const KeyInterval ia = allowed_interval(a, qa), ib = allowed_interval(a, qb);
  lo = ia.lo;
  hi = ib.hi;
  return lo <= hi;
}

// Permitted key interval of work unit u (both blocks).
__device__ bool unit_bounds(const BalParams& p, int u, int64_t& lo, int64_t& hi) {
  lo = INT64_MAX;
  hi = INT64_MIN;
  for (int x = 0; x < 2; ++x) {
    const Block b = block_of(p.a.Hq, p.head_pairs, p.n_qtiles, u, x);
    int64_t l, h;
    if (block_bounds(p.a, b.q0, l, h)) {
      lo = min(lo, l);
      hi = max(hi, h);
    }
  }
  return lo <= hi;
}

// The live KV tiles of a unit with permitted keys [lo, hi], in physical
// order: per KV chunk (the whole key range when there is no chunk map) the
// tiles whose logical keys meet [lo, hi], one range since a chunk's keys are
// consecutive logical positions and tiles never straddle chunks.
struct LiveTiles {
  const cpattn_attn_args* a;
  int64_t lo, hi;
  int n_chunks, clen;   // chunks and keys per chunk (1 and Tk without a map)
  int c, j, j1;         // cursor: chunk c, its tile j (last live one j1)
  __device__ void init(const cpattn_attn_args& args, int64_t l, int64_t h) {
    a = &args;
    lo = l;
    hi = h;
    if (args.kv_chunk_map != nullptr) {
      n_chunks = (args.Tk + args.chunk_len - 1) / args.chunk_len;
      clen = args.chunk_len;
    } else {
      n_chunks = 1;
      clen = args.Tk;
    }
    c = -1;
    j = j1 = 0;
  }
  // live tiles [t0, t1] of chunk cc within the chunk; false if none
  __device__ bool range(int cc, int& t0, int& t1) const {
    const int64_t start = (int64_t)cc * clen;
    const int64_t len = min((int64_t)clen, (int64_t)a->Tk - start);
    const int64_t L = a->kv_chunk_map != nullptr ? (int64_t)__ldg(a->kv_chunk_map + cc) * clen : 0;
    const int64_t l = max(lo, L), h = min(hi, L + len - 1);
    if (l > h) return false;
    t0 = (int)((l - L) / BN);
    t1 = (int)((h - L) / BN);
    return true;
  }
  __device__ int count() const {
    if (lo > hi) return 0;
    int n = 0, t0, t1;
    for (int cc = 0; cc < n_chunks; ++cc)
      if (range(cc, t0, t1)) n += t1 - t0 + 1;
    return n;
  }
  // place the cursor on the t-th live tile
  __device__ void seek(int t) {
    int t0, t1;
    for (c = 0; c < n_chunks; ++c) {
      if (!range(c, t0, t1)) continue;
      if (t <= t1 - t0) {
        j = t0 + t;
        j1 = t1;
        return;
      }
      t -= t1 - t0 + 1;
    }
  }
  // current tile (physical index, logical position of its first key); advance
  __device__ void next(int& kt, int64_t& kb) {
    kt = (int)((int64_t)c * clen / BN) + j;
    kb = (a->kv_chunk_map != nullptr ? (int64_t)__ldg(a->kv_chunk_map + c) * clen : 0) + (int64_t)j * BN;
    if (++j > j1) {
      int t0, t1;
      for (++c; c < n_chunks; ++c)
        if (range(c, t0, t1)) {
          j = t0;
          j1 = t1;
          break;
        }
    }
  }
};

// Largest u with pref[u] <= pos (pos < W, so pref[u + 1] > pos).
__device__ __forceinline__ int unit_at(const int* pref, int n, int pos) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pref[mid] <= pos) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// CTA whose segment [g*W/G, (g+1)*W/G) holds stream position x.
__device__ __forceinline__ int cta_of(int64_t x, int64_t W, int G) {
  return (int)(((x + 1) * G - 1) / W);
}
__device__ __forceinline__ int64_t seg_start(int g, int64_t W, int G) { return (int64_t)g * W / G; }

// Partial-summary slot of CTA g's piece of unit u: 0 if u holds the start of
// g's segment (its first or only piece), 1 otherwise (its last piece).
// Element j of a row is at row[j * BM], so a warp touches 512 contiguous bytes.
__device__ __forceinline__ float4* part_row(const BalParams& p, int g, int slot, int X, int r) {
  return p.part + (((int64_t)g * 2 + slot) * 2 + X) * kPartChunks * BM + r;
}

// Pieces of a unit held by CTAs ca..cb (CTAs with an empty segment hold none).
__device__ __forceinline__ int pieces_of(int ca, int cb, int64_t W, int G) {
  int n = 0;
  for (int c = ca; c <= cb; ++c) n += seg_start(c + 1, W, G) > seg_start(c, W, G);
  return n;
}

// Counts one finished piece of block X of unit u on its tagged word (one
// word per block, so the two blocks of a unit finish independently); true
// for the piece that completes the count (that CTA merges the block).
__device__ bool count_piece(const BalParams& p, int u, int X, int n_pieces) {
  unsigned long long* word = p.pieces + 2 * u + X;
  unsigned long long cur = *reinterpret_cast<volatile unsigned long long*>(word);
  for (int it = 0; it < (1 << 20); ++it) {
    const unsigned long long nxt =
        ((unsigned)(cur >> 32) == p.tag) ? cur + 1 : (((unsigned long long)p.tag << 32) | 1ull);
    const unsigned long long seen = atomicCAS(word, cur, nxt);
    if (seen == cur) return (int)(nxt & 0xffffffffull) == n_pieces;
    cur = seen;
  }
  report_status(p.a.dev_status, CPATTN_ERR_TIMEOUT);
  return false;
}

// Walks the pieces of this CTA's segment: unit u, tiles [t0, t1) of it.
struct PieceWalk {
  const int* pref;
  int n;
  int64_t pos, end;
  int u, t0, t1;
  __device__ bool next() {
    if (pos >= end) return false;
    u = unit_at(pref, n, (int)pos);
    t0 = (int)(pos - pref[u]);
    t1 = (int)(min(end, (int64_t)pref[u + 1]) - pref[u]);
    pos = pref[u] + t1;
    return true;
  }
};

// Final O and LSE of row r of block X of a unit computed in pieces by CTAs
// ca..cb: every piece's summary is rescaled to the largest max and added
// ("... merge softmax globally" para 3-4).  The summaries of up to kMaxP
// pieces are loaded together so that their latencies overlap.
__device__ __noinline__ void merge_unit(const BalParams& p, int X, int r, int pref_u, int ca, int cb,
                                        int64_t W, int G, __nv_bfloat16* orow, float* lse_out) {
  constexpr int kMaxP = 8;
  if (cb - ca + 1 > kMaxP) {
    // many pieces (a unit much longer than a segment): one piece at a time
    float M = -CUDART_INF_F, L = 0.f;
    for (int c = ca; c <= cb; ++c) {
      const int64_t s0 = seg_start(c, W, G);
      if (seg_start(c + 1, W, G) == s0) continue;
      const float4 st = __ldcg(part_row(p, c, pref_u <= s0 ? 0 : 1, X, r) + (HD / 4) * BM);
      if (!(st.y > 0.f)) continue;
      const float Mn = fmaxf(M, st.x);
      const float a0 = ex2_approx(M - Mn), a1 = ex2_approx(st.x - Mn);
      L = L * a0 + st.y * a1;
      M = Mn;
    }
    const bool live = L > 0.f;
    const float inv = live ? 1.f / L : 0.f;
#pragma unroll 1
    for (int c8 = 0; c8 < HD / 8; ++c8) {
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      for (int c = ca; c <= cb && live; ++c) {
        const int64_t s0 = seg_start(c, W, G);
        if (seg_start(c + 1, W, G) == s0) continue;
        const float4* row = part_row(p, c, pref_u <= s0 ? 0 : 1, X, r);
        const float4 st = __ldcg(row + (HD / 4) * BM);
        if (!(st.y > 0.f)) continue;
        const float w = ex2_approx(st.x - M);
        const float4 z0 = __ldcg(row + (2 * c8) * BM);
        const float4 z1 = __ldcg(row + (2 * c8 + 1) * BM);
        acc[0] += z0.x * w; acc[1] += z0.y * w; acc[2] += z0.z * w; acc[3] += z0.w * w;
        acc[4] += z1.x * w; acc[5] += z1.y * w; acc[6] += z1.z * w; acc[7] += z1.w * w;
      }
      uint4 val;
      val.x = pack_bf16(acc[0] * inv, acc[1] * inv);
      val.y = pack_bf16(acc[2] * inv, acc[3] * inv);
      val.z = pack_bf16(acc[4] * inv, acc[5] * inv);
      val.w = pack_bf16(acc[6] * inv, acc[7] * inv);
      *reinterpret_cast<uint4*>(orow + 8 * c8) = val;
    }
    if (lse_out != nullptr) *lse_out = live ? (M + log2f(L)) * kLn2 : -CUDART_INF_F;
    return;
  }
  const float4* rows[kMaxP];
  int np = 0;
  for (int c = ca; c <= cb && np < kMaxP; ++c) {
    const int64_t s0 = seg_start(c, W, G);
    if (seg_start(c + 1, W, G) == s0) continue;   // empty segment: no piece
    rows[np++] = part_row(p, c, pref_u <= s0 ? 0 : 1, X, r);
  }
  float4 st[kMaxP];
#pragma unroll
  for (int i = 0; i < kMaxP; ++i)
    st[i] = i < np ? __ldcg(rows[i] + (HD / 4) * BM) : make_float4(0.f, 0.f, 0.f, 0.f);
  float M = -CUDART_INF_F;
#pragma unroll
  for (int i = 0; i < kMaxP; ++i)
    if (st[i].y > 0.f) M = fmaxf(M, st[i].x);
  float wt[kMaxP], L = 0.f;
#pragma unroll
  for (int i = 0; i < kMaxP; ++i) {
    wt[i] = st[i].y > 0.f ? ex2_approx(st[i].x - M) : 0.f;
    L += st[i].y * wt[i];
  }
  const bool live = L > 0.f;
  const float inv = live ? 1.f / L : 0.f;
  // 64 columns at a time, two pieces per round: 32 loads in flight per thread
#pragma unroll 1
  for (int c64 = 0; c64 < HD / 64; ++c64) {
    float acc[64];
#pragma unroll
    for (int j = 0; j < 64; ++j) acc[j] = 0.f;
#pragma unroll 1
    for (int i = 0; i < np; i += 2) {
      float4 z[2][16];
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int j = 0; j < 16; ++j)
          z[h][j] = (i + h < np) ? __ldcg(rows[i + h] + (16 * c64 + j) * BM)
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const float w = (i + h < np) ? wt[i + h] : 0.f;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          acc[4 * j] += z[h][j].x * w;
          acc[4 * j + 1] += z[h][j].y * w;
          acc[4 * j + 2] += z[h][j].z * w;
          acc[4 * j + 3] += z[h][j].w * w;
        }
      }
    }
#pragma unroll
    for (int j = 0; j < 64; j += 8) {
      uint4 val;
      val.x = pack_bf16(acc[j] * inv, acc[j + 1] * inv);
      val.y = pack_bf16(acc[j + 2] * inv, acc[j + 3] * inv);
      val.z = pack_bf16(acc[j + 4] * inv, acc[j + 5] * inv);
      val.w = pack_bf16(acc[j + 6] * inv, acc[j + 7] * inv);
      *reinterpret_cast<uint4*>(orow + 64 * c64 + j) = val;
    }
  }
  if (lse_out != nullptr) *lse_out = live ? (M + log2f(L)) * kLn2 : -CUDART_INF_F;
}

// Like merge_unit, for the CTA that holds the unit's last running piece when
// every other piece has already been written: its own summary is taken from
// registers and TMEM (z of row r of block X at o_col) instead of the
// workspace.  All lanes of the warp call it (TMEM loads are warp-wide);
// `write` says whether row r is a query row.
__device__ __noinline__ void merge_unit_direct(const BalParams& p, int X, int r, int pref_u, int ca,
                                               int cb, int64_t W, int G, int self, bool ok,
                                               float m_own, float l_own, uint32_t o_col,
                                               bool write, __nv_bfloat16* orow, float* lse_out) {
  constexpr int kMaxP = 8;
  const float4* rows[kMaxP];
  int np = 0;
  for (int c = ca; c <= cb && np < kMaxP; ++c) {
    const int64_t s0 = seg_start(c, W, G);
    if (c == self || seg_start(c + 1, W, G) == s0) continue;
    rows[np++] = part_row(p, c, pref_u <= s0 ? 0 : 1, X, r);
  }
  float4 st[kMaxP];
#pragma unroll
  for (int i = 0; i < kMaxP; ++i)
    st[i] = i < np ? __ldcg(rows[i] + (HD / 4) * BM) : make_float4(0.f, 0.f, 0.f, 0.f);
  if (!ok) l_own = 0.f;
  float M = l_own > 0.f ? m_own : -CUDART_INF_F;
#pragma unroll
  for (int i = 0; i < kMaxP; ++i)
    if (st[i].y > 0.f) M = fmaxf(M, st[i].x);
  const float w_own = l_own > 0.f ? ex2_approx(m_own - M) : 0.f;
  float wt[kMaxP], L = l_own * w_own;
#pragma unroll
  for (int i = 0; i < kMaxP; ++i) {
    wt[i] = st[i].y > 0.f ? ex2_approx(st[i].x - M) : 0.f;
    L += st[i].y * wt[i];
  }
  const bool live = L > 0.f;
  const float inv = live ? 1.f / L : 0.f;
  // 64 columns per round: this piece's z from TMEM and the first other
  // piece's z from the workspace are in flight together
#pragma unroll 1
  for (int c64 = 0; c64 < HD / 64; ++c64) {
    float4 z[16];
    uint32_t oa[32], ob[32];
#pragma unroll
    for (int j = 0; j < 16; ++j)
      z[j] = np > 0 ? __ldcg(rows[0] + (16 * c64 + j) * BM) : make_float4(0.f, 0.f, 0.f, 0.f);
    tmem_ld32(o_col + 64 * c64, oa);
    tmem_ld32(o_col + 64 * c64 + 32, ob);
    tmem_wait_ld();
    float acc[64];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      acc[j] = w_own > 0.f ? __uint_as_float(oa[j]) * w_own : 0.f;
      acc[32 + j] = w_own > 0.f ? __uint_as_float(ob[j]) * w_own : 0.f;
    }
    const float w0 = np > 0 ? wt[0] : 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      acc[4 * j] += z[j].x * w0;
      acc[4 * j + 1] += z[j].y * w0;
      acc[4 * j + 2] += z[j].z * w0;
      acc[4 * j + 3] += z[j].w * w0;
    }
#pragma unroll 1
    for (int i = 1; i < np; ++i) {   // more than two pieces: one more at a time
      float4 zi[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) zi[j] = __ldcg(rows[i] + (16 * c64 + j) * BM);
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        acc[4 * j] += zi[j].x * wt[i];
        acc[4 * j + 1] += zi[j].y * wt[i];
        acc[4 * j + 2] += zi[j].z * wt[i];
        acc[4 * j + 3] += zi[j].w * wt[i];
      }
    }
    if (write) {
#pragma unroll
      for (int j = 0; j < 64; j += 8) {
        uint4 val;
        val.x = pack_bf16(acc[j] * inv, acc[j + 1] * inv);
        val.y = pack_bf16(acc[j + 2] * inv, acc[j + 3] * inv);
        val.z = pack_bf16(acc[j + 4] * inv, acc[j + 5] * inv);
        val.w = pack_bf16(acc[j + 6] * inv, acc[j + 7] * inv);
        *reinterpret_cast<uint4*>(orow + 64 * c64 + j) = val;
      }
    }
  }
  if (write && lse_out != nullptr) *lse_out = live ? (M + log2f(L)) * kLn2 : -CUDART_INF_F;
}

__global__ void __launch_bounds__(kThreads, 1)
dense_tc_bal_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const BalParams p) {
  extern __shared__ uint8_t smem_raw[];
  BalSmem& s = *reinterpret_cast<BalSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  const cpattn_attn_args& a = p.a;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x, g = blockIdx.x, nu = p.n_units;
  const int group = a.Hq / a.Hkv;
  volatile int* abort_flag = &s.abort;
  const uint64_t lim = wait_limit(a);

  if (threadIdx.x == 0) {
    mbar_init(&s.q_full, 1);
    mbar_init(&s.q_empty, 1);
    for (int i = 0; i < NS; ++i) {
      mbar_init(&s.k_full[i], 1);
      mbar_init(&s.k_empty[i], 1);
      mbar_init(&s.v_full[i], 1);
      mbar_init(&s.v_empty[i], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&s.s_full[x], 1);
      mbar_init(&s.p_full[x], 128);
      mbar_init(&s.o_ready[x], 1);
      mbar_init(&s.o_free[x], 128);
    }
    mbar_init(&s.drain, 1);
    s.abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  if (warp == 1) {
    tmem_alloc(&s.tmem_base, kTmemCols);
    tmem_relinquish();
  }

  // Live KV tiles of every unit.
  for (int u = threadIdx.x; u < nu; u += kThreads) {
    int64_t lo, hi;
    int count = 0;
    if (unit_bounds(p, u, lo, hi)) {
      LiveTiles lt;
      lt.init(a, lo, hi);
      count = lt.count();
    }
    s.pref[u] = count;
  }
  __syncthreads();
  {  // exclusive prefix sum of the counts; pref[nu] = W
    const int per = (nu + kThreads - 1) / kThreads;
    const int b0 = min(nu, (int)threadIdx.x * per), b1 = min(nu, b0 + per);
    int sum = 0;
    for (int i = b0; i < b1; ++i) sum += s.pref[i];
    int x = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kFullMask, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) s.scan[warp] = x;
    __syncthreads();
    if (threadIdx.x == 0) {
      int acc = 0;
      for (int w = 0; w < kThreads / 32; ++w) {
        const int t = s.scan[w];
        s.scan[w] = acc;
        acc += t;
      }
      s.pref[nu] = acc;
    }
    __syncthreads();
    int run = s.scan[warp] + x - sum;
    for (int i = b0; i < b1; ++i) {
      const int c = s.pref[i];
      s.pref[i] = run;
      run += c;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s.tmem_base;
  const int64_t W = s.pref[nu];
  const int64_t S0 = W > 0 ? seg_start(g, W, G) : 0, S1 = W > 0 ? seg_start(g + 1, W, G) : 0;

  if (warp < 4) {
  regs_dec<kBalRegsControl>();
  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int gj = 0, pc = 0, k_issued = 0, v_issued = 0;
      bool ok = true;
      PieceWalk pw{s.pref, nu, S0, S1, 0, 0, 0};
      while (ok && pw.next()) {
        const Block b0 = block_of(a.Hq, p.head_pairs, p.n_qtiles, pw.u, 0);
        const Block b1 = block_of(a.Hq, p.head_pairs, p.n_qtiles, pw.u, 1);
        const int kvh = b0.head / group;
        // Q of this unit once the previous piece's S MMAs are done with Q
        if (!mbar_wait(&s.q_empty, (pc & 1) ^ 1, abort_flag, lim)) break;
        mbar_arrive_expect_tx(&s.q_full, 2 * kTileBytes);
        tma_load_3d(s.q[0], &tm_q, &s.q_full, 0, b0.head, b0.q0);
        tma_load_3d(s.q[0] + kHalf, &tm_q, &s.q_full, 64, b0.head, b0.q0);
        tma_load_3d(s.q[1], &tm_q, &s.q_full, 0, b1.head, b1.q0);
        tma_load_3d(s.q[1] + kHalf, &tm_q, &s.q_full, 64, b1.head, b1.q0);
        ++pc;
        int64_t ulo, uhi, kb;
        unit_bounds(p, pw.u, ulo, uhi);
        LiveTiles lt;
        lt.init(a, ulo, uhi);
        lt.seek(pw.t0);
        for (int t = pw.t0; t < pw.t1; ++t) {
          int kt;
          lt.next(kt, kb);
          const int st = gj % NS;
          const uint32_t ph = (gj / NS) & 1;
          if (!mbar_wait(&s.k_empty[st], ph ^ 1, abort_flag, lim)) { ok = false; break; }
          mbar_arrive_expect_tx(&s.k_full[st], kTileBytes);
          tma_load_3d(s.k[st], &tm_k, &s.k_full[st], 0, kvh, kt * BN);
          tma_load_3d(s.k[st] + kHalf, &tm_k, &s.k_full[st], 64, kvh, kt * BN);
          ++k_issued;
          if (!mbar_wait(&s.v_empty[st], ph ^ 1, abort_flag, lim)) { ok = false; break; }
          mbar_arrive_expect_tx(&s.v_full[st], kTileBytes);
          tma_load_3d(s.v[st], &tm_v, &s.v_full[st], 0, kvh, kt * BN);
          tma_load_3d(s.v[st] + kHalf, &tm_v, &s.v_full[st], 64, kvh, kt * BN);
          ++v_issued;
          ++gj;
        }
      }
      if (*abort_flag) {  // let every copy in flight land before the CTA exits
        int no_abort = 0;
        if (pc > 0) mbar_wait(&s.q_full, (pc - 1) & 1, &no_abort, 200000000ull);
        for (int j = max(0, k_issued - NS); j < k_issued; ++j)
          mbar_wait(&s.k_full[j % NS], (j / NS) & 1, &no_abort, 200000000ull);
        for (int j = max(0, v_issued - NS); j < v_issued; ++j)
          mbar_wait(&s.v_full[j % NS], (j / NS) & 1, &no_abort, 200000000ull);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // Per piece: S_A(0) S_B(0) | PV_A(j) S_A(j+1) PV_B(j) S_B(j+1) | ...
    // The first PV of a piece overwrites O_X, so it waits until the softmax
    // warps have read O_X of the previous piece (o_free).
    // The whole warp runs the issue loop, converged, and one elected lane
    // issues each MMA group (waits made warp-uniform).
    {
      auto wait_w = [&](uint64_t* bar, uint32_t ph) {
        return __all_sync(kFullMask, mbar_wait(bar, ph, abort_flag, lim));
      };
      const uint32_t idesc_qk = idesc_bf16_f32(BM, BN, 0, 0);
      const uint32_t idesc_pv = idesc_bf16_f32(BM, HD, 0, 1);
      const uint32_t q_lo0 = desc_lo(smem_u32(s.q[0]), 16), q_lo1 = desc_lo(smem_u32(s.q[1]), 16);
      const uint32_t k_lo0 = desc_lo(smem_u32(s.k[0]), 16), k_lo1 = desc_lo(smem_u32(s.k[1]), 16);
      const uint32_t v_lo0 = desc_lo(smem_u32(s.v[0]), kHalf), v_lo1 = desc_lo(smem_u32(s.v[1]), kHalf);
      auto issue_s = [&](int j, int x) {   // S_x = Q_x K_j^T
        umma8_ss_kmajor<true>(tmem + kColS + x * BN, x ? q_lo1 : q_lo0, (j & 1) ? k_lo1 : k_lo0, idesc_qk);
        umma_commit<true>(&s.s_full[x]);
      };
      auto issue_pv = [&](int j, int x, bool first) {  // O_x (+)= P_x V_j
        const uint32_t d = tmem + kColO + x * HD, pa = tmem + kColS + x * BN;
        const uint32_t vb = (j & 1) ? v_lo1 : v_lo0;
        if (first) umma8_ts_mnmajor<0, true>(d, pa, vb, idesc_pv);
        else umma8_ts_mnmajor<1, true>(d, pa, vb, idesc_pv);
      };
      int gj = 0, pc = 0;
      bool ok = true;
      PieceWalk pw{s.pref, nu, S0, S1, 0, 0, 0};
      while (ok && pw.next()) {
        const int n = pw.t1 - pw.t0;
        if (!wait_w(&s.q_full, pc & 1) ||
            !wait_w(&s.k_full[gj % NS], (gj / NS) & 1)) { ok = false; break; }
        tc_fence_after();
        issue_s(gj, 0);
        issue_s(gj, 1);
        umma_commit<true>(&s.k_empty[gj % NS]);
        if (n == 1) umma_commit<true>(&s.q_empty);
        for (int jt = 0; jt < n && ok; ++jt) {
          const int j = gj + jt, st = j % NS, st1 = (j + 1) % NS;
          const bool more = jt + 1 < n;
          // block A: PV_A(j), then S_A(j+1)
          if (!wait_w(&s.v_full[st], (j / NS) & 1) ||
              !wait_w(&s.p_full[0], j & 1) ||
              (jt == 0 && pc > 0 && !wait_w(&s.o_free[0], (pc - 1) & 1))) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_pv(j, 0, jt == 0);
          if (!more) umma_commit<true>(&s.o_ready[0]);
          if (more) {
            if (!wait_w(&s.k_full[st1], ((j + 1) / NS) & 1)) { ok = false; break; }
            tc_fence_after();
            issue_s(j + 1, 0);
          }
          // block B: PV_B(j), then S_B(j+1)
          if (!wait_w(&s.p_full[1], j & 1) ||
              (jt == 0 && pc > 0 && !wait_w(&s.o_free[1], (pc - 1) & 1))) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_pv(j, 1, jt == 0);
          umma_commit<true>(&s.v_empty[st]);
          if (!more) umma_commit<true>(&s.o_ready[1]);
          if (more) {
            issue_s(j + 1, 1);
            umma_commit<true>(&s.k_empty[st1]);
            if (jt + 2 == n) umma_commit<true>(&s.q_empty);   // last S of the piece
          }
        }
        gj += n;
        ++pc;
      }
      umma_commit<true>(&s.drain);
      int no_abort = 0;
      mbar_wait(&s.drain, 0, &no_abort, 1000000000ull);
    }
  }
  } else {
    regs_inc<kRegsSoftmax>();
    // ------------------------------------------------------------ softmax + epilogue
    const int X = (warp - 4) >> 2;
    const int r = (warp & 3) * 32 + lane;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t s_col = tmem + lane_base + kColS + X * BN;
    const uint32_t o_col = tmem + lane_base + kColO + X * HD;
    const float sl2 = a.scale * 1.4426950408889634f;   // scores in exp2 units

    // Units without a live tile: O = 0, LSE = -inf (CTA u mod G writes them).
    for (int u = g; u < nu; u += G) {
      if (s.pref[u + 1] != s.pref[u]) continue;
      const Block b = block_of(a.Hq, p.head_pairs, p.n_qtiles, u, X);
      const int64_t tok = (int64_t)b.q0 + r;
      if (tok >= a.Tq) continue;
      uint4* orow = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(a.o) + tok * a.o_stride_t +
                                             (int64_t)b.head * a.o_stride_h);
#pragma unroll
      for (int i = 0; i < HD / 8; ++i) orow[i] = make_uint4(0u, 0u, 0u, 0u);
      if (a.lse != nullptr) a.lse[tok * a.Hq + b.head] = -CUDART_INF_F;
    }

    int jt = 0, pc = 0;
    bool ok = true;
    PieceWalk pw{s.pref, nu, S0, S1, 0, 0, 0};
    // Every piece is walked even after an abort, so that both softmax
    // warpgroups pass the same named barriers; the waits then fail at once.
    while (pw.next()) {
      const int u = pw.u;
      const Block b = block_of(a.Hq, p.head_pairs, p.n_qtiles, u, X);
      const int64_t tok = (int64_t)b.q0 + r;
      KeyInterval iv{1, 0};
      if (tok < a.Tq) iv = allowed_interval(a, query_pos(a, tok));
      float m2 = -CUDART_INF_F, l = 0.f;
      int64_t ulo, uhi;
      unit_bounds(p, u, ulo, uhi);
      LiveTiles lt;
      lt.init(a, ulo, uhi);
      lt.seek(pw.t0);
      for (int t = pw.t0; t < pw.t1 && ok; ++t) {
        int kt;
        int64_t kbase;
        lt.next(kt, kbase);
        const int kvalid = min(BN, a.Tk - kt * BN);
        int lo_c = 1, hi_c = 0;   // permitted columns of this row in this tile
        if (iv.lo <= iv.hi) {
          lo_c = (int)max((int64_t)0, min((int64_t)BN, iv.lo - kbase));
          hi_c = (int)max((int64_t)-1, min((int64_t)kvalid - 1, iv.hi - kbase));
        }
        ok = __all_sync(kFullMask, mbar_wait(&s.s_full[X], jt & 1, abort_flag, lim));
        if (!ok) break;
        tc_fence_after();
        float sv[BN];
        {
          uint32_t rr[BN];
          tmem_ld128_sync(s_col, rr);
  #pragma unroll
          for (int c = 0; c < BN; ++c) sv[c] = __uint_as_float(rr[c]);
        }
        if (!(lo_c == 0 && hi_c == BN - 1)) {
  #pragma unroll
          for (int c = 0; c < BN; ++c)
            if (c < lo_c || c > hi_c) sv[c] = -CUDART_INF_F;
        }
        // row max: four independent chains of 3-input max
        float pm[4];
  #pragma unroll
        for (int i = 0; i < 4; ++i) pm[i] = fmaxf(sv[2 * i], sv[2 * i + 1]);
  #pragma unroll
        for (int c = 8; c < BN; c += 8) {
  #pragma unroll
          for (int i = 0; i < 4; ++i) pm[i] = fmax3(pm[i], sv[c + 2 * i], sv[c + 2 * i + 1]);
        }
        float mx = fmax3(pm[0], pm[1], fmaxf(pm[2], pm[3])) * sl2;
        float alpha = 1.f;
        bool rescale = false;
        if (mx > m2) {
          if (m2 == -CUDART_INF_F) {
            m2 = mx;                      // nothing accumulated yet for this row
          } else if (mx > m2 + kRescaleThreshold) {
            alpha = ex2_approx(m2 - mx);
            m2 = mx;
            rescale = true;
          }
        }
        const float mref = (m2 == -CUDART_INF_F) ? 0.f : m2;
        // p = 2^(s*scale*log2e - m): one packed FFMA per two scores, one ex2 each.
        // P_X over the first 64 columns of S_X (column c holds keys 2c, 2c+1),
        // written in two halves as soon as each is packed.
        const uint64_t sl2x2 = f2_pack(sl2, sl2), nm2 = f2_pack(-mref, -mref);
        uint64_t rs2[2] = {0ull, 0ull};
  #pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t pk[32];
  #pragma unroll
          for (int c = 0; c < 32; ++c) {
            const int e = 64 * half + 2 * c;
            float x0, x1;
            f2_unpack(f2_fma(f2_pack(sv[e], sv[e + 1]), sl2x2, nm2), x0, x1);
            const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
            rs2[c & 1] = f2_add(rs2[c & 1], f2_pack(p0, p1));
            pk[c] = pack_bf16(p0, p1);
          }
          tmem_st32(s_col + 32 * half, pk);
        }
        float a0, a1;
        f2_unpack(f2_add(rs2[0], rs2[1]), a0, a1);
        l = l * alpha + (a0 + a1);
        // PV_X(jt-1) has finished: S_X(jt) was issued after it and has landed.
        if (__any_sync(kFullMask, rescale)) {
  #pragma unroll
          for (int c4 = 0; c4 < HD / 32; ++c4) {
            uint32_t oo[32];
            tmem_ld32_sync(o_col + c4 * 32, oo);
  #pragma unroll
            for (int i = 0; i < 32; ++i) oo[i] = __float_as_uint(__uint_as_float(oo[i]) * alpha);
            tmem_st32(o_col + c4 * 32, oo);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&s.p_full[X]);
        ++jt;
      }
      ok = ok && __all_sync(kFullMask, mbar_wait(&s.o_ready[X], pc & 1, abort_flag, lim));
      if (ok) tc_fence_after();
      const int cnt_u = s.pref[u + 1] - s.pref[u];
      const bool whole = pw.t0 == 0 && pw.t1 == cnt_u;
      __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(a.o) + tok * a.o_stride_t +
                            (int64_t)b.head * a.o_stride_h;
      if (whole) {
        // O = z / l, LSE = m + ln l (natural log); no key -> (0, -inf)
        const bool live = ok && l > 0.f;
        const float inv = live ? 1.f / l : 0.f;
#pragma unroll
        for (int c4 = 0; c4 < HD / 32; ++c4) {
          uint32_t oo[32];
          if (ok) {
            tmem_ld32_sync(o_col + c4 * 32, oo);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) oo[i] = 0u;
          }
          if (tok < a.Tq) {
#pragma unroll
            for (int i = 0; i < 32; i += 8) {
              uint4 val;
              val.x = pack_bf16(__uint_as_float(oo[i + 0]) * inv, __uint_as_float(oo[i + 1]) * inv);
              val.y = pack_bf16(__uint_as_float(oo[i + 2]) * inv, __uint_as_float(oo[i + 3]) * inv);
              val.z = pack_bf16(__uint_as_float(oo[i + 4]) * inv, __uint_as_float(oo[i + 5]) * inv);
              val.w = pack_bf16(__uint_as_float(oo[i + 6]) * inv, __uint_as_float(oo[i + 7]) * inv);
              *reinterpret_cast<uint4*>(orow + c4 * 32 + i) = val;
            }
          }
        }
        if (tok < a.Tq && a.lse != nullptr)
          a.lse[tok * a.Hq + b.head] = live ? (m2 + log2f(l)) * kLn2 : -CUDART_INF_F;
        tc_fence_before();
        mbar_arrive(&s.o_free[X]);
      } else {
        // CTAs ca..cb cover the unit; those with an empty segment (possible
        // when there are fewer live tiles than CTAs) hold no piece of it.
        const int ca = cta_of(s.pref[u], W, G), cb = cta_of(s.pref[u + 1] - 1, W, G);
        const bool last = pw.pos >= S1;
        // The last piece of a segment usually ends after the unit's other
        // pieces (they open later segments).  If they are all written, merge
        // straight from this CTA's accumulator.
        // Each block's warpgroup decides for itself (barrier 2 + X).
        const bool lead = (threadIdx.x & 127) == 0;
        bool direct = false;
        if (last && cb - ca + 1 <= 8) {
          if (lead) {
            const unsigned long long cur = atomicAdd(p.pieces + 2 * u + X, 0ull);
            s.merge[X] = ((unsigned)(cur >> 32) == p.tag &&
                          (int)(cur & 0xffffffffull) == pieces_of(ca, cb, W, G) - 1) ? 2 : 0;
            __threadfence();
          }
          named_bar_sync(2 + X, 128);
          direct = s.merge[X] == 2;
        }
        if (direct) {
          merge_unit_direct(p, X, r, s.pref[u], ca, cb, W, G, g, ok, m2, l, o_col, tok < a.Tq, orow,
                            a.lse != nullptr ? a.lse + tok * a.Hq + b.head : nullptr);
          tc_fence_before();
          mbar_arrive(&s.o_free[X]);
        } else {
          // Running summary of this piece to its slot.
          const int slot = (s.pref[u] <= S0) ? 0 : 1;
          float4* prow = part_row(p, g, slot, X, r);
#pragma unroll
          for (int c4 = 0; c4 < HD / 32; ++c4) {
            uint32_t oo[32];
            if (ok) {
              tmem_ld32_sync(o_col + c4 * 32, oo);
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i) oo[i] = 0u;
            }
#pragma unroll
            for (int i = 0; i < 32; i += 4)
              prow[(c4 * 8 + i / 4) * BM] = make_float4(__uint_as_float(oo[i]), __uint_as_float(oo[i + 1]),
                                                        __uint_as_float(oo[i + 2]), __uint_as_float(oo[i + 3]));
          }
          prow[(HD / 4) * BM] = make_float4(ok ? m2 : -CUDART_INF_F, ok ? l : 0.f, 0.f, 0.f);
          tc_fence_before();
          mbar_arrive(&s.o_free[X]);
          {
            // The barrier orders the warpgroup's stores before the lead
            // thread's fence and count (the fence is cumulative), as in a
            // grid-wide barrier; the CTA that completes the count merges.
            named_bar_sync(2 + X, 128);
            if (lead) {
              __threadfence();
              s.merge[X] = count_piece(p, u, X, pieces_of(ca, cb, W, G));
              __threadfence();
            }
            named_bar_sync(2 + X, 128);
            if (s.merge[X] && tok < a.Tq)
              merge_unit(p, X, r, s.pref[u], ca, cb, W, G, orow,
                         a.lse != nullptr ? a.lse + tok * a.Hq + b.head : nullptr);
          }
        }
      }
      ++pc;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
  if (threadIdx.x == 0 && s.abort) report_status(a.dev_status, CPATTN_ERR_TIMEOUT);
}

size_t dense_tc_bal_part_bytes(int grid) {
  return (size_t)grid * 2 * 2 * kPartChunks * BM * sizeof(float4);
}

int dense_tc_grid() {
  const int n_sm = device_sm_count();
  return n_sm > 0 ? n_sm : 1;
}

int dense_units(const cpattn_attn_args& a, int* head_pairs) {
  const int n_qtiles = (a.Tq + BM - 1) / BM;
  *head_pairs = ((a.Hq / a.Hkv) % 2 == 0) ? 1 : 0;
  return *head_pairs ? n_qtiles * (a.Hq / 2) : ((n_qtiles + 1) / 2) * a.Hq;
}

}  // namespace

size_t dense_tc_bal_workspace(const cpattn_attn_args& a) {
  if (!dense_tc_supported(a) || a.kv_chunk_len != 0) return 0;   // no partial summaries here
  int hp = 0;
  const int nu = dense_units(a, &hp);
  if (nu > kMaxUnits) return 0;
  // Cutting units into pieces costs a Q reload, a partial summary and a merge
  // per piece.  Measured on one GB300: with units filling more than 3/4 of
  // the SMs (128 units on 152) one unit per CTA was 2 % faster, and on many
  // short varlen units (256) 34 % faster; balancing pays when most SMs would
  // otherwise idle.
  if (4 * nu > 3 * dense_tc_grid()) return 0;
  // every CTA counts every unit's tiles chunk by chunk
  if (a.kv_chunk_map != nullptr && (int64_t)nu * a.n_kv_chunks > 131072) return 0;
  return dense_tc_bal_part_bytes(dense_tc_grid()) + (size_t)2 * nu * sizeof(unsigned long long);
}

cudaError_t launch_dense_tc_bal(const cpattn_attn_args& a, void* ws, size_t ws_bytes,
                                cudaStream_t stream, bool* launched) {
  *launched = false;
  const size_t need = dense_tc_bal_workspace(a);
  if (need == 0 || ws == nullptr || ws_bytes < need) return cudaSuccess;
  CUtensorMap tq, tk, tv;
  if (!make_map(&tq, a.q, a.Tq, a.Hq, a.q_stride_t, a.q_stride_h) ||
      !make_map(&tk, a.k, a.Tk, a.Hkv, a.k_stride_t, a.k_stride_h) ||
      !make_map(&tv, a.v, a.Tk, a.Hkv, a.v_stride_t, a.v_stride_h))
    return cudaSuccess;
  static std::atomic<unsigned> next_tag{1u};
  BalParams p;
  p.a = a;
  p.n_qtiles = (a.Tq + BM - 1) / BM;
  p.n_ktiles = (a.Tk + BN - 1) / BN;
  p.n_units = dense_units(a, &p.head_pairs);
  const int grid = dense_tc_grid();
  p.part = static_cast<float4*>(ws);
  p.pieces = reinterpret_cast<unsigned long long*>(static_cast<char*>(ws) + dense_tc_bal_part_bytes(grid));
  p.tag = next_tag.fetch_add(1u);
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(dense_tc_bal_kernel), (int)kBalSmemBytes);
  if (e != cudaSuccess) return e;
  dense_tc_bal_kernel<<<grid, kThreads, kBalSmemBytes, stream>>>(tq, tk, tv, p);
  *launched = true;
  return cudaGetLastError();
}

}  // namespace cpattn
