// Dense CP-chunk attention on the 5th-generation tensor cores (sm_103a).
//
// TMA loads Q/K/V tiles into 128-byte-swizzled shared memory; one elected
// lane of the converged MMA warp issues tcgen05.mma (bf16 x bf16 -> fp32
// accumulators in tensor memory; elect.sync of a full warp always picks the
// same lane, so every MMA comes from one thread);
// softmax warps read S from TMEM, apply the permitted relation and fold each
// KV tile into the running summary (m, l, z) of "Context parallel attention:
// exchange keys and merge softmax globally" para 3: z is the PV accumulator
// in TMEM, m and l live in registers, one query row per thread.
//
// Each CTA owns two 128-row blocks A and B that read the same KV head: two
// query heads of one GQA group at the same query tile, or (one KV head per
// query head) two adjacent query tiles of one head.  For one causal sequence
// the GQA pair is folded instead: query tile t of one head with tile
// n_qtiles-1-t of the other, so every CTA has the same number of block-tiles;
// the block with fewer live KV tiles drops out of the ping-pong when its tiles
// end.  The blocks ping-pong on
// the tensor core so that each softmax warpgroup has the other block's MMAs
// to hide behind:
//
//   tensor core:  S_A(j) S_B(j) | PV_A(j) S_A(j+1) | PV_B(j) S_B(j+1) | ...
//   softmax A:           [ softmax A(j) ]            [ softmax A(j+1) ]
//   softmax B:                     [ softmax B(j) ]           ...
//
// TMEM (512 columns): S_A [0,128), S_B [128,256), O_A [256,384), O_B [384,512).
// P_X (bf16, two per column) is written back over the first 64 columns of
// S_X and read from there by the PV MMA (A operand in tensor memory).  MMAs
// from one thread execute in issue order, so S_X(j+1), issued after PV_X(j),
// never overwrites P_X(j) early, and its commit also certifies that PV_X(j)
// has finished before softmax X(j+1) touches O_X.
//
// Roles (384 threads): warp 0 TMA producer, warp 1 MMA issuer + TMEM owner,
// warps 4-7 softmax of block A, warps 8-11 softmax of block B (warp w reads
// TMEM lanes 32*(w%4) .. +31); warps 2-3 idle.
//
// Softmax per score: one FFMA (scale and subtract the row max, in exp2
// units) and one ex2.  The row max is refreshed lazily: O is rescaled only
// when it grows by more than 2^8.  l sums the fp32 weights; O = z / l and
// LSE = m + ln l.  The weights enter PV rounded to bf16 (relative error at
// most 2^-9 each), so O carries at most 2^-9 max|v| from that rounding.
//
// Masking ("... merge softmax globally" para 1-2, 5): a row's permitted keys
// are one interval of logical positions; KV tiles never straddle a chunk of
// the chunk map (chunk_len % 128 == 0), so the mask of a row in a tile is two
// column bounds.  Tiles outside every row's interval are skipped by all
// roles, so an all-masked chunk costs nothing and stays neutral.
//
// Per-KV-chunk summaries (kv_chunk_len > 0, a multiple of 128): the CHUNKS
// instantiation closes the running summary whenever the next KV tile belongs
// to another chunk of kv_chunk_len physical rows.  The softmax thread reads
// z_c from TMEM (the PV that finished it completed before the next S), writes
// the finalised (z_c / l_c, m_c + ln l_c) to partial_o / partial_lse, and
// starts the next chunk from (m, l) = (-inf, 0) while the MMA issuer
// overwrites O with that chunk's first PV.  Chunks a row never reaches are
// written neutral (0, -inf).  The row's o / lse are the merge of its own
// partials, read back at the end ("... merge softmax globally", para 3-4).
//
// Every wait is bounded (2 s).  On expiry the CTA raises an abort flag, all
// roles stop, in-flight TMA and MMA work is drained with bounded waits, TMEM
// is freed, and CPATTN_ERR_TIMEOUT is written to dev_status.
#include "dense_tc_common.cuh"

namespace cpattn {
namespace {

struct TcParams {
  cpattn_attn_args a;
  int n_qtiles;
  int n_ktiles;
  int head_pairs;   // 1: blocks are two heads of a GQA group; 0: two query tiles
  int fold;         // 1: head pairs at query tiles t and n_qtiles-1-t
  int n_units;      // CTAs
  int part_tiles;   // KV tiles per partial-summary chunk (CHUNKS)
  int n_parts;      // partial summaries per row (CHUNKS)
};

struct Smem {
  uint8_t q[2][kTileBytes];
  uint8_t k[NS][kTileBytes];
  uint8_t v[NS][kTileBytes];
  uint64_t q_full;
  uint64_t k_full[NS], k_empty[NS], v_full[NS], v_empty[NS];
  uint64_t s_full[2], p_full[2], o_ready[2];
  uint64_t drain, pv_done;
  uint32_t tmem_base;
  int abort;
  int n_blk[2];     // live-list entries block X runs (a prefix of the list)
  long long min_lo[2], max_hi[2];
  uint16_t live_kt[kMaxKTiles];
};

constexpr size_t kSmemBytes = sizeof(Smem) + 1024;  // + alignment slack

// Per softmax warp, a staging slice (store_rows32) for its rows' partial
// summaries, after the Smem block.
constexpr size_t kStageBytes = 8 * kStageSliceBytes;
constexpr size_t kStageOffset = (sizeof(Smem) + 15) / 16 * 16;   // from the 1024-aligned base
constexpr size_t kSmemBytesChunks = kStageOffset + kStageBytes + 1024;
static_assert(kSmemBytesChunks <= 232448, "shared memory budget");

// Finalised summary of one chunk for the warp's 32 rows (one per lane): z
// from the 128 O columns at o_col, scaled by 1/l, stored row-contiguously
// through the warp's staging slice.  Rows past Tq store nothing.  Called by
// all lanes of the warp together; ends with the rows written and visible to
// the whole warp.
__device__ __forceinline__ void write_partial(const cpattn_attn_args& a, int c, int64_t tok, int h,
                                              uint32_t o_col, float l, float m2, bool from_tmem,
                                              float (*stage)[kStageStride]) {
  const bool live = from_tmem && l > 0.f;
  const float inv = live ? 1.f / l : 0.f;
  const bool valid = tok < a.Tq;
  const int64_t row = ((int64_t)c * a.Tq + tok) * a.Hq + h;
  const StagedRows t = staged_rows(a.partial_o + row * HD, valid);
#pragma unroll 1
  for (int c4 = 0; c4 < HD / 32; ++c4) {
    uint32_t oo[32];
    if (from_tmem) {
      tmem_ld32_sync(o_col + c4 * 32, oo);
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) oo[i] = 0u;
    }
    store_rows32(stage, t, oo, inv, c4 * 32);
  }
  if (valid) a.partial_lse[row] = live ? (m2 + log2f(l)) * 0.6931471805599453f : -CUDART_INF_F;
  __syncwarp();   // orders the rows' stores before the lanes' own reads of them
}

template <bool CHUNKS>
__global__ void __launch_bounds__(kThreads, 1)
dense_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  Smem& s = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                     ~uintptr_t(1023));
  const cpattn_attn_args& a = p.a;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int u = blockIdx.x;
  // The two blocks as separate values (a runtime-indexed array would live in
  // local memory); the softmax warps select theirs once.
  const Block blk0 = p.fold ? folded_block_of(a.Hq, p.n_qtiles, u, 0)
                            : block_of(a.Hq, p.head_pairs, p.n_qtiles, u, 0);
  const Block blk1 = p.fold ? folded_block_of(a.Hq, p.n_qtiles, u, 1)
                            : block_of(a.Hq, p.head_pairs, p.n_qtiles, u, 1);
  const int g = blk0.head / (a.Hq / a.Hkv);
  volatile int* abort_flag = &s.abort;
  const uint64_t lim = wait_limit(a);

  if (threadIdx.x == 0) {
    mbar_init(&s.q_full, 1);
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
    }
    mbar_init(&s.drain, 1);
    mbar_init(&s.pv_done, 1);
    s.abort = 0;
    s.min_lo[0] = s.min_lo[1] = LLONG_MAX;
    s.max_hi[0] = s.max_hi[1] = LLONG_MIN;
    fence_mbar_init();
    // Q of both blocks needs no tile list: its load overlaps the list's
    // construction below (rows past Tq read the fill value).
    mbar_arrive_expect_tx(&s.q_full, 2 * kTileBytes);
    tma_load_3d(s.q[0], &tm_q, &s.q_full, 0, blk0.head, blk0.q0);
    tma_load_3d(s.q[0] + kHalf, &tm_q, &s.q_full, 64, blk0.head, blk0.q0);
    tma_load_3d(s.q[1], &tm_q, &s.q_full, 0, blk1.head, blk1.q0);
    tma_load_3d(s.q[1] + kHalf, &tm_q, &s.q_full, 64, blk1.head, blk1.q0);
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
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s.tmem_base;

  // Softmax threads: block X = (warp - 4) / 4, row r = lane of TMEM.
  const bool softmax_role = warp >= 4;
  const int X = softmax_role ? (warp - 4) >> 2 : 0;
  const int r = (warp & 3) * 32 + lane;
  const int my_head = X ? blk1.head : blk0.head, my_q0 = X ? blk1.q0 : blk0.q0;
  KeyInterval iv{1, 0};
  if (softmax_role) {
    const int64_t tok = (int64_t)my_q0 + r;
    if (tok < a.Tq) iv = allowed_interval(a, query_pos(a, tok));
    long long lo = iv.lo <= iv.hi ? (long long)iv.lo : LLONG_MAX;
    long long hi = iv.lo <= iv.hi ? (long long)iv.hi : LLONG_MIN;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      lo = min(lo, __shfl_xor_sync(kFullMask, lo, o));
      hi = max(hi, __shfl_xor_sync(kFullMask, hi, o));
    }
    if (lane == 0 && lo <= hi) {
      atomicMin(&s.min_lo[X], lo);
      atomicMax(&s.max_hi[X], hi);
    }
  }
  __syncthreads();
  const int64_t min_lo = min(s.min_lo[0], s.min_lo[1]), max_hi = max(s.max_hi[0], s.max_hi[1]);

  // Live KV tiles (those whose logical key range meets some row's interval),
  // listed once by warp 3 for every role.  Block X stops after n_blk[X]
  // entries when the tiles live for its own rows are a prefix of the list
  // (one causal sequence: every block starts at key 0); otherwise it runs the
  // whole list and its rows mask what they do not permit.
  if (warp == 3) {
    int base = 0;
    for (int kt0 = 0; kt0 < p.n_ktiles; kt0 += 32) {
      const int kt = kt0 + lane;
      bool live = false;
      if (kt < p.n_ktiles && min_lo <= max_hi) {
        const int64_t j0 = (int64_t)kt * BN;
        const int64_t kb = logical_pos(a.kv_chunk_map, a.chunk_len, j0);
        const int64_t kv = min((int64_t)BN, (int64_t)a.Tk - j0);
        live = kb <= max_hi && kb + kv - 1 >= min_lo;
      }
      const unsigned m = __ballot_sync(kFullMask, live);
      if (live) s.live_kt[base + __popc(m & ((1u << lane) - 1))] = (uint16_t)kt;
      base += __popc(m);
    }
    __syncwarp();
    for (int x = 0; x < 2; ++x) {
      const long long lo_x = s.min_lo[x], hi_x = s.max_hi[x];
      int cnt = 0, last = -1;
      for (int i0 = 0; i0 < base; i0 += 32) {
        const int i = i0 + lane;
        bool live = false;
        if (i < base && lo_x <= hi_x) {
          const int64_t j0 = (int64_t)s.live_kt[i] * BN;
          const int64_t kb = logical_pos(a.kv_chunk_map, a.chunk_len, j0);
          const int64_t kv = min((int64_t)BN, (int64_t)a.Tk - j0);
          live = kb <= hi_x && kb + kv - 1 >= lo_x;
        }
        const unsigned m = __ballot_sync(kFullMask, live);
        cnt += __popc(m);
        if (m) last = i0 + 31 - __clz(m);
      }
      if (lane == 0) s.n_blk[x] = (cnt == last + 1) ? cnt : base;
    }
  }
  __syncthreads();
  const int nx0 = s.n_blk[0], nx1 = s.n_blk[1];
  const int n_run = max(nx0, nx1);   // list entries loaded and multiplied
  // Tail: once the short block Sb has run its n_short tiles, the long block
  // Lb alternates its S between its own S columns and Sb's, so S(j+1) runs on
  // the tensor core while softmax(j) runs.  Tail tile n_short + u uses Lb's
  // columns for even u, Sb's for odd u; both barriers have then completed
  // n_short + u/2 phases before it.
  const int Sb = nx0 < nx1 ? 0 : 1, Lb = 1 - Sb;
  const int n_short = min(nx0, nx1);
  const bool tail2 = n_short >= 1 && n_run > n_short;

  if (warp < 4) {
  regs_dec<kRegsControl>();
  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int k_issued = 0, v_issued = 0;
      for (int i = 0; i < n_run; ++i) {
        const int kt = s.live_kt[i];
        const int jt = k_issued, st = jt % NS;
        const uint32_t ph = (jt / NS) & 1;
        if (!mbar_wait(&s.k_empty[st], ph ^ 1, abort_flag, lim)) break;
        mbar_arrive_expect_tx(&s.k_full[st], kTileBytes);
        tma_load_3d(s.k[st], &tm_k, &s.k_full[st], 0, g, kt * BN);
        tma_load_3d(s.k[st] + kHalf, &tm_k, &s.k_full[st], 64, g, kt * BN);
        ++k_issued;
        if (!mbar_wait(&s.v_empty[st], ph ^ 1, abort_flag, lim)) break;
        mbar_arrive_expect_tx(&s.v_full[st], kTileBytes);
        tma_load_3d(s.v[st], &tm_v, &s.v_full[st], 0, g, kt * BN);
        tma_load_3d(s.v[st] + kHalf, &tm_v, &s.v_full[st], 64, g, kt * BN);
        ++v_issued;
      }
      if (*abort_flag || n_run == 0) {  // let every copy in flight land before the CTA exits
        int no_abort = 0;
        mbar_wait(&s.q_full, 0, &no_abort, 200000000ull);
        for (int j = max(0, k_issued - NS); j < k_issued; ++j)
          mbar_wait(&s.k_full[j % NS], (j / NS) & 1, &no_abort, 200000000ull);
        for (int j = max(0, v_issued - NS); j < v_issued; ++j)
          mbar_wait(&s.v_full[j % NS], (j / NS) & 1, &no_abort, 200000000ull);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The warp issues both blocks' MMAs in the ping-pong order
    //   S_A(0) S_B(0) | PV_A(j) S_A(j+1) PV_B(j) S_B(j+1) | ...
    // from one elected lane (MMAs from one thread execute in issue order).
    // The whole warp runs the loop, converged, with every wait's outcome
    // made warp-uniform: a converged issuer loses fewer issue slots to the
    // softmax warps of its sub-partition than a single-lane branch.
    {
      auto wait_w = [&](uint64_t* bar, uint32_t ph) {
        return __all_sync(kFullMask, mbar_wait(bar, ph, abort_flag, lim));
      };
      const uint32_t idesc_qk = idesc_bf16_f32(BM, BN, 0, 0);   // Q, K both K-major
      const uint32_t idesc_pv = idesc_bf16_f32(BM, HD, 0, 1);   // P (TMEM), V MN-major
      // Descriptor low words: K-major Q and K step 32 B along K inside a
      // 64-column swizzled box and 16 KiB to the next box; V (MN-major,
      // leading offset 16 KiB to the next 64 value channels) steps 2 KiB per
      // 16 keys.
      const uint32_t q_lo0 = desc_lo(smem_u32(s.q[0]), 16), q_lo1 = desc_lo(smem_u32(s.q[1]), 16);
      const uint32_t k_lo0 = desc_lo(smem_u32(s.k[0]), 16), k_lo1 = desc_lo(smem_u32(s.k[1]), 16);
      const uint32_t v_lo0 = desc_lo(smem_u32(s.v[0]), kHalf), v_lo1 = desc_lo(smem_u32(s.v[1]), kHalf);
      const int n = n_run;
      // PV(j) overwrites O when tile j opens a partial-summary chunk
      auto opens_chunk = [&](int j) {
        if (j == 0) return true;
        if (!CHUNKS) return false;
        return s.live_kt[j] / p.part_tiles != s.live_kt[j - 1] / p.part_tiles;
      };
      auto issue_s = [&](int j, int x) {   // S_x(j) = Q_x K_j^T
        umma8_ss_kmajor<true>(tmem + kColS + x * BN, x ? q_lo1 : q_lo0, (j & 1) ? k_lo1 : k_lo0, idesc_qk);
        umma_commit<true>(&s.s_full[x]);
      };
      auto issue_pv = [&](int j, int x) {  // O_x += P_x(j) V_j
        const uint32_t d = tmem + kColO + x * HD, pa = tmem + kColS + x * BN;
        const uint32_t vb = (j & 1) ? v_lo1 : v_lo0;
        if (!opens_chunk(j)) umma8_ts_mnmajor<1, true>(d, pa, vb, idesc_pv);
        else umma8_ts_mnmajor<0, true>(d, pa, vb, idesc_pv);
      };
      bool ok = n > 0 && wait_w(&s.q_full, 0) && wait_w(&s.k_full[0], 0);
      if (ok) {
        tc_fence_after();
        for (int x = 0; x < 2; ++x)
          if ((x ? nx1 : nx0) > 0) issue_s(0, x);
        umma_commit<true>(&s.k_empty[0]);
      }
      // Step jt: for each block still running, PV_X(jt) then S_X(jt+1).  A
      // block past its last tile drops out; the V stage is released after the
      // step's last PV, the next K stage after the step's last S.
      const uint32_t q_lo_l = Lb ? q_lo1 : q_lo0;
      for (int jt = 0; jt < n && ok; ++jt) {
        const int st = jt & 1, st1 = (jt + 1) & 1;
        if (!wait_w(&s.v_full[st], (jt >> 1) & 1)) { ok = false; break; }
        if (tail2 && jt >= n_short) {
          // tail step: PV(jt) from the buffer holding P(jt), then S(jt+2) into it
          const int u = jt - n_short, xb = (u & 1) ? Sb : Lb;
          if (!wait_w(&s.p_full[xb], (n_short + (u >> 1)) & 1)) { ok = false; break; }
          tc_fence_after();
          if (CHUNKS && opens_chunk(jt))
            umma8_ts_mnmajor<0, true>(tmem + kColO + Lb * HD, tmem + kColS + xb * BN, st ? v_lo1 : v_lo0,
                                idesc_pv);
          else
            umma8_ts_mnmajor<1, true>(tmem + kColO + Lb * HD, tmem + kColS + xb * BN, st ? v_lo1 : v_lo0,
                                idesc_pv);
          umma_commit<true>(&s.v_empty[st]);
          umma_commit<true>(&s.pv_done);
          if (jt + 1 == n) umma_commit<true>(&s.o_ready[Lb]);
          if (jt + 2 < n) {
            if (!wait_w(&s.k_full[st], ((jt + 2) >> 1) & 1)) { ok = false; break; }
            tc_fence_after();
            umma8_ss_kmajor<true>(tmem + kColS + xb * BN, q_lo_l, st ? k_lo1 : k_lo0, idesc_qk);
            umma_commit<true>(&s.s_full[xb]);
            umma_commit<true>(&s.k_empty[st]);
          }
          continue;
        }
        bool k_ready = false;
        for (int x = 0; x < 2 && ok; ++x) {
          const int nxx = x ? nx1 : nx0;
          if (jt >= nxx) continue;
          if (!wait_w(&s.p_full[x], jt & 1)) { ok = false; break; }
          tc_fence_after();
          issue_pv(jt, x);
          if (x == 1 || jt >= nx1) umma_commit<true>(&s.v_empty[st]);
          if (jt + 1 == nxx) {
            umma_commit<true>(&s.o_ready[x]);
          } else {
            if (!k_ready) {
              if (!wait_w(&s.k_full[st1], ((jt + 1) >> 1) & 1)) { ok = false; break; }
              tc_fence_after();
              k_ready = true;
            }
            issue_s(jt + 1, x);
          }
        }
        if (ok && k_ready) umma_commit<true>(&s.k_empty[st1]);
        if (ok && tail2 && jt + 1 == n_short && n_short + 1 < n) {
          // first tail tile's successor: S(n_short+1) into Sb's columns, which
          // PV_Sb(n_short-1), issued before it, has finished reading
          if (!wait_w(&s.k_full[st], ((n_short + 1) >> 1) & 1)) { ok = false; break; }
          tc_fence_after();
          umma8_ss_kmajor<true>(tmem + kColS + Sb * BN, q_lo_l, st ? k_lo1 : k_lo0, idesc_qk);
          umma_commit<true>(&s.s_full[Sb]);
          umma_commit<true>(&s.k_empty[st]);
        }
      }
      // every MMA issued so far must finish before TMEM is released
      umma_commit<true>(&s.drain);
      int no_abort = 0;
      mbar_wait(&s.drain, 0, &no_abort, 1000000000ull);
    }
  }
  } else {
    regs_inc<kRegsSoftmax>();
    // ------------------------------------------------------------ softmax + epilogue
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t s_col = tmem + lane_base + kColS + X * BN;
    const uint32_t o_col = tmem + lane_base + kColO + X * HD;
    // CHUNKS: this warp's staging slice (softmax warps 4..11) after the Smem block
    float (*stage)[kStageStride] = reinterpret_cast<float (*)[kStageStride]>(
        reinterpret_cast<uint8_t*>(&s) + kStageOffset + (size_t)(warp - 4) * kStageSliceBytes);
    const float sl2 = a.scale * 1.4426950408889634f;   // scores in exp2 units
    float m2 = -CUDART_INF_F, l = 0.f;
    int jt = 0;
    bool ok = true;
    const int64_t tok_row = (int64_t)my_q0 + r;
    int cur_c = 0;                       // CHUNKS: the chunk being summarised
    const int my_n = X ? nx1 : nx0;
    for (int i = 0; i < my_n; ++i) {
      const int kt = s.live_kt[i];
      const int64_t kbase = logical_pos(a.kv_chunk_map, a.chunk_len, (int64_t)kt * BN);
      const int kvalid = min(BN, a.Tk - kt * BN);
      int lo_c = 1, hi_c = 0;   // permitted columns of this row in this tile
      if (iv.lo <= iv.hi) {
        lo_c = (int)max((int64_t)0, min((int64_t)BN, iv.lo - kbase));
        hi_c = (int)max((int64_t)-1, min((int64_t)kvalid - 1, iv.hi - kbase));
      }
      // S buffer of this tile and the phase its barriers are in
      int xb = X;
      uint32_t ph = jt & 1;
      const bool in_tail = tail2 && X == Lb && i >= n_short;
      if (in_tail) {
        const int u = i - n_short;
        xb = (u & 1) ? Sb : Lb;
        ph = (n_short + (u >> 1)) & 1;
      }
      const uint32_t sb_col = s_col + (uint32_t)((xb - X) * BN);
      ok = __all_sync(kFullMask, mbar_wait(&s.s_full[xb], ph, abort_flag, lim));
      if (!ok) break;
      tc_fence_after();
      if constexpr (CHUNKS) {
        const int c_tile = kt / p.part_tiles;
        if (c_tile != cur_c || jt == 0) {
          if (jt > 0) {
            // PV(jt-1) closed chunk cur_c; in the tail S(jt) follows only PV(jt-2)
            if (in_tail && i > n_short) {
              ok = __all_sync(kFullMask, mbar_wait(&s.pv_done, (i - n_short - 1) & 1, abort_flag, lim));
              if (!ok) break;
              tc_fence_after();
            }
            write_partial(a, cur_c, tok_row, my_head, o_col, l, m2, true, stage);
            ++cur_c;
          }
          for (; cur_c < c_tile; ++cur_c)
            write_partial(a, cur_c, tok_row, my_head, o_col, 0.f, 0.f, false, stage);
          m2 = -CUDART_INF_F;
          l = 0.f;
        }
      }
      float sv[BN];
      {
        uint32_t rr[BN];
        tmem_ld128_sync(sb_col, rr);
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
      for (int q = 0; q < 4; ++q) pm[q] = fmaxf(sv[2 * q], sv[2 * q + 1]);
#pragma unroll
      for (int c = 8; c < BN; c += 8) {
#pragma unroll
        for (int q = 0; q < 4; ++q) pm[q] = fmax3(pm[q], sv[c + 2 * q], sv[c + 2 * q + 1]);
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
        tmem_st32(sb_col + 32 * half, pk);
      }
      float a0, a1;
      f2_unpack(f2_add(rs2[0], rs2[1]), a0, a1);
      l = l * alpha + (a0 + a1);
      // PV_X(jt-1) has finished: S_X(jt) was issued after it and has landed.
      // In the tail S(jt) follows only PV(jt-2): wait for PV(jt-1), the
      // (jt - n_short)-th tail PV, unless jt is the first tail tile.
      if (__any_sync(kFullMask, rescale)) {
        if (in_tail && i > n_short) {
          ok = __all_sync(kFullMask, mbar_wait(&s.pv_done, (i - n_short - 1) & 1, abort_flag, lim));
          if (!ok) break;
          tc_fence_after();
        }
#pragma unroll
        for (int c4 = 0; c4 < HD / 32; ++c4) {
          uint32_t oo[32];
          tmem_ld32_sync(o_col + c4 * 32, oo);
#pragma unroll
          for (int q = 0; q < 32; ++q) oo[q] = __float_as_uint(__uint_as_float(oo[q]) * alpha);
          tmem_st32(o_col + c4 * 32, oo);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&s.p_full[xb]);
      ++jt;
    }
    if (ok && jt > 0) {
      ok = __all_sync(kFullMask, mbar_wait(&s.o_ready[X], 0, abort_flag, lim));
      if (ok) tc_fence_after();
    }
    const int64_t tok = tok_row;
    const int h = my_head;
    if constexpr (CHUNKS) {
      // close the last chunk, write the unreached ones neutral, then merge
      // this row's partials: L = max_c LSE_c, w_c = exp(LSE_c - L),
      // O = sum_c w_c O_c / sum_c w_c, LSE = L + ln sum_c w_c
      if (ok && jt > 0) {
        write_partial(a, cur_c, tok, h, o_col, l, m2, true, stage);
        ++cur_c;
      }
      for (; cur_c < p.n_parts; ++cur_c) write_partial(a, cur_c, tok, h, o_col, 0.f, 0.f, false, stage);
      if (tok < a.Tq && a.o != nullptr) {   // o == NULL: the partial summaries only
        const int64_t stride = (int64_t)a.Tq * a.Hq;
        const int64_t row0 = tok * a.Hq + h;
        float L = -CUDART_INF_F;
        for (int c = 0; c < p.n_parts; ++c) L = fmaxf(L, a.partial_lse[row0 + c * stride]);
        const bool any = L > -CUDART_INF_F;
        float wsum = 0.f;
        for (int c = 0; c < p.n_parts; ++c) {
          const float lc = a.partial_lse[row0 + c * stride];
          wsum += lc > -CUDART_INF_F ? exp2f((lc - L) * 1.4426950408889634f) : 0.f;
        }
        const float inv = any ? 1.f / wsum : 0.f;
        __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(a.o) + tok * a.o_stride_t + (int64_t)h * a.o_stride_h;
        for (int c4 = 0; c4 < HD / 32; ++c4) {
          float acc[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) acc[i] = 0.f;
          for (int c = 0; c < p.n_parts; ++c) {
            const float lc = a.partial_lse[row0 + c * stride];
            if (!(lc > -CUDART_INF_F)) continue;
            const float wc = exp2f((lc - L) * 1.4426950408889634f) * inv;
            const float4* src = reinterpret_cast<const float4*>(a.partial_o + (row0 + c * stride) * HD + c4 * 32);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float4 v4 = src[i];
              acc[4 * i] += wc * v4.x;
              acc[4 * i + 1] += wc * v4.y;
              acc[4 * i + 2] += wc * v4.z;
              acc[4 * i + 3] += wc * v4.w;
            }
          }
#pragma unroll
          for (int i = 0; i < 32; i += 8) {
            uint4 val;
            val.x = pack_bf16(acc[i + 0], acc[i + 1]);
            val.y = pack_bf16(acc[i + 2], acc[i + 3]);
            val.z = pack_bf16(acc[i + 4], acc[i + 5]);
            val.w = pack_bf16(acc[i + 6], acc[i + 7]);
            *reinterpret_cast<uint4*>(orow + c4 * 32 + i) = val;
          }
        }
        if (a.lse != nullptr) a.lse[row0] = any ? L + logf(wsum) : -CUDART_INF_F;
      }
    } else {
    // epilogue: O = z / l, LSE = m + ln l (natural log); no key -> (0, -inf)
    const bool live = ok && jt > 0 && l > 0.f;
    const float inv = live ? 1.f / l : 0.f;
    __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(a.o) + tok * a.o_stride_t + (int64_t)h * a.o_stride_h;
#pragma unroll
    for (int c4 = 0; c4 < HD / 32; ++c4) {
      uint32_t oo[32];
      if (ok && jt > 0) {
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
      a.lse[tok * a.Hq + h] = live ? (m2 + log2f(l)) * 0.6931471805599453f : -CUDART_INF_F;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
  if (threadIdx.x == 0 && s.abort) report_status(a.dev_status, CPATTN_ERR_TIMEOUT);
}

}  // namespace

bool dense_tc_supported(const cpattn_attn_args& a) {
  if (a.dtype != CPATTN_BF16 || a.Dqk != HD || a.Dv != HD) return false;
  if (a.Tq <= 0 || a.Tk <= 0) return false;
  if (a.kv_chunk_len != 0 && (a.kv_chunk_len % BN != 0 || a.partial_o == nullptr ||
                              a.partial_lse == nullptr))
    return false;
  if (!(a.scale > 0.f)) return false;   // the row max is taken on unscaled scores
  if ((a.q_chunk_map || a.kv_chunk_map) && a.chunk_len % BN != 0) return false;
  if ((a.Tk + BN - 1) / BN > kMaxKTiles) return false;
  // strides must be positive for the TMA descriptors
  if (a.q_stride_h <= 0 || a.k_stride_h <= 0 || a.v_stride_h <= 0) return false;
  return true;
}

cudaError_t launch_dense_tc(const cpattn_attn_args& a, cudaStream_t stream, bool* launched) {
  *launched = false;
  CUtensorMap tq, tk, tv;
  if (!make_map(&tq, a.q, a.Tq, a.Hq, a.q_stride_t, a.q_stride_h) ||
      !make_map(&tk, a.k, a.Tk, a.Hkv, a.k_stride_t, a.k_stride_h) ||
      !make_map(&tv, a.v, a.Tk, a.Hkv, a.v_stride_t, a.v_stride_h))
    return cudaSuccess;  // layout not expressible as a tensor map: caller falls back
  TcParams p;
  p.a = a;
  p.n_qtiles = (a.Tq + BM - 1) / BM;
  p.n_ktiles = (a.Tk + BN - 1) / BN;
  p.head_pairs = ((a.Hq / a.Hkv) % 2 == 0) ? 1 : 0;
  // One causal sequence without chunk maps: later query tiles see more keys,
  // so fold the tiles to give every unit the same number of block-tiles.
  p.fold = (p.head_pairs && a.causal && a.cu_seqlens == nullptr && a.q_chunk_map == nullptr &&
            a.kv_chunk_map == nullptr) ? 1 : 0;
  p.n_units = p.head_pairs ? p.n_qtiles * (a.Hq / 2) : ((p.n_qtiles + 1) / 2) * a.Hq;
  p.part_tiles = a.kv_chunk_len > 0 ? a.kv_chunk_len / BN : 1;
  p.n_parts = a.kv_chunk_len > 0 ? (a.Tk + a.kv_chunk_len - 1) / a.kv_chunk_len : 1;
  auto kern = a.kv_chunk_len > 0 ? dense_tc_kernel<true> : dense_tc_kernel<false>;
  const size_t smem = a.kv_chunk_len > 0 ? kSmemBytesChunks : kSmemBytes;
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(kern), (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)p.n_units, kThreads, smem, stream>>>(tq, tk, tv, p);
  *launched = true;
  return cudaGetLastError();
}

}  // namespace cpattn
