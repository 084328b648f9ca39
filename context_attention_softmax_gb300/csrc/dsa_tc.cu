// DSA top-k sparse attention on absorbed-MLA shapes, on the tensor cores.
//
// "[Feature-request] Context Parallel support for DSAttention" (allgather CP
// mode, step 6: iterate only over the top-k indices) and "[1/2] Enable DSA
// CP, THD with absorbed MLA - #3674" (sequence diagram: QK scores -> top-k ->
// sparse gather; Background: the key row is [latent 512 | rope 64], the
// value is the latent).  One query's 128 heads share every selected key row,
// so per query this is a dense 128 x 576 x k contraction followed by a
// 128 x k x 512 one.
//
// Capacity shapes the kernel: O of one query (128 x 512 fp32) fills all of
// tensor memory, and Q (128 x 576 bf16, 144 KiB) does not fit shared memory
// beside a key tile.  So:
//   * two CTAs per query, each owning half of the value channels (S is
//     computed by both);
//   * Q channels 0..255 are held in TMEM and used as the MMA's A operand,
//     channels 256..575 stay in shared memory (80 KiB);
//   * keys come in tiles of 64 gathered rows (72 KiB, two stages), fetched
//     with 16-byte cp.async straight into the 128-byte-swizzled layout; the
//     value rows are the first 512 channels of the same rows;
//   * the permitted relation (causal + packed bounds) is re-applied to every
//     index and kept as one flag per key slot of the tile; -1 and
//     out-of-range indices are masked (out-of-range also sets dev_status).
// TMEM: Q^T part [0,128), S double buffer [128,192) / [192,256), O half
// [256,512).  Work items (query, half) are taken in a fixed stride by
// persistent CTAs; all roles walk the same sequence.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"
#include "sm100.cuh"

namespace cpattn {
namespace {

using namespace sm100;

constexpr int HQ = 128;                  // heads = MMA rows
constexpr int DQK = 576, DVH = 256;      // key width, value channels per CTA
constexpr int BNK = 64;                  // keys per tile
constexpr int NS = 2;
constexpr int kThreads = 384;
constexpr int kPartThreads = 96;        // gather threads per stage part
constexpr int kChunks = DQK / 64;        // 9 channel chunks of a key row
constexpr int kQT = 4;                   // Q channel chunks in TMEM (0..255)
constexpr int kQS = kChunks - kQT;       // 5 chunks in shared memory
constexpr uint32_t kKChunkBytes = BNK * 128;             // 8 KiB
constexpr uint32_t kStageBytes = kChunks * kKChunkBytes; // 72 KiB
constexpr uint32_t kQChunkBytes = HQ * 128;              // 16 KiB
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColQ = 0, kColS = 128, kColO = 256;
constexpr float kRescaleThreshold = 8.f;

struct DsaParams {
  cpattn_attn_args a;
  const int32_t* idx;   // [Tq, topk], shared by all heads
  int topk;
  int n_tiles;
  int n_items;          // 2 * Tq
};

struct DSmem {
  uint8_t qs[kQS][kQChunkBytes];
  uint8_t kv[NS][kStageBytes];
  uint64_t qs_full, qs_empty, qt_full;
  uint64_t ka_full[NS], ka_empty[NS];   // key chunks this half's PV does not read
  uint64_t kb_full[NS], kb_empty[NS];   // the four value chunks of this half
  uint64_t s_full[2], p_full[2];
  uint64_t pv_done, o_full, o_free, drain;
  uint32_t tmem_base;
  int abort;
};
constexpr size_t kDSmemBytes = sizeof(DSmem) + 1024;
static_assert(kDSmemBytes <= 232448, "shared memory budget");

__device__ __forceinline__ void tmem_ld32_sync(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 t = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&t);
}

// Roles (384 threads): warp 9 Q loader (TMA, channels 256..575), warp 1 MMA
// issuer + TMEM owner, warps 0, 2, 3, 8, 10, 11 key-row gather, warps 4-7
// softmax, Q^T TMEM fill and epilogue (row = head).  Warp w runs on
// sub-partition w % 4: the MMA thread's (1) holds only a softmax warp and
// the light Q loader besides it.
__global__ void __launch_bounds__(kThreads, 1)
dsa_attn_kernel(const __grid_constant__ CUtensorMap tm_q, const DsaParams p) {
  extern __shared__ uint8_t smem_raw[];
  DSmem& s = *reinterpret_cast<DSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                       ~uintptr_t(1023));
  const cpattn_attn_args& a = p.a;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = &s.abort;
  const uint64_t lim = wait_limit(a);

  if (threadIdx.x == 0) {
    mbar_init(&s.qs_full, 1);
    mbar_init(&s.qs_empty, 1);
    mbar_init(&s.qt_full, 128);
    for (int i = 0; i < NS; ++i) {
      mbar_init(&s.ka_full[i], kPartThreads);
      mbar_init(&s.ka_empty[i], 1);
      mbar_init(&s.kb_full[i], kPartThreads);
      mbar_init(&s.kb_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.s_full[i], 1);
      mbar_init(&s.p_full[i], 128);
    }
    mbar_init(&s.pv_done, 1);
    mbar_init(&s.o_full, 1);
    mbar_init(&s.o_free, 128);
    mbar_init(&s.drain, 1);
    s.abort = 0;
    fence_mbar_init();
  }
  if (warp == 9 && lane == 0) tma_prefetch_desc(&tm_q);
  if (warp == 1) {
    tmem_alloc(&s.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s.tmem_base;
  const int T = p.n_tiles;

  if (warp == 9) {
    // ------------------------------------------------------------ Q channels 256..575
    if (lane == 0) {
      int ui = 0;
      bool ok = true;
      for (int it = blockIdx.x; it < p.n_items && ok; it += gridDim.x, ++ui) {
        const int i = it >> 1;
        if (!mbar_wait(&s.qs_empty, (ui & 1) ^ 1, abort_flag, lim)) { ok = false; break; }
        mbar_arrive_expect_tx(&s.qs_full, kQS * kQChunkBytes);
        for (int c = 0; c < kQS; ++c)
          tma_load_3d(s.qs[c], &tm_q, &s.qs_full, 64 * (kQT + c), 0, i);
      }
      if (!ok) {
        int no_abort = 0;
        mbar_wait(&s.qs_full, ui & 1, &no_abort, 200000000ull);
      }
    }
  } else if (warp == 0 || warp == 2 || warp == 3 || warp == 8 || warp == 10 || warp == 11) {
    // ------------------------------------------------------------ key-row gather
    // A stage is filled in two parts with their own barriers: part A (the
    // five 64-channel chunks that this half's PV does not read) is free again
    // as soon as S is done, part B (the four value chunks 4c..4c+3) only
    // after PV.  Warps 0, 2, 3 fetch part A and warps 8, 10, 11 part B, so
    // part A of the next tiles never queues behind a part B that waits for
    // PV; none of them shares a sub-partition with the MMA thread (warp 1),
    // whose issue slots the copies' address arithmetic would take.  A
    // warp takes key slots w, w + 3, ... and its lanes copy consecutive
    // 16-byte pieces of the row (whole 32-byte sectors).  The barriers are
    // arrived on by the copies themselves when they land.
    const bool part_a = warp <= 3;
    const int gw = (warp == 0 || warp == 8) ? 0 : (part_a ? warp - 1 : warp - 9);   // 0..2
    const __nv_bfloat16* kbase = reinterpret_cast<const __nv_bfloat16*>(a.k);
    uint64_t* empty = part_a ? s.ka_empty : s.kb_empty;
    uint64_t* full = part_a ? s.ka_full : s.kb_full;
    int gj = 0;
    bool ok = true;
    for (int it = blockIdx.x; it < p.n_items && ok; it += gridDim.x) {
      const int i = it >> 1, hc = it & 1;
      const KeyInterval iv = allowed_interval(a, query_pos(a, i));
      for (int j = 0; j < T; ++j, ++gj) {
        const int st = gj % NS;
        const uint32_t ph = ((gj / NS) & 1) ^ 1;
        const uint32_t stage = smem_u32(s.kv[st]);
        ok = __all_sync(kFullMask, mbar_wait(&empty[st], ph, abort_flag, lim));
        if (!ok) break;
        // The tile's 64 indices, two per lane; masked slots fetch row 0.
        int64_t e2[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int slot = BNK * j + 32 * h + lane;
          const int64_t e = slot < p.topk ? (int64_t)__ldg(p.idx + (int64_t)i * p.topk + slot) : -1;
          if (part_a && gw == 0 && (e < -1 || e >= a.Tk))
            report_status(a.dev_status, CPATTN_ERR_BAD_INDEX);
          e2[h] = (e >= 0 && e < a.Tk && e >= iv.lo && e <= iv.hi) ? e : 0;
        }
        if (part_a) {
          // 40 pieces per row
          for (int t = gw; t < BNK; t += 3) {
            const __nv_bfloat16* src =
                kbase + __shfl_sync(kFullMask, t < 32 ? e2[0] : e2[1], t & 31) * a.k_stride_t;
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              const int pc = lane + 32 * k;
              if (pc < 40) {
                const int q = pc >> 3;
                const int ch = hc == 0 ? 4 + q : (q < 4 ? q : 8);
                const uint32_t dst = stage + ch * kKChunkBytes + t * 128 + (((pc & 7) ^ (t & 7)) << 4);
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst),
                             "l"(src + 64 * ch + 8 * (pc & 7))
                             : "memory");
              }
            }
          }
        } else {
          // 32 pieces per row, one per lane
          const int ch = 4 * hc + (lane >> 3);
          for (int t = gw; t < BNK; t += 3) {
            const __nv_bfloat16* src =
                kbase + __shfl_sync(kFullMask, t < 32 ? e2[0] : e2[1], t & 31) * a.k_stride_t;
            const uint32_t dst = stage + ch * kKChunkBytes + t * 128 + (((lane & 7) ^ (t & 7)) << 4);
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst),
                         "l"(src + 64 * ch + 8 * (lane & 7))
                         : "memory");
          }
        }
        cp_async_mbar_arrive_noinc(&full[st]);
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the issue loop, converged, and one elected lane
    // issues each MMA group (waits made warp-uniform).
    {
      auto wait_w = [&](uint64_t* bar, uint32_t ph) {
        return __all_sync(kFullMask, mbar_wait(bar, ph, abort_flag, lim));
      };
      const uint32_t idesc_s = idesc_bf16_f32(HQ, BNK, 0, 0);    // A (TMEM or smem) K-major
      const uint32_t idesc_pv = idesc_bf16_f32(HQ, DVH, 0, 1);   // P (TMEM), V MN-major
      const uint32_t qs_lo = desc_lo(smem_u32(s.qs[0]), 16);
      int gj = 0, ui = 0;
      bool ok = true;
      int prev = -1, prev_first = 0, prev_last = 0, prev_ui = 0, prev_c = 0;
      auto issue_pv = [&]() -> bool {
        const int g = prev;
        if (!wait_w(&s.p_full[g & 1], (g >> 1) & 1)) return false;
        if (prev_first && prev_ui > 0 && !wait_w(&s.o_free, (prev_ui - 1) & 1))
          return false;
        tc_fence_after();
        // value channels [256c, 256c + 256) = chunks 4c..4c+3 of the key rows
        const uint32_t vb = desc_lo(smem_u32(s.kv[g % NS]) + 4 * prev_c * kKChunkBytes, kKChunkBytes);
        const uint32_t pa = tmem + kColS + (g & 1) * BNK;
        if (prev_first) umma4_ts_mn<0, true>(tmem + kColO, pa, vb, idesc_pv);
        else umma4_ts_mn<1, true>(tmem + kColO, pa, vb, idesc_pv);
        umma_commit<true>(&s.kb_empty[g % NS]);
        umma_commit<true>(&s.pv_done);
        if (prev_last) umma_commit<true>(&s.o_full);
        return true;
      };
      for (int it = blockIdx.x; it < p.n_items && ok; it += gridDim.x, ++ui) {
        const int hc = it & 1;
        // The previous item's last PV goes first: the softmax warps fill
        // this item's Q^T only after that item's last P.
        if (prev >= 0) {
          if (!issue_pv()) { ok = false; break; }
          prev = -1;
        }
        if (!wait_w(&s.qt_full, ui & 1) ||
            !wait_w(&s.qs_full, ui & 1)) { ok = false; break; }
        for (int j = 0; j < T; ++j, ++gj) {
          const int st = gj % NS;
          const uint32_t ph = (gj / NS) & 1;
          if (!wait_w(&s.ka_full[st], ph)) { ok = false; break; }
          fence_proxy_async_smem();   // the gathered rows were written by cp.async
          tc_fence_after();
          const uint32_t d = tmem + kColS + (gj & 1) * BNK;
          const uint32_t kb = desc_lo(smem_u32(s.kv[st]), 16);
          constexpr uint32_t kC = kKChunkBytes >> 4, kQC = kQChunkBytes >> 4;
          // Channels 0..255 take A = Q^T from TMEM (32 columns per 64
          // channels), channels 256..575 A = Q from shared memory.  Part A
          // chunks first, then the value chunks of this half.
          if (hc == 0) {
            umma4_ss_k<0, true>(d, qs_lo, kb + 4 * kC, idesc_s);
#pragma unroll
            for (int c = 1; c < kQS; ++c) umma4_ss_k<1, true>(d, qs_lo + c * kQC, kb + (kQT + c) * kC, idesc_s);
          } else {
            umma4_ts_k<0, true>(d, tmem + kColQ + 0, kb + 0 * kC, idesc_s);
            umma4_ts_k<1, true>(d, tmem + kColQ + 32, kb + 1 * kC, idesc_s);
            umma4_ts_k<1, true>(d, tmem + kColQ + 64, kb + 2 * kC, idesc_s);
            umma4_ts_k<1, true>(d, tmem + kColQ + 96, kb + 3 * kC, idesc_s);
            umma4_ss_k<1, true>(d, qs_lo + 4 * kQC, kb + 8 * kC, idesc_s);
          }
          umma_commit<true>(&s.ka_empty[st]);
          // PV of the previous tile goes between the two parts of S, so that
          // its value chunks are released as early as possible.
          if (prev >= 0 && !issue_pv()) { ok = false; break; }
          prev = -1;
          if (!wait_w(&s.kb_full[st], ph)) { ok = false; break; }
          fence_proxy_async_smem();
          tc_fence_after();
          if (hc == 0) {
            umma4_ts_k<1, true>(d, tmem + kColQ + 0, kb + 0 * kC, idesc_s);
            umma4_ts_k<1, true>(d, tmem + kColQ + 32, kb + 1 * kC, idesc_s);
            umma4_ts_k<1, true>(d, tmem + kColQ + 64, kb + 2 * kC, idesc_s);
            umma4_ts_k<1, true>(d, tmem + kColQ + 96, kb + 3 * kC, idesc_s);
          } else {
#pragma unroll
            for (int c = 0; c < 4; ++c) umma4_ss_k<1, true>(d, qs_lo + c * kQC, kb + (kQT + c) * kC, idesc_s);
          }
          umma_commit<true>(&s.s_full[gj & 1]);
          if (j == T - 1) umma_commit<true>(&s.qs_empty);
          prev = gj;
          prev_first = (j == 0);
          prev_last = (j == T - 1);
          prev_ui = ui;
          prev_c = it & 1;
        }
      }
      if (ok && prev >= 0) issue_pv();
      umma_commit<true>(&s.drain);
      int no_abort = 0;
      mbar_wait(&s.drain, 0, &no_abort, 1000000000ull);
    }
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------ softmax + epilogue
    const int r = (warp & 3) * 32 + lane;   // head
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const float sl2 = a.scale * 1.4426950408889634f;
    // Q channels 0..255 of (query, head r) into TMEM as bf16 pairs.  An
    // item's fill runs as soon as the previous item's last S is complete
    // (before that item's epilogue), so the MMA thread can start this
    // item's S while the epilogue drains O.
    auto fill_qt = [&](int item) {
      const uint4* qsrc = reinterpret_cast<const uint4*>(
          reinterpret_cast<const __nv_bfloat16*>(a.q) + (int64_t)(item >> 1) * a.q_stride_t +
          (int64_t)r * a.q_stride_h);
#pragma unroll
      for (int cc = 0; cc < kQT; ++cc) {
        uint32_t w[32];
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          const uint4 x = __ldg(qsrc + cc * 8 + v);
          w[4 * v] = x.x; w[4 * v + 1] = x.y; w[4 * v + 2] = x.z; w[4 * v + 3] = x.w;
        }
        tmem_st32(tmem + lane_base + kColQ + 32 * cc, w);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&s.qt_full);
    };
    int gj = 0, ui = 0;
    bool ok = true;
    if ((int)blockIdx.x < p.n_items) fill_qt(blockIdx.x);
    for (int it = blockIdx.x; it < p.n_items && ok; it += gridDim.x, ++ui) {
      const int i = it >> 1, c = it & 1;
      const KeyInterval iv = allowed_interval(a, query_pos(a, i));
      float m2 = -CUDART_INF_F, l = 0.f;
      {   // this head's channels 0..255 of the next item's query, into L2, so
          // the TMEM fill after the last tile reads L2
        const int nx = it + (int)gridDim.x;
        if (nx < p.n_items) {
          const char* nq = reinterpret_cast<const char*>(
              reinterpret_cast<const __nv_bfloat16*>(a.q) + (int64_t)(nx >> 1) * a.q_stride_t +
              (int64_t)r * a.q_stride_h);
#pragma unroll
          for (int k = 0; k < 4; ++k) asm volatile("prefetch.global.L2 [%0];" ::"l"(nq + 128 * k));
        }
      }
      for (int j = 0; j < T; ++j, ++gj) {
        // column mask of the tile: the index is present, in range and
        // permitted for this query (lane holds keys lane and lane + 32)
        uint32_t m0, m1;
        {
          const int slot = BNK * j + lane;
          const int64_t e0 = slot < p.topk ? (int64_t)__ldg(p.idx + (int64_t)i * p.topk + slot) : -1;
          const int64_t e1 =
              slot + 32 < p.topk ? (int64_t)__ldg(p.idx + (int64_t)i * p.topk + slot + 32) : -1;
          m0 = __ballot_sync(kFullMask, e0 >= 0 && e0 < a.Tk && e0 >= iv.lo && e0 <= iv.hi);
          m1 = __ballot_sync(kFullMask, e1 >= 0 && e1 < a.Tk && e1 >= iv.lo && e1 <= iv.hi);
        }
        ok = __all_sync(kFullMask, mbar_wait(&s.s_full[gj & 1], (gj >> 1) & 1, abort_flag, lim));
        if (!ok) break;
        tc_fence_after();
        const uint32_t s_col = tmem + lane_base + kColS + (gj & 1) * BNK;
        float sv[BNK];
        {
          uint32_t r0[32], r1[32];
          tmem_ld32_sync(s_col, r0);
          tmem_ld32_sync(s_col + 32, r1);
#pragma unroll
          for (int q = 0; q < 32; ++q) {
            sv[q] = ((m0 >> q) & 1u) ? __uint_as_float(r0[q]) : -CUDART_INF_F;
            sv[32 + q] = ((m1 >> q) & 1u) ? __uint_as_float(r1[q]) : -CUDART_INF_F;
          }
        }
        float pm[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) pm[q] = fmaxf(sv[2 * q], sv[2 * q + 1]);
#pragma unroll
        for (int q = 8; q < BNK; q += 8) {
#pragma unroll
          for (int x = 0; x < 4; ++x) pm[x] = fmax3(pm[x], sv[q + 2 * x], sv[q + 2 * x + 1]);
        }
        const float mx = fmax3(pm[0], pm[1], fmaxf(pm[2], pm[3])) * sl2;
        float alpha = 1.f;
        bool rescale = false;
        if (mx > m2) {
          if (m2 == -CUDART_INF_F) {
            m2 = mx;
          } else if (mx > m2 + kRescaleThreshold) {
            alpha = ex2_approx(m2 - mx);
            m2 = mx;
            rescale = true;
          }
        }
        const float mref = (m2 == -CUDART_INF_F) ? 0.f : m2;
        const uint64_t sl2x2 = f2_pack(sl2, sl2), nm2 = f2_pack(-mref, -mref);
        uint64_t rs2[2] = {0ull, 0ull};
        uint32_t pk[32];
#pragma unroll
        for (int q = 0; q < 32; ++q) {
          float x0, x1;
          f2_unpack(f2_fma(f2_pack(sv[2 * q], sv[2 * q + 1]), sl2x2, nm2), x0, x1);
          const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
          rs2[q & 1] = f2_add(rs2[q & 1], f2_pack(p0, p1));
          pk[q] = pack_bf16(p0, p1);
        }
        tmem_st32(s_col, pk);
        float a0, a1;
        f2_unpack(f2_add(rs2[0], rs2[1]), a0, a1);
        l = l * alpha + (a0 + a1);
        if (__any_sync(kFullMask, rescale)) {
          ok = __all_sync(kFullMask, mbar_wait(&s.pv_done, (gj - 1) & 1, abort_flag, lim));
          if (!ok) break;
          tc_fence_after();
#pragma unroll 1
          for (int c4 = 0; c4 < DVH / 32; ++c4) {
            uint32_t oo[32];
            const uint32_t addr = tmem + lane_base + kColO + c4 * 32;
            tmem_ld32_sync(addr, oo);
#pragma unroll
            for (int q = 0; q < 32; ++q) oo[q] = __float_as_uint(__uint_as_float(oo[q]) * alpha);
            tmem_st32(addr, oo);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&s.p_full[gj & 1]);
      }
      if (!ok) break;
      // Every S of this item is complete (s_full of its last tile was
      // observed), so Q^T may be overwritten with the next item's.
      if (it + (int)gridDim.x < p.n_items) fill_qt(it + (int)gridDim.x);
      ok = __all_sync(kFullMask, mbar_wait(&s.o_full, ui & 1, abort_flag, lim));
      if (!ok) break;
      tc_fence_after();
      // epilogue: O[i, r, 256c ...] = z / l; LSE = m + ln l (half 0 writes it)
      const bool live = l > 0.f;
      const float inv = live ? 1.f / l : 0.f;
      __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(a.o) + (int64_t)i * a.o_stride_t +
                            (int64_t)r * a.o_stride_h + DVH * c;
#pragma unroll 1
      for (int c4 = 0; c4 < DVH / 32; ++c4) {
        uint32_t oo[32];
        tmem_ld32_sync(tmem + lane_base + kColO + c4 * 32, oo);
#pragma unroll
        for (int q = 0; q < 32; q += 8) {
          uint4 val;
          val.x = pack_bf16(__uint_as_float(oo[q + 0]) * inv, __uint_as_float(oo[q + 1]) * inv);
          val.y = pack_bf16(__uint_as_float(oo[q + 2]) * inv, __uint_as_float(oo[q + 3]) * inv);
          val.z = pack_bf16(__uint_as_float(oo[q + 4]) * inv, __uint_as_float(oo[q + 5]) * inv);
          val.w = pack_bf16(__uint_as_float(oo[q + 6]) * inv, __uint_as_float(oo[q + 7]) * inv);
          *reinterpret_cast<uint4*>(orow + c4 * 32 + q) = val;
        }
      }
      if (c == 0 && a.lse != nullptr)
        a.lse[(int64_t)i * a.Hq + r] = live ? (m2 + log2f(l)) * 0.6931471805599453f : -CUDART_INF_F;
      tc_fence_before();
      mbar_arrive(&s.o_free);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
  if (threadIdx.x == 0 && s.abort) report_status(a.dev_status, CPATTN_ERR_TIMEOUT);
}

}  // namespace

bool dsa_tc_supported(const cpattn_attn_args& a, int32_t index_heads, int32_t block_size) {
  if (a.dtype != CPATTN_BF16 || a.Dqk != DQK || a.Dv != 2 * DVH) return false;
  if (a.Hq != HQ || a.Hkv != 1 || index_heads != 1 || block_size != 1) return false;
  if (a.kv_chunk_map != nullptr || !(a.scale > 0.f) || a.Tq <= 0 || a.Tk <= 0) return false;
  // values are the first 512 channels of the key rows (absorbed MLA)
  if (a.v != a.k || a.v_stride_t != a.k_stride_t) return false;
  if (a.q_stride_h <= 0 || a.q_stride_t <= 0) return false;
  return true;
}

cudaError_t launch_dsa_tc(const cpattn_attn_args& a, const int32_t* indices, int32_t topk,
                          cudaStream_t stream, bool* launched) {
  *launched = false;
  CUtensorMap tq;
  const uint64_t dims[3] = {(uint64_t)DQK, (uint64_t)HQ, (uint64_t)a.Tq};
  const uint64_t strides[2] = {(uint64_t)a.q_stride_h * 2, (uint64_t)a.q_stride_t * 2};
  const uint32_t box[3] = {64, (uint32_t)HQ, 1};
  if (!encode_bf16_3d(&tq, a.q, dims, strides, box)) return cudaSuccess;
  DsaParams p;
  p.a = a;
  p.idx = indices;
  p.topk = topk;
  p.n_tiles = (topk + BNK - 1) / BNK;
  p.n_items = 2 * a.Tq;
  const int n_sm = device_sm_count();
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(dsa_attn_kernel), (int)kDSmemBytes);
  if (e != cudaSuccess) return e;
  const int grid = p.n_items < n_sm ? p.n_items : n_sm;
  dsa_attn_kernel<<<grid, kThreads, kDSmemBytes, stream>>>(tq, p);
  *launched = true;
  return cudaGetLastError();
}

}  // namespace cpattn
