// MoBA block-sparse attention on the tensor cores, grouped by key block.
//
// "Question on Implementing Context Parallelism with MoBA Efficient
// Attention": each (query, head) attends to the top-k gated KV blocks plus
// its own block.  Attending query by query would read every selected block
// once per (query, head); grouping by block reads each block's keys once per
// 128 selecting queries instead:
//
//   1. moba_count_head_kernel - count the selections of every (head, block)
//                            in shared-memory histograms (one head, 512
//                            queries per CTA); empty slots get LSE = -inf
//                            straight away.
//   2. moba_scan_kernel    - exclusive scan of the counts into list offsets
//                            and a list of work units: (head, block, first
//                            list entry, up to 128 entries).
//   3. moba_scatter_head_kernel - place every (query, slot) into its block's
//                            list (one reservation per bin and CTA).
//   4. moba_attn_kernel    - persistent tcgen05 kernel: per unit, gather the
//                            unit's 128 query rows, attend to the
//                            block's keys (128-key tiles, permitted relation
//                            re-applied so the own block is causal), and
//                            write the finalised summary (O_c, LSE_c) of
//                            that (query, head, slot).
//   5. the LSE merge (lse_merge.cu) folds the slots of every (query, head)
//      by rescaling to the larger max ("Context parallel attention: exchange
//      keys and merge softmax globally", para 3-4).
//
// Workspace (256-byte aligned regions): counts, cursors, offsets [H*NB(+1)],
// lists [Tq*H*S], units [max_units], n_units, partial O bf16 [S][Tq][H][128],
// partial LSE fp32 [S][Tq][H], with NB = ceil(Tk / B) and S = slots per row.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"
#include "sm100.cuh"

namespace cpattn {
namespace {

using namespace sm100;

constexpr int BM = 128, BN = 128, HD = 128;
constexpr int NS = 2;
constexpr int kThreads = 384;
// Register split at a launch budget of 168 x 384: control warps 64, softmax
// warps 216, epilogue warps 80.
constexpr uint32_t kRegsControl = 64, kRegsSoftmax = 216, kRegsEpilogue = 80;
static_assert(128 * (kRegsControl + kRegsSoftmax + kRegsEpilogue) <= 168 * kThreads, "register split");
constexpr uint32_t kTileBytes = BN * HD * 2;   // 32 KiB
constexpr uint32_t kHalf = 16384;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColO = 256;     // S double buffer at 0 / 128, O double buffer at 256 / 384
constexpr float kRescaleThreshold = 8.f;

struct MobaWs {
  int32_t* counts;
  int32_t* cursors;
  int32_t* offsets;
  int32_t* lists;
  int4* units;
  int32_t* n_units;
  __nv_bfloat16* part_o;   // finalised O of each (slot, query, head), bf16
  float* part_lse;
  int64_t max_units;
};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct Dims {
  int64_t Tq, H, S, NB, entries, max_units;
};
Dims moba_dims(const cpattn_attn_args& a, int32_t slots, int32_t block_size) {
  Dims d;
  d.Tq = a.Tq;
  d.H = a.Hq;
  d.S = slots;
  d.NB = (a.Tk + block_size - 1) / block_size;
  d.entries = d.Tq * d.H * d.S;
  d.max_units = d.entries / BM + d.H * d.NB + 1;
  return d;
}

MobaWs carve(void* ws, const Dims& d) {
  MobaWs w;
  char* p = reinterpret_cast<char*>(ws);
  const size_t nhb = (size_t)(d.H * d.NB + 1);
  w.counts = reinterpret_cast<int32_t*>(p);  p += align256(nhb * 4);
  w.cursors = reinterpret_cast<int32_t*>(p); p += align256(nhb * 4);
  w.offsets = reinterpret_cast<int32_t*>(p); p += align256(nhb * 4);
  w.lists = reinterpret_cast<int32_t*>(p);   p += align256((size_t)d.entries * 4);
  w.units = reinterpret_cast<int4*>(p);      p += align256((size_t)d.max_units * 16);
  w.n_units = reinterpret_cast<int32_t*>(p); p += 256;
  w.part_o = reinterpret_cast<__nv_bfloat16*>(p); p += align256((size_t)d.entries * HD * 2);
  w.part_lse = reinterpret_cast<float*>(p);  p += align256((size_t)d.entries * 4);
  w.max_units = d.max_units;
  return w;
}

size_t ws_bytes(const Dims& d) {
  const size_t nhb = (size_t)(d.H * d.NB + 1);
  return 3 * align256(nhb * 4) + align256((size_t)d.entries * 4) +
         align256((size_t)d.max_units * 16) + 256 + align256((size_t)d.entries * HD * 2) +
         align256((size_t)d.entries * 4);
}

// Selection entry of (query q, head h, slot s).
__device__ __forceinline__ int32_t sel_at(const int32_t* sel, int64_t q, int h, int s, int H,
                                          int index_heads, int S) {
  return __ldg(sel + ((q * index_heads + (index_heads == 1 ? 0 : h)) * S + s));
}

__global__ void moba_count_kernel(const int32_t* __restrict__ sel, int64_t Tq, int H, int S,
                                  int index_heads, int B, int Tk, int NB, int32_t* counts,
                                  float* part_lse, int32_t* dev_status) {
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= Tq * H * S) return;
  const int s = (int)(idx % S);
  const int64_t row = idx / S;
  const int h = (int)(row % H);
  const int64_t q = row / H;
  const int32_t b = sel_at(sel, q, h, s, H, index_heads, S);
  if (b == -1 || b < -1 || (int64_t)b * B >= Tk) {
    if (b != -1) report_status(dev_status, CPATTN_ERR_BAD_INDEX);
    part_lse[((int64_t)s * Tq + q) * H + h] = -CUDART_INF_F;
    return;
  }
  atomicAdd(counts + (int64_t)h * NB + b, 1);
}

// One CTA of 1024 threads: offsets = exclusive scan of counts; units: every
// list cut into chunks of up to 128 entries; cursors reset to 0.
__global__ void __launch_bounds__(1024) moba_scan_kernel(int n, int NB, const int32_t* counts,
                                                          int32_t* cursors, int32_t* offsets,
                                                          int4* units, int32_t* n_units) {
  __shared__ int warp_c[32], warp_u[32];
  __shared__ int carry_c, carry_u;
  const int t = threadIdx.x, lane = t & 31, wid = t >> 5;
  if (t == 0) { carry_c = 0; carry_u = 0; }
  __syncthreads();
  for (int base = 0; base < n; base += 1024) {
    const int i = base + t;
    const int c = i < n ? counts[i] : 0;
    const int u = (c + BM - 1) / BM;
    int ic = c, iu = u;   // inclusive warp scans
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int yc = __shfl_up_sync(kFullMask, ic, o), yu = __shfl_up_sync(kFullMask, iu, o);
      if (lane >= o) { ic += yc; iu += yu; }
    }
    if (lane == 31) { warp_c[wid] = ic; warp_u[wid] = iu; }
    __syncthreads();
    if (wid == 0) {
      int wc = warp_c[lane], wu = warp_u[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int yc = __shfl_up_sync(kFullMask, wc, o), yu = __shfl_up_sync(kFullMask, wu, o);
        if (lane >= o) { wc += yc; wu += yu; }
      }
      warp_c[lane] = wc;
      warp_u[lane] = wu;
    }
    __syncthreads();
    const int ec = carry_c + (wid ? warp_c[wid - 1] : 0) + ic - c;
    const int eu = carry_u + (wid ? warp_u[wid - 1] : 0) + iu - u;
    if (i < n) {
      offsets[i] = ec;
      cursors[i] = 0;
      for (int k = 0; k < u; ++k)
        units[eu + k] = make_int4(i / NB, i % NB, ec + k * BM, min(BM, c - k * BM));
    }
    __syncthreads();
    if (t == 1023) { carry_c += warp_c[31]; carry_u += warp_u[31]; }
    __syncthreads();
  }
  if (t == 0) {
    offsets[n] = carry_c;
    *n_units = carry_u;
  }
}

__global__ void moba_scatter_kernel(const int32_t* __restrict__ sel, int64_t Tq, int H, int S,
                                    int index_heads, int B, int Tk, int NB,
                                    const int32_t* offsets, int32_t* cursors, int32_t* lists) {
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= Tq * H * S) return;
  const int s = (int)(idx % S);
  const int64_t row = idx / S;
  const int h = (int)(row % H);
  const int64_t q = row / H;
  const int32_t b = sel_at(sel, q, h, s, H, index_heads, S);
  if (b < 0 || (int64_t)b * B >= Tk) return;
  const int64_t hb = (int64_t)h * NB + b;
  const int pos = atomicAdd(cursors + hb, 1);
  lists[offsets[hb] + pos] = (int32_t)(q * S + s);
}


// The same count and scatter with shared-memory histograms: a block takes
// one head and kCountQ queries, counts its (head, block) bins in shared
// memory and touches each global counter or cursor once per bin, instead of
// once per selection.  The list order inside a bin follows the blocks'
// reservations; each (query, slot) result does not depend on it.
constexpr int kCountQ = 512;
constexpr int kMaxSmemBins = 6144;   // 2 x 24 KiB of bins

__global__ void moba_count_head_kernel(const int32_t* __restrict__ sel, int64_t Tq, int H, int S,
                                       int index_heads, int B, int Tk, int NB, int32_t* counts,
                                       float* part_lse, int32_t* dev_status) {
  extern __shared__ int32_t hist[];
  const int h = blockIdx.y;
  for (int b = threadIdx.x; b < NB; b += blockDim.x) hist[b] = 0;
  __syncthreads();
  const int64_t q0 = (int64_t)blockIdx.x * kCountQ;
  const int n = (int)min((int64_t)kCountQ, Tq - q0) * S;
  for (int e = threadIdx.x; e < n; e += blockDim.x) {
    const int64_t q = q0 + e / S;
    const int s = e % S;
    const int32_t b = sel_at(sel, q, h, s, H, index_heads, S);
    if (b == -1 || b < -1 || (int64_t)b * B >= Tk) {
      if (b != -1) report_status(dev_status, CPATTN_ERR_BAD_INDEX);
      part_lse[((int64_t)s * Tq + q) * H + h] = -CUDART_INF_F;
      continue;
    }
    atomicAdd(&hist[b], 1);
  }
  __syncthreads();
  for (int b = threadIdx.x; b < NB; b += blockDim.x)
    if (hist[b] != 0) atomicAdd(counts + (int64_t)h * NB + b, hist[b]);
}

__global__ void moba_scatter_head_kernel(const int32_t* __restrict__ sel, int64_t Tq, int H, int S,
                                         int index_heads, int B, int Tk, int NB,
                                         const int32_t* offsets, int32_t* cursors, int32_t* lists) {
  extern __shared__ int32_t sm[];
  int32_t* hist = sm;        // [NB] this block's count, then its running rank
  int32_t* base = sm + NB;   // [NB] this block's reserved start in each list
  const int h = blockIdx.y;
  for (int b = threadIdx.x; b < NB; b += blockDim.x) hist[b] = 0;
  __syncthreads();
  const int64_t q0 = (int64_t)blockIdx.x * kCountQ;
  const int n = (int)min((int64_t)kCountQ, Tq - q0) * S;
  for (int e = threadIdx.x; e < n; e += blockDim.x) {
    const int32_t b = sel_at(sel, q0 + e / S, h, e % S, H, index_heads, S);
    if (b >= 0 && (int64_t)b * B < Tk) atomicAdd(&hist[b], 1);
  }
  __syncthreads();
  for (int b = threadIdx.x; b < NB; b += blockDim.x) {
    const int c = hist[b];
    base[b] = c != 0 ? offsets[(int64_t)h * NB + b] + atomicAdd(cursors + (int64_t)h * NB + b, c) : 0;
    hist[b] = 0;
  }
  __syncthreads();
  for (int e = threadIdx.x; e < n; e += blockDim.x) {
    const int64_t q = q0 + e / S;
    const int s = e % S;
    const int32_t b = sel_at(sel, q, h, s, H, index_heads, S);
    if (b < 0 || (int64_t)b * B >= Tk) continue;
    const int li = atomicAdd(&hist[b], 1);
    lists[base[b] + li] = (int32_t)(q * S + s);
  }
}

struct MobaParams {
  cpattn_attn_args a;
  int B;            // key block size (multiple of 128)
  int S;            // selection slots per (query, head)
  int NB;
  const int32_t* lists;
  const int4* units;
  const int32_t* n_units;
  __nv_bfloat16* part_o;
  float* part_lse;
};

struct MSmem {
  uint8_t q[2][kTileBytes];
  uint8_t k[NS][kTileBytes];
  uint8_t v[NS][kTileBytes];
  uint64_t q_full[2], q_empty[2];
  uint64_t k_full[NS], k_empty[NS], v_full[NS], v_empty[NS];
  uint64_t s_full[2], p_full[2];
  uint64_t pv_done, o_full[2], o_free[2], st_full[2], drain;
  float4 stats[2][BM];             // (m, l, -, -) of each row at the end of a unit
  uint32_t tmem_base;
  int abort;
};
constexpr size_t kMSmemBytes = sizeof(MSmem) + 1024;

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

// Tiles (of 128 keys) of block b: the block cut to the key range.
__device__ __forceinline__ int unit_tiles(const MobaParams& p, int b) {
  const int keys = min(p.B, p.a.Tk - b * p.B);
  return (keys + BN - 1) / BN;
}

// Roles (384 threads): warp 0 K/V TMA producer, warp 1 MMA issuer (the
// converged warp, one elected lane issuing) + TMEM owner, warps 2-3 gather
// the unit's query rows (cp.async), warps 4-7 softmax, warps 8-11 epilogue
// (row = TMEM lane).  Units are taken in a fixed stride (blockIdx.x,
// + gridDim.x, ...); all roles walk the same sequence, with a global tile
// counter jt across units.  S and O are double buffered in TMEM: S(jt+1)
// runs while softmax(jt) does, P(jt) goes over S(jt), and unit u
// accumulates in O buffer u & 1 while the epilogue warps drain unit u - 1.
__global__ void __launch_bounds__(kThreads, 1)
moba_attn_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                 const MobaParams p) {
  extern __shared__ uint8_t smem_raw[];
  MSmem& s = *reinterpret_cast<MSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                       ~uintptr_t(1023));
  const cpattn_attn_args& a = p.a;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = &s.abort;
  const uint64_t lim = wait_limit(a);
  const int n_units = *p.n_units;
  const int group = a.Hq / a.Hkv;

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.q_full[i], 64);
      mbar_init(&s.q_empty[i], 1);
      mbar_init(&s.s_full[i], 1);
      mbar_init(&s.p_full[i], 128);
    }
    for (int i = 0; i < NS; ++i) {
      mbar_init(&s.k_full[i], 1);
      mbar_init(&s.k_empty[i], 1);
      mbar_init(&s.v_full[i], 1);
      mbar_init(&s.v_empty[i], 1);
    }
    mbar_init(&s.pv_done, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.o_full[i], 1);
      mbar_init(&s.o_free[i], 128);
      mbar_init(&s.st_full[i], 128);
    }
    mbar_init(&s.drain, 1);
    s.abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
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

  if (warp < 4) {
  regs_dec<kRegsControl>();
  if (warp == 0) {
    // ------------------------------------------------------------ K/V producer
    if (lane == 0) {
      int jt = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
        const int4 un = p.units[u];
        const int g = un.x / group, T = unit_tiles(p, un.y);
        for (int t = 0; t < T; ++t, ++jt) {
          const int st = jt % NS;
          const uint32_t ph = (jt / NS) & 1;
          const int row0 = un.y * p.B + t * BN;
          if (!mbar_wait(&s.k_empty[st], ph ^ 1, abort_flag, lim)) { ok = false; break; }
          mbar_arrive_expect_tx(&s.k_full[st], kTileBytes);
          tma_load_3d(s.k[st], &tm_k, &s.k_full[st], 0, g, row0);
          tma_load_3d(s.k[st] + kHalf, &tm_k, &s.k_full[st], 64, g, row0);
          if (!mbar_wait(&s.v_empty[st], ph ^ 1, abort_flag, lim)) { ok = false; break; }
          mbar_arrive_expect_tx(&s.v_full[st], kTileBytes);
          tma_load_3d(s.v[st], &tm_v, &s.v_full[st], 0, g, row0);
          tma_load_3d(s.v[st] + kHalf, &tm_v, &s.v_full[st], 64, g, row0);
        }
      }
      if (!ok) {  // let copies in flight land
        int no_abort = 0;
        for (int j = max(0, jt - NS); j <= jt; ++j) {
          mbar_wait(&s.k_full[j % NS], (j / NS) & 1, &no_abort, 200000000ull);
          mbar_wait(&s.v_full[j % NS], (j / NS) & 1, &no_abort, 200000000ull);
        }
      }
    }
  } else if (warp == 2 || warp == 3) {
    // ------------------------------------------------------------ query-row gather
    // 64 threads, rows t and t + 64; each row's 16 chunks of 16 bytes go to
    // the 128-byte-swizzled K-major layout (chunk c of row r of a 64-column
    // box at r * 128 + ((c ^ (r % 8)) * 16)); cp.async, then a proxy fence
    // so the tensor core sees the rows.
    const int t = threadIdx.x - 64;
    int ui = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++ui) {
      const int4 un = p.units[u];
      const int qb = ui & 1;
      ok = __all_sync(kFullMask, mbar_wait(&s.q_empty[qb], ((ui >> 1) & 1) ^ 1, abort_flag, lim));
      if (!ok) break;
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int r = t + 64 * k;
        // rows past the unit's count repeat its first entry (masked later)
        const int32_t e = __ldg(p.lists + un.z + (r < un.w ? r : 0));
        const int64_t q = e / p.S;
        const __nv_bfloat16* src = reinterpret_cast<const __nv_bfloat16*>(a.q) + q * a.q_stride_t +
                                   (int64_t)un.x * a.q_stride_h;
        const uint32_t dst0 = smem_u32(s.q[qb]) + r * 128;
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const uint32_t dst = dst0 + (c >> 3) * kHalf + (((c & 7) ^ (r & 7)) << 4);
          asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src + 8 * c)
                       : "memory");
        }
      }
      asm volatile("cp.async.wait_all;" ::: "memory");
      fence_proxy_async_smem();
      mbar_arrive(&s.q_full[qb]);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
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
      int jt = 0, ui = 0;
      bool ok = true;
      // the previous tile, whose PV is still to be issued
      int prev = -1, prev_first = 0, prev_last = 0, prev_ui = 0;
      auto issue_pv = [&]() -> bool {
        const int j = prev;
        if (!wait_w(&s.p_full[j & 1], (j >> 1) & 1) ||
            !wait_w(&s.v_full[j % NS], (j / NS) & 1)) return false;
        // O of unit u lives in buffer u & 1; its first PV waits until the
        // epilogue has read unit u - 2 out of that buffer
        const int ob = prev_ui & 1;
        if (prev_first && prev_ui >= 2 &&
            !wait_w(&s.o_free[ob], ((prev_ui - 2) >> 1) & 1)) return false;
        tc_fence_after();
        const uint32_t vb = (j % NS) ? v_lo1 : v_lo0;
        const uint32_t pa = tmem + kColS + (j & 1) * BN;
        const uint32_t od = tmem + kColO + ob * HD;
        if (prev_first) umma8_ts_mnmajor<0, true>(od, pa, vb, idesc_pv);
        else umma8_ts_mnmajor<1, true>(od, pa, vb, idesc_pv);
        umma_commit<true>(&s.v_empty[j % NS]);
        umma_commit<true>(&s.pv_done);
        if (prev_last) umma_commit<true>(&s.o_full[ob]);
        return true;
      };
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++ui) {
        const int4 un = p.units[u];
        const int T = unit_tiles(p, un.y), qb = ui & 1;
        if (!wait_w(&s.q_full[qb], (ui >> 1) & 1)) { ok = false; break; }
        for (int t = 0; t < T; ++t, ++jt) {
          const int st = jt % NS;
          if (!wait_w(&s.k_full[st], (jt / NS) & 1)) { ok = false; break; }
          tc_fence_after();
          umma8_ss_kmajor<true>(tmem + kColS + (jt & 1) * BN, qb ? q_lo1 : q_lo0, st ? k_lo1 : k_lo0,
                          idesc_qk);
          umma_commit<true>(&s.s_full[jt & 1]);
          umma_commit<true>(&s.k_empty[st]);
          if (t == T - 1) umma_commit<true>(&s.q_empty[qb]);
          if (prev >= 0 && !issue_pv()) { ok = false; break; }
          prev = jt;
          prev_first = (t == 0);
          prev_last = (t == T - 1);
          prev_ui = ui;
        }
      }
      if (ok && prev >= 0) issue_pv();
      umma_commit<true>(&s.drain);
      int no_abort = 0;
      mbar_wait(&s.drain, 0, &no_abort, 1000000000ull);
    }
  }
  } else if (warp < 8) {
    regs_inc<kRegsSoftmax>();
    // ------------------------------------------------------------ softmax
    const int r = (warp & 3) * 32 + lane;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const float sl2 = a.scale * 1.4426950408889634f;
    int jt = 0, ui = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++ui) {
      const int4 un = p.units[u];
      const int T = unit_tiles(p, un.y);
      const bool row_live = r < un.w;
      int64_t q = 0;
      KeyInterval iv{1, 0};
      if (row_live) {
        const int32_t e = __ldg(p.lists + un.z + r);
        q = e / p.S;
        iv = allowed_interval(a, query_pos(a, q));
      }
      float m2 = -CUDART_INF_F, l = 0.f;
      for (int t = 0; t < T; ++t, ++jt) {
        const int64_t kbase = (int64_t)un.y * p.B + t * BN;
        const int kvalid = min(BN, a.Tk - (int)kbase);
        int lo_c = 1, hi_c = 0;
        if (iv.lo <= iv.hi) {
          lo_c = (int)max((int64_t)0, min((int64_t)BN, iv.lo - kbase));
          hi_c = (int)max((int64_t)-1, min((int64_t)kvalid - 1, iv.hi - kbase));
        }
        ok = __all_sync(kFullMask, mbar_wait(&s.s_full[jt & 1], (jt >> 1) & 1, abort_flag, lim));
        if (!ok) break;
        tc_fence_after();
        const uint32_t s_col = tmem + lane_base + kColS + (jt & 1) * BN;
        float sv[BN];
        {   // the row's 128 scores in four loads and one wait
          uint32_t rr[BN];
#pragma unroll
          for (int c4 = 0; c4 < BN / 32; ++c4)
            tmem_ld32(s_col + c4 * 32, *reinterpret_cast<uint32_t(*)[32]>(rr + 32 * c4));
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < BN; ++i) sv[i] = __uint_as_float(rr[i]);
        }
        if (!(lo_c == 0 && hi_c == BN - 1)) {
#pragma unroll
          for (int c = 0; c < BN; ++c)
            if (c < lo_c || c > hi_c) sv[c] = -CUDART_INF_F;
        }
        float pm[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) pm[i] = fmaxf(sv[2 * i], sv[2 * i + 1]);
#pragma unroll
        for (int c = 8; c < BN; c += 8) {
#pragma unroll
          for (int i = 0; i < 4; ++i) pm[i] = fmax3(pm[i], sv[c + 2 * i], sv[c + 2 * i + 1]);
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
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t pk[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const int e2 = 64 * half + 2 * c;
            float x0, x1;
            f2_unpack(f2_fma(f2_pack(sv[e2], sv[e2 + 1]), sl2x2, nm2), x0, x1);
            const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
            rs2[c & 1] = f2_add(rs2[c & 1], f2_pack(p0, p1));
            pk[c] = pack_bf16(p0, p1);
          }
          tmem_st32(s_col + 32 * half, pk);
        }
        float a0, a1;
        f2_unpack(f2_add(rs2[0], rs2[1]), a0, a1);
        l = l * alpha + (a0 + a1);
        if (__any_sync(kFullMask, rescale)) {
          // O holds PV of this unit's earlier tiles: wait for the last one
          ok = __all_sync(kFullMask, mbar_wait(&s.pv_done, (jt - 1) & 1, abort_flag, lim));
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int c4 = 0; c4 < HD / 32; ++c4) {
            uint32_t oo[32];
            const uint32_t addr = tmem + lane_base + kColO + (ui & 1) * HD + c4 * 32;
            tmem_ld32_sync(addr, oo);
#pragma unroll
            for (int i = 0; i < 32; ++i) oo[i] = __float_as_uint(__uint_as_float(oo[i]) * alpha);
            tmem_st32(addr, oo);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&s.p_full[jt & 1]);
      }
      if (!ok) break;
      // the row's running summary to the epilogue warps
      s.stats[ui & 1][r] = make_float4(m2, l, 0.f, 0.f);
      mbar_arrive(&s.st_full[ui & 1]);
    }
  } else {
    regs_dec<kRegsEpilogue>();
    // ------------------------------------------------------------ epilogue
    // Finalised summary (O_c, LSE_c) of each (query, head, slot) of a unit,
    // from O in TMEM buffer ui & 1 and the row's (m, l); the softmax
    // warps meanwhile run the next unit.
    const int r = (warp & 3) * 32 + lane;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    // the slot summaries are read once, by the merge: let them leave L2
    // first, before the K/V tiles that a neighbouring unit may still read
    const uint64_t stream = l2_policy_evict_first();
    int ui = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++ui) {
      const int4 un = p.units[u];
      const int ob = ui & 1;
      ok = __all_sync(kFullMask, mbar_wait(&s.o_full[ob], (ui >> 1) & 1, abort_flag, lim) &&
                                     mbar_wait(&s.st_full[ob], (ui >> 1) & 1, abort_flag, lim));
      if (!ok) break;
      tc_fence_after();
      const float4 st = s.stats[ob][r];
      const bool row_live = r < un.w;
      int64_t q = 0;
      int slot = 0;
      if (row_live) {
        const int32_t e = __ldg(p.lists + un.z + r);
        q = e / p.S;
        slot = e - (int)q * p.S;
      }
      const bool live = row_live && st.y > 0.f;
      const float inv = live ? 1.f / st.y : 0.f;
      const int64_t prow = ((int64_t)slot * a.Tq + q) * a.Hq + un.x;
      __nv_bfloat16* orow = p.part_o + prow * HD;
#pragma unroll
      for (int c4 = 0; c4 < HD / 32; ++c4) {
        uint32_t oo[32];
        tmem_ld32_sync(tmem + lane_base + kColO + ob * HD + c4 * 32, oo);
        if (row_live) {
#pragma unroll
          for (int i = 0; i < 32; i += 8) {
            uint4 val;
            val.x = pack_bf16(__uint_as_float(oo[i + 0]) * inv, __uint_as_float(oo[i + 1]) * inv);
            val.y = pack_bf16(__uint_as_float(oo[i + 2]) * inv, __uint_as_float(oo[i + 3]) * inv);
            val.z = pack_bf16(__uint_as_float(oo[i + 4]) * inv, __uint_as_float(oo[i + 5]) * inv);
            val.w = pack_bf16(__uint_as_float(oo[i + 6]) * inv, __uint_as_float(oo[i + 7]) * inv);
            st_global_v4_hint(orow + c4 * 32 + i, val, stream);
          }
        }
      }
      if (row_live) p.part_lse[prow] = live ? (st.x + log2f(st.y)) * 0.6931471805599453f : -CUDART_INF_F;
      tc_fence_before();
      mbar_arrive(&s.o_free[ob]);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
  if (threadIdx.x == 0 && s.abort) report_status(a.dev_status, CPATTN_ERR_TIMEOUT);
}

// [rows, heads, 128] bf16 with element strides; box = 64 x 1 x box_rows.
bool make_map(CUtensorMap* m, const void* base, int64_t rows, int heads, int64_t st_t,
              int64_t st_h, int box_rows) {
  const uint64_t dims[3] = {(uint64_t)HD, (uint64_t)heads, (uint64_t)rows};
  const uint64_t strides[2] = {(uint64_t)st_h * 2, (uint64_t)st_t * 2};
  const uint32_t box[3] = {64, 1, (uint32_t)box_rows};
  return encode_bf16_3d(m, base, dims, strides, box);
}

}  // namespace

bool moba_tc_supported(const cpattn_attn_args& a, int32_t index_heads, int32_t block_size,
                       int32_t slots) {
  if (a.dtype != CPATTN_BF16 || a.Dqk != HD || a.Dv != HD) return false;
  if (block_size % BN != 0 || a.kv_chunk_map != nullptr) return false;
  if (!(a.scale > 0.f) || a.Tq <= 0 || a.Tk <= 0 || slots <= 0) return false;
  if (a.q_stride_h <= 0 || a.k_stride_h <= 0 || a.v_stride_h <= 0) return false;
  if ((int64_t)a.Tq * slots >= (int64_t)1 << 31) return false;
  if ((int64_t)a.Tq * a.Hq * slots >= (int64_t)1 << 31) return false;
  (void)index_heads;
  return true;
}

size_t moba_tc_workspace(const cpattn_attn_args& a, int32_t slots, int32_t block_size) {
  return ws_bytes(moba_dims(a, slots, block_size)) + 256;
}

cudaError_t launch_moba_tc(const cpattn_attn_args& a, const int32_t* sel, int32_t slots,
                           int32_t index_heads, int32_t block_size, void* workspace,
                           cudaStream_t stream) {
  const Dims d = moba_dims(a, slots, block_size);
  void* ws = reinterpret_cast<void*>((reinterpret_cast<uintptr_t>(workspace) + 255) & ~uintptr_t(255));
  const MobaWs w = carve(ws, d);
  const int nhb = (int)(d.H * d.NB);
  cudaError_t e = cudaMemsetAsync(w.counts, 0, (size_t)(nhb + 1) * 4, stream);
  if (e != cudaSuccess) return e;
  const int64_t n = d.entries;
  const unsigned blocks = (unsigned)((n + 255) / 256);
  const bool smem_bins = d.NB <= kMaxSmemBins && d.H <= 65535;
  const dim3 hgrid((unsigned)((d.Tq + kCountQ - 1) / kCountQ), (unsigned)d.H);
  if (smem_bins)
    moba_count_head_kernel<<<hgrid, 256, (size_t)d.NB * 4, stream>>>(
        sel, d.Tq, (int)d.H, slots, index_heads, block_size, a.Tk, (int)d.NB, w.counts, w.part_lse,
        a.dev_status);
  else
    moba_count_kernel<<<blocks, 256, 0, stream>>>(sel, d.Tq, (int)d.H, slots, index_heads,
                                                  block_size, a.Tk, (int)d.NB, w.counts, w.part_lse,
                                                  a.dev_status);
  moba_scan_kernel<<<1, 1024, 0, stream>>>(nhb, (int)d.NB, w.counts, w.cursors, w.offsets, w.units,
                                           w.n_units);
  if (smem_bins)
    moba_scatter_head_kernel<<<hgrid, 256, (size_t)d.NB * 8, stream>>>(
        sel, d.Tq, (int)d.H, slots, index_heads, block_size, a.Tk, (int)d.NB, w.offsets, w.cursors,
        w.lists);
  else
    moba_scatter_kernel<<<blocks, 256, 0, stream>>>(sel, d.Tq, (int)d.H, slots, index_heads,
                                                    block_size, a.Tk, (int)d.NB, w.offsets,
                                                    w.cursors, w.lists);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  CUtensorMap tk, tv;
  if (!make_map(&tk, a.k, a.Tk, a.Hkv, a.k_stride_t, a.k_stride_h, BN) ||
      !make_map(&tv, a.v, a.Tk, a.Hkv, a.v_stride_t, a.v_stride_h, BN))
    return cudaErrorInvalidValue;
  MobaParams p;
  p.a = a;
  p.B = block_size;
  p.S = slots;
  p.NB = (int)d.NB;
  p.lists = w.lists;
  p.units = w.units;
  p.n_units = w.n_units;
  p.part_o = w.part_o;
  p.part_lse = w.part_lse;
  const int n_sm = device_sm_count();
  e = ensure_smem_attr(reinterpret_cast<const void*>(moba_attn_kernel), (int)kMSmemBytes);
  if (e != cudaSuccess) return e;
  const int grid = (int)(d.max_units < (int64_t)n_sm ? d.max_units : (int64_t)n_sm);
  moba_attn_kernel<<<grid, kThreads, kMSmemBytes, stream>>>(tk, tv, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_lse_merge_bf16parts(slots, w.part_o, w.part_lse, a.Tq, a.Hq, HD, a.o, CPATTN_BF16,
                                    a.o_stride_t, a.o_stride_h, a.lse, stream);
}

}  // namespace cpattn
