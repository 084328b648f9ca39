// The MLA projections around the CP-chunk attention, as one persistent
// tcgen05 GEMM kernel (bf16 x bf16 -> fp32 in tensor memory -> bf16):
//
//  * value up-projection after absorbed attention ("[1/2] Enable DSA CP, THD
//    with absorbed MLA - #3674", sequence diagram and Background):
//      out[t, h, :] = o_latent[t, h, :] @ up_v_weight[h]      (per head)
//    a batch of H GEMMs, M = tokens, N = V, K = L; up_v_weight[h] is [L, V]
//    with V contiguous, read as an MN-major B operand;
//  * local K/V materialisation from gathered latents ("[BC][MLA][CP] Optimize
//    MLA all-gather and Ulysses communication for Kimi K3 and dpskV3",
//    "K/V all-gather CP"):
//      kv = kv_c @ wkv_b^T, viewed [T, H, N + V];  k = [k_nope | k_shared],
//    one GEMM, M = tokens, N = H * (N + V), K = L; wkv_b is a linear layer's
//    weight [H * (N + V), L], read as a K-major B operand.  The epilogue sends
//    each 128-column tile to the key or the value of its head and appends
//    the head-shared key to every head's key row.
//
// The up-projection: tiles of 128 x 128 outputs, K in steps of 64 (one
// 128-byte swizzled box of bf16 per operand), six stages of 32 KiB.  The
// materialisation: tiles of 128 x 256, four stages of 48 KiB (see
// mla_kv_kernel).  Roles (256 threads): warp 0 TMA producer, warp 1 MMA
// issuer and TMEM owner (two accumulators, so the epilogue of one tile
// overlaps the main loop of the next), warps 4-7 epilogue (TMEM lane =
// output row).  Persistent CTAs take tiles in a fixed stride (up-projection:
// consecutive tiles share their head's weight) or in contiguous runs
// (materialisation: the CTAs running at one time share their A rows), so
// those reads come from L2.
//
// Every wait is bounded (wait_limit_ns, 2 s by default); on expiry the CTA
// drains its copies and MMAs in flight, frees TMEM and reports
// CPATTN_ERR_TIMEOUT in dev_status.
#include "common.cuh"
#include "internal.h"
#include "sm100.cuh"

namespace cpattn {
namespace {

using namespace sm100;

constexpr int GM = 128, GN = 128, GK = 64;
constexpr int kStages = 6;
constexpr int kGemmThreads = 256;
constexpr uint32_t kABytes = GM * GK * 2;   // 16 KiB
constexpr uint32_t kBBytes = GN * GK * 2;   // 16 KiB
constexpr uint32_t kBHalf = GK * 64 * 2;    // MN-major B: 64 K-rows x 64 N-columns, 8 KiB

struct GemmParams {
  int M;              // output rows (tokens)
  int m_tiles, n_tiles, batches, k_steps;
  int n_total_tiles;  // m_tiles * n_tiles * batches
  __nv_bfloat16* out; int64_t out_st, out_sh;       // up-projection [T, H, V]
  __nv_bfloat16* k_out; int64_t k_st, k_sh;         // materialised key [T, H, N + R]
  __nv_bfloat16* v_out; int64_t v_st, v_sh;         // materialised value [T, H, V]
  const __nv_bfloat16* k_shared; int64_t ks_st;     // [T, R]
  int N, V, R, H;
  int32_t* dev_status;
  uint64_t limit;
};

struct GemmSmem {
  uint8_t a[kStages][kABytes];
  uint8_t b[kStages][kBBytes];
  uint64_t full[kStages], empty[kStages];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};
constexpr size_t kGemmSmemBytes = sizeof(GemmSmem) + 1024;

__device__ __forceinline__ void tile_coords(const GemmParams& p, int tile, int& b, int& mt, int& nt) {
  const int per_b = p.m_tiles * p.n_tiles;
  b = tile / per_b;
  const int rem = tile - b * per_b;
  mt = rem / p.n_tiles;
  nt = rem - mt * p.n_tiles;
}

// One stage: four MMAs of K = 16 (W: issued by the converged warp).  A K-major (32 B per step); B K-major
// (32 B per step) or MN-major (16 K-rows = 2 KiB per step).
template <int B_MN, bool W = false>
__device__ __forceinline__ void mma_stage(uint32_t d, uint32_t a_lo, uint32_t b_lo, uint32_t idesc,
                                          bool acc_first) {
#pragma unroll
  for (int k = 0; k < 4; ++k)
    umma_ss_lo<W>(d, a_lo + 2 * k, b_lo + (B_MN ? 128 * k : 2 * k), idesc,
                  (k > 0 || acc_first) ? 1u : 0u);
}

__device__ __forceinline__ void tmem_ld32_wait(uint32_t taddr, uint32_t (&r)[32]) {
  tmem_ld32(taddr, r);
  tmem_wait_ld();
}

__device__ __forceinline__ uint32_t pack2_bf16(float lo, float hi) {
  __nv_bfloat162 t = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&t);
}

template <int B_MN>
__global__ void __launch_bounds__(kGemmThreads, 1)
mla_gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  GemmSmem& s = *reinterpret_cast<GemmSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = &s.abort;
  const uint64_t lim = p.limit;

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
      for (int tile = blockIdx.x; tile < p.n_total_tiles && ok; tile += gridDim.x) {
        int b, mt, nt;
        tile_coords(p, tile, b, mt, nt);
        for (int ks = 0; ks < p.k_steps; ++ks, ++it) {
          const int st = it % kStages;
          if (!mbar_wait(&s.empty[st], ((it / kStages) & 1) ^ 1, abort_flag, lim)) { ok = false; break; }
          mbar_arrive_expect_tx(&s.full[st], kABytes + kBBytes);
          tma_load_3d(s.a[st], &tm_a, &s.full[st], ks * GK, b, mt * GM);
          tma_load_3d(s.b[st], &tm_b, &s.full[st], nt * GN, ks * GK, b);
          tma_load_3d(s.b[st] + kBHalf, &tm_b, &s.full[st], nt * GN + 64, ks * GK, b);
        }
      }
      if (!ok || *abort_flag) {   // let the copies in flight land before the CTA exits
        // fill j was issued only after fill j - kStages had been consumed, so
        // at most the last kStages fills can still be in flight
        int no_abort = 0;
        for (int j = max(0, it - kStages); j < it; ++j)
          mbar_wait(&s.full[j % kStages], (j / kStages) & 1, &no_abort, 200000000ull);
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
      const uint32_t idesc = idesc_bf16_f32(GM, GN, 0, B_MN);
      int it = 0, ti = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < p.n_total_tiles && ok; tile += gridDim.x, ++ti) {
        const int buf = ti & 1;
        if (!wait_w(&s.acc_empty[buf], ((ti >> 1) & 1) ^ 1)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(buf * GN);
        for (int ks = 0; ks < p.k_steps; ++ks, ++it) {
          const int st = it % kStages;
          if (!wait_w(&s.full[st], (it / kStages) & 1)) { ok = false; break; }
          tc_fence_after();
          mma_stage<B_MN, true>(d, desc_lo(smem_u32(s.a[st]), 16),
                          desc_lo(smem_u32(s.b[st]), B_MN ? kBHalf : 16), idesc, ks > 0);
          umma_commit<true>(&s.empty[st]);
        }
        if (ok) umma_commit<true>(&s.acc_full[buf]);
      }
      umma_commit<true>(&s.drain);
      int no_abort = 0;
      mbar_wait(&s.drain, 0, &no_abort, 1000000000ull);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ epilogue
    const int r = (warp - 4) * 32 + lane;
    const uint32_t lane_base = (uint32_t)((warp - 4) * 32) << 16;
    int ti = 0;
    for (int tile = blockIdx.x; tile < p.n_total_tiles; tile += gridDim.x, ++ti) {
      const int buf = ti & 1;
      const bool ok = __all_sync(kFullMask, mbar_wait(&s.acc_full[buf], (ti >> 1) & 1, abort_flag, lim));
      if (!ok) break;
      tc_fence_after();
      int b, mt, nt;
      tile_coords(p, tile, b, mt, nt);
      const int64_t t = (int64_t)mt * GM + r;
      __nv_bfloat16* dst = p.out + t * p.out_st + (int64_t)b * p.out_sh + nt * GN;
#pragma unroll
      for (int c4 = 0; c4 < GN / 32; ++c4) {
        uint32_t acc[32];
        tmem_ld32_wait(tmem + lane_base + (uint32_t)(buf * GN + c4 * 32), acc);
        if (t < p.M) {
#pragma unroll
          for (int i = 0; i < 32; i += 8) {
            uint4 val;
            val.x = pack2_bf16(__uint_as_float(acc[i + 0]), __uint_as_float(acc[i + 1]));
            val.y = pack2_bf16(__uint_as_float(acc[i + 2]), __uint_as_float(acc[i + 3]));
            val.z = pack2_bf16(__uint_as_float(acc[i + 4]), __uint_as_float(acc[i + 5]));
            val.w = pack2_bf16(__uint_as_float(acc[i + 6]), __uint_as_float(acc[i + 7]));
            *reinterpret_cast<uint4*>(dst + c4 * 32 + i) = val;
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&s.acc_empty[buf]);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 256);
  if (threadIdx.x == 0 && s.abort) report_status(p.dev_status, CPATTN_ERR_TIMEOUT);
}

// ---------------------------------------------------------------- K/V materialisation
// 128 x 256 output tiles: per K step a stage holds the A box (128 tokens x 64
// latent channels, 16 KiB) and the B box (256 rows of wkv_b x 64, 32 KiB),
// four stages deep so that enough bytes are in flight to keep the operand
// stream from L2 going (a 128 x 512 A block kept resident left room for only
// three 32 KiB B stages and ran at ~20 B/clk per SM).  A 256-wide tile reads
// 384 KiB of operands for 33.5 MFLOP (87 FLOP/B, against 64 for 128 x 128
// tiles).  CTAs take contiguous runs of tiles in (row block, N tile) order,
// so the CTAs running at one time share their A rows in L2; wkv_b (33.5 MB)
// is loaded with an evict-last policy so that it stays in L2 against the
// K/V output stream, which is written evict-first.  The epilogue writes each
// 64-column box of a tile (and the shared rope key) into a swizzled staging
// buffer and stores it with one TMA store, instead of 16-byte stores of 128
// different rows per warp instruction.
constexpr int KN = 256;                       // N tile
constexpr int kKvStages = 4;
constexpr uint32_t kKvABox = GM * GK * 2;     // 16 KiB
constexpr uint32_t kKvBBox = KN * GK * 2;     // 32 KiB

struct KvSmem {
  uint8_t a[kKvStages][kKvABox];
  uint8_t b[kKvStages][kKvBBox];
  uint8_t out[2][GM * 128];      // two 128 x 64 bf16 output boxes (swizzled) for TMA stores
  uint64_t full[kKvStages], empty[kKvStages];
  uint64_t acc_full[2], acc_empty[2], drain;
  uint32_t tmem_base;
  int abort;
  int fills;                     // stage fills issued (for the drain on abort)
};
constexpr size_t kKvSmemBytes = sizeof(KvSmem) + 1024;
static_assert(kKvSmemBytes <= 232448, "shared memory budget");

__global__ void __launch_bounds__(kGemmThreads, 1)
mla_kv_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
              const __grid_constant__ CUtensorMap tm_ko, const __grid_constant__ CUtensorMap tm_vo,
              const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  KvSmem& s = *reinterpret_cast<KvSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                         ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort_flag = &s.abort;
  const uint64_t lim = p.limit;
  // this CTA's run of tiles (row block major, N tile minor)
  const int t0 = (int)((int64_t)blockIdx.x * p.n_total_tiles / gridDim.x);
  const int t1 = (int)((int64_t)(blockIdx.x + 1) * p.n_total_tiles / gridDim.x);

  if (threadIdx.x == 0) {
    for (int i = 0; i < kKvStages; ++i) {
      mbar_init(&s.full[i], 1);
      mbar_init(&s.empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&s.acc_full[i], 1);
      mbar_init(&s.acc_empty[i], 128);
    }
    mbar_init(&s.drain, 1);
    s.abort = 0;
    s.fills = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_a);
    tma_prefetch_desc(&tm_b);
  }
  if (warp == 1) {
    tmem_alloc(&s.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s.tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t keep = l2_policy_evict_last();
      int fills = 0;
      bool ok = true;
      for (int tile = t0; tile < t1 && ok; ++tile) {
        const int mt = tile / p.n_tiles, nt = tile - mt * p.n_tiles;
        for (int ks = 0; ks < p.k_steps; ++ks, ++fills) {
          const int st = fills % kKvStages;
          if (!mbar_wait(&s.empty[st], ((fills / kKvStages) & 1) ^ 1, abort_flag, lim)) { ok = false; break; }
          mbar_arrive_expect_tx(&s.full[st], kKvABox + kKvBBox);
          tma_load_3d(s.a[st], &tm_a, &s.full[st], ks * GK, 0, mt * GM);
          // every CTA streams all of wkv_b: keep it in L2 against the output stream
          tma_load_3d_hint(s.b[st], &tm_b, &s.full[st], ks * GK, nt * KN, 0, keep);
        }
      }
      s.fills = fills;
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the issue loop, converged, and one elected lane
    // issues each MMA group (waits made warp-uniform).
    {
      auto wait_w = [&](uint64_t* bar, uint32_t ph) {
        return __all_sync(kFullMask, mbar_wait(bar, ph, abort_flag, lim));
      };
      const uint32_t idesc = idesc_bf16_f32(GM, KN, 0, 0);
      int it = 0, ti = 0;
      bool ok = true;
      for (int tile = t0; tile < t1 && ok; ++tile, ++ti) {
        const int buf = ti & 1;
        if (!wait_w(&s.acc_empty[buf], ((ti >> 1) & 1) ^ 1)) { ok = false; break; }
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(buf * KN);
        for (int ks = 0; ks < p.k_steps; ++ks, ++it) {
          const int st = it % kKvStages;
          if (!wait_w(&s.full[st], (it / kKvStages) & 1)) { ok = false; break; }
          tc_fence_after();
          mma_stage<0, true>(d, desc_lo(smem_u32(s.a[st]), 16), desc_lo(smem_u32(s.b[st]), 16), idesc, ks > 0);
          umma_commit<true>(&s.empty[st]);
        }
        if (!ok) break;
        umma_commit<true>(&s.acc_full[buf]);
      }
      umma_commit<true>(&s.drain);
      int no_abort = 0;
      mbar_wait(&s.drain, 0, &no_abort, 1000000000ull);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ epilogue
    // Per 64-column box: wait until the store of the box before last has
    // read its buffer, fill the buffer (thread r = row r, its 128 bytes as
    // eight 16-byte pieces at r * 128 + ((c ^ (r % 8)) * 16), the 128-byte
    // swizzle the map describes), fence for the async proxy, and one thread
    // issues the TMA store.  Rows beyond the last token are not written.
    const int r = (warp - 4) * 32 + lane;
    const uint32_t lane_base = (uint32_t)((warp - 4) * 32) << 16;
    const bool issuer = threadIdx.x == 128;
    const int per_head = p.N + p.V;
    const uint64_t stream = l2_policy_evict_first();   // K/V are written once
    int ti = 0, bx = 0;
    auto box_begin = [&]() {
      if (issuer) bulk_wait_group_read<1>();   // the buffer's previous store has read it
      named_bar_sync(1, 128);
      return s.out[bx & 1];
    };
    auto box_end = [&](const CUtensorMap* map, int c0, int h, int t0) {
      fence_proxy_async_smem();
      named_bar_sync(1, 128);
      if (issuer) {
        tma_store_3d_hint(map, s.out[bx & 1], c0, h, t0, stream);
        bulk_commit_group();
      }
      ++bx;
    };
    for (int tile = t0; tile < t1; ++tile, ++ti) {
      const int buf = ti & 1;
      // all 128 threads leave together (they share named barriers below)
      const bool ok = named_bar_and(2, 128, mbar_wait(&s.acc_full[buf], (ti >> 1) & 1, abort_flag, lim));
      if (!ok) break;
      tc_fence_after();
      const int mt = tile / p.n_tiles, nt = tile - mt * p.n_tiles;
      const int64_t t = (int64_t)mt * GM + r;
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        const int col = nt * KN + half * GN;
        const int h = col / per_head;
        const int part = col - h * per_head;
        const bool present = h < p.H;                  // the padded last tile's second half is not
        const bool is_key = part < p.N;
#pragma unroll 1
        for (int x = 0; x < 2; ++x) {                 // two 64-column boxes of the half
          uint32_t acc[2][32];
          tmem_ld32(tmem + lane_base + (uint32_t)(buf * KN + half * GN + x * 64), acc[0]);
          tmem_ld32(tmem + lane_base + (uint32_t)(buf * KN + half * GN + x * 64 + 32), acc[1]);
          tmem_wait_ld();
          if (!present) continue;
          uint8_t* stage = box_begin();
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const uint32_t* a4 = acc[c >> 2] + 8 * (c & 3);
            uint4 val;
            val.x = pack2_bf16(__uint_as_float(a4[0]), __uint_as_float(a4[1]));
            val.y = pack2_bf16(__uint_as_float(a4[2]), __uint_as_float(a4[3]));
            val.z = pack2_bf16(__uint_as_float(a4[4]), __uint_as_float(a4[5]));
            val.w = pack2_bf16(__uint_as_float(a4[6]), __uint_as_float(a4[7]));
            *reinterpret_cast<uint4*>(stage + r * 128 + ((c ^ (r & 7)) << 4)) = val;
          }
          box_end(is_key ? &tm_ko : &tm_vo, (is_key ? part : part - p.N) + 64 * x, h, mt * GM);
        }
        if (present && is_key && part + GN == p.N) {
          // the head-shared key after this head's last key tile, 64 channels per box
          for (int c0 = 0; c0 < p.R; c0 += 64) {
            uint8_t* stage = box_begin();
            const bool row_ok = t < p.M;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              const int ch = c0 + 8 * c;
              uint4 val = make_uint4(0u, 0u, 0u, 0u);
              if (row_ok && ch < p.R) val = __ldg(reinterpret_cast<const uint4*>(p.k_shared + t * p.ks_st + ch));
              *reinterpret_cast<uint4*>(stage + r * 128 + ((c ^ (r & 7)) << 4)) = val;
            }
            box_end(&tm_ko, p.N + c0, h, mt * GM);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&s.acc_empty[buf]);
    }
    if (issuer) bulk_wait_group_all();   // every store complete before the buffers go away
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (s.abort && warp == 0 && lane == 0) {
    // every role has stopped: let the copies in flight land (at most the
    // last kKvStages fills; earlier ones were consumed)
    int no_abort = 0;
    for (int j = max(0, s.fills - kKvStages); j < s.fills; ++j)
      mbar_wait(&s.full[j % kKvStages], (j / kKvStages) & 1, &no_abort, 200000000ull);
  }
  if (warp == 1) tmem_dealloc(tmem, 512);
  if (threadIdx.x == 0 && s.abort) report_status(p.dev_status, CPATTN_ERR_TIMEOUT);
}

cudaError_t launch_v_up(const GemmParams& p, const CUtensorMap& ta, const CUtensorMap& tb,
                        cudaStream_t stream) {
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(mla_gemm_kernel<1>),
                                   (int)kGemmSmemBytes);
  if (e != cudaSuccess) return e;
  const int n_sm = device_sm_count();
  const int grid = p.n_total_tiles < n_sm ? p.n_total_tiles : n_sm;
  mla_gemm_kernel<1><<<grid, kGemmThreads, kGemmSmemBytes, stream>>>(ta, tb, p);
  return cudaGetLastError();
}

}  // namespace

cpattn_status mla_v_up_impl(const void* o_latent, int64_t o_st, int64_t o_sh,
                            const void* up_v_weight, int32_t T, int32_t H, int32_t L, int32_t V,
                            void* out, int64_t out_st, int64_t out_sh, int32_t* dev_status,
                            int64_t wait_limit_ns, cudaStream_t stream) {
  if (T == 0) return CPATTN_OK;
  CUtensorMap ta, tb;
  const uint64_t ad[3] = {(uint64_t)L, (uint64_t)H, (uint64_t)T};
  const uint64_t as[2] = {(uint64_t)o_sh * 2, (uint64_t)o_st * 2};
  const uint32_t ab[3] = {GK, 1, GM};
  const uint64_t bd[3] = {(uint64_t)V, (uint64_t)L, (uint64_t)H};
  const uint64_t bs[2] = {(uint64_t)V * 2, (uint64_t)L * V * 2};
  const uint32_t bb[3] = {64, GK, 1};
  if (!encode_bf16_3d(&ta, o_latent, ad, as, ab) || !encode_bf16_3d(&tb, up_v_weight, bd, bs, bb))
    return report_error(CPATTN_ERR_INVALID_ARG, "cpattn_mla_v_up: a TMA descriptor cannot describe the operands");
  GemmParams p{};
  p.M = T;
  p.m_tiles = (T + GM - 1) / GM;
  p.n_tiles = V / GN;
  p.batches = H;
  p.k_steps = L / GK;
  p.n_total_tiles = p.m_tiles * p.n_tiles * p.batches;
  p.out = static_cast<__nv_bfloat16*>(out);
  p.out_st = out_st;
  p.out_sh = out_sh;
  p.dev_status = dev_status;
  p.limit = wait_limit_ns > 0 ? (uint64_t)wait_limit_ns : 2000000000ull;
  const cudaError_t e = launch_v_up(p, ta, tb, stream);
  if (e != cudaSuccess) return report_error(CPATTN_ERR_CUDA, cudaGetErrorString(e));
  return CPATTN_OK;
}

cpattn_status mla_kv_impl(const void* kv_c, int64_t c_st, const void* k_shared, int64_t ks_st,
                          const void* wkv_b, int32_t T, int32_t L, int32_t H, int32_t N, int32_t R,
                          int32_t V, void* k_out, int64_t k_st, int64_t k_sh, void* v_out,
                          int64_t v_st, int64_t v_sh, int32_t* dev_status, int64_t wait_limit_ns,
                          cudaStream_t stream) {
  if (T == 0) return CPATTN_OK;
  CUtensorMap ta, tb;
  const int64_t n_rows = (int64_t)H * (N + V);
  const uint64_t ad[3] = {(uint64_t)L, 1, (uint64_t)T};
  const uint64_t as[2] = {(uint64_t)c_st * 2, (uint64_t)c_st * 2};
  const uint32_t ab[3] = {GK, 1, GM};
  const uint64_t bd[3] = {(uint64_t)L, (uint64_t)n_rows, 1};
  const uint64_t bs[2] = {(uint64_t)L * 2, (uint64_t)n_rows * L * 2};
  const uint32_t bb[3] = {GK, (uint32_t)KN, 1};
  if (!encode_bf16_3d(&ta, kv_c, ad, as, ab) || !encode_bf16_3d(&tb, wkv_b, bd, bs, bb))
    return report_error(CPATTN_ERR_INVALID_ARG,
                        "cpattn_mla_kv_materialise: a TMA descriptor cannot describe the operands");
  GemmParams p{};
  p.M = T;
  p.H = H;
  p.m_tiles = (T + GM - 1) / GM;
  p.n_tiles = (int)((n_rows + KN - 1) / KN);
  p.batches = 1;
  p.k_steps = L / GK;
  p.n_total_tiles = p.m_tiles * p.n_tiles;
  p.k_out = static_cast<__nv_bfloat16*>(k_out);
  p.k_st = k_st;
  p.k_sh = k_sh;
  p.v_out = static_cast<__nv_bfloat16*>(v_out);
  p.v_st = v_st;
  p.v_sh = v_sh;
  p.k_shared = static_cast<const __nv_bfloat16*>(k_shared);
  p.ks_st = ks_st;
  p.N = N;
  p.V = V;
  p.R = R;
  p.dev_status = dev_status;
  p.limit = wait_limit_ns > 0 ? (uint64_t)wait_limit_ns : 2000000000ull;
  CUtensorMap tko, tvo;
  const uint64_t kd[3] = {(uint64_t)(N + R), (uint64_t)H, (uint64_t)T};
  const uint64_t ks[2] = {(uint64_t)k_sh * 2, (uint64_t)k_st * 2};
  const uint64_t vd[3] = {(uint64_t)V, (uint64_t)H, (uint64_t)T};
  const uint64_t vs[2] = {(uint64_t)v_sh * 2, (uint64_t)v_st * 2};
  const uint32_t ob[3] = {64, 1, GM};
  if (!encode_bf16_3d(&tko, k_out, kd, ks, ob) || !encode_bf16_3d(&tvo, v_out, vd, vs, ob))
    return report_error(CPATTN_ERR_INVALID_ARG,
                        "cpattn_mla_kv_materialise: a TMA descriptor cannot describe the outputs");
  cudaError_t e = ensure_smem_attr(reinterpret_cast<const void*>(mla_kv_kernel), (int)kKvSmemBytes);
  if (e == cudaSuccess) {
    const int n_sm = device_sm_count();
    const int grid = p.n_total_tiles < n_sm ? p.n_total_tiles : n_sm;
    mla_kv_kernel<<<grid, kGemmThreads, kKvSmemBytes, stream>>>(ta, tb, tko, tvo, p);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) return report_error(CPATTN_ERR_CUDA, cudaGetErrorString(e));
  return CPATTN_OK;
}

}  // namespace cpattn
