// Dense CP-chunk attention on the 5th-generation tensor cores (sm_103a):
// TMA loads Q/K/V tiles into 128-byte-swizzled shared memory, one thread
// issues tcgen05.mma (bf16 x bf16 -> fp32 in tensor memory), four softmax
// warps read S from TMEM, apply the permitted relation, and fold each KV
// tile into the running summary (m, l, z) of "Context parallel attention:
// exchange keys and merge softmax globally" para 3 - z lives in TMEM as the
// PV accumulator, m and l in registers, one query row per thread.
//
// Tile: 128 queries (one head) x 128 keys x d 128.  Roles per CTA (192
// threads): warp 0 TMA producer, warp 1 MMA issuer (and TMEM owner), warps
// 2-5 softmax + epilogue (warp w reads TMEM lanes 32*(w%4) .. +31).
//
// Per KV tile j:  S_j = Q K_j^T (TMEM buffer j%2) -> softmax_j writes P_j
// (bf16) to shared memory -> O += P_j V_j.  S_{j+1} runs on the tensor core
// while softmax_j runs.  The running max is refreshed lazily: O is rescaled
// only when a row's max grows by more than 2^8 (in exp2 units), otherwise
// the stale max is kept (values stay <= 256, exact in the final division).
//
// Masking ("... merge softmax globally" para 1-2, para 5): a row's permitted
// keys are one interval of logical positions; KV tiles never straddle a
// chunk of the chunk map (chunk_len % 128 == 0), so a tile's keys are
// contiguous logical positions and the mask of a row is two column bounds.
// Tiles outside every row's interval are skipped by all roles alike, so an
// all-masked chunk costs nothing and leaves the neutral summary.
//
// Every wait is bounded (2 s).  On expiry the CTA raises an abort flag, all
// roles stop, in-flight TMA and MMA work is drained with bounded waits, TMEM
// is freed, and CPATTN_ERR_TIMEOUT is written to dev_status.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <climits>

#include "common.cuh"
#include "internal.h"
#include "sm100.cuh"

namespace cpattn {
namespace {

using namespace sm100;

constexpr int BM = 128, BN = 128, HD = 128;
constexpr int NS = 2;                          // K and V pipeline stages
constexpr int kThreads = 192;
constexpr uint32_t kTileBytes = BN * HD * 2;   // 32 KiB
constexpr uint32_t kHalf = 16384;              // one 64-column swizzled box
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS0 = 0, kColO = 256;    // S double buffer at 0 / 128, O at 256
constexpr float kRescaleThreshold = 8.f;       // log2 units

struct TcParams {
  cpattn_attn_args a;
  int n_qtiles;
  int n_ktiles;
};

struct Smem {
  uint8_t q[kTileBytes];
  uint8_t k[NS][kTileBytes];
  uint8_t v[NS][kTileBytes];
  uint8_t p[kTileBytes];
  uint64_t q_full;
  uint64_t k_full[NS], k_empty[NS], v_full[NS], v_empty[NS];
  uint64_t s_full[2];
  uint64_t p_full;
  uint64_t o_ready;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  long long min_lo, max_hi;
};

constexpr size_t kSmemBytes = sizeof(Smem) + 1024;  // + alignment slack

// 32 TMEM columns of this warp's 32 lanes, complete when it returns.
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

__global__ void __launch_bounds__(kThreads, 1)
dense_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  Smem& s = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                     ~uintptr_t(1023));
  const cpattn_attn_args& a = p.a;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // CTA -> (query tile, head); later query tiles (more keys) are launched first.
  const int qt = p.n_qtiles - 1 - (int)(blockIdx.x / a.Hq);
  const int h = (int)(blockIdx.x % a.Hq);
  const int g = h / (a.Hq / a.Hkv);
  const int q0 = qt * BM;
  volatile int* abort_flag = &s.abort;

  if (threadIdx.x == 0) {
    mbar_init(&s.q_full, 1);
    for (int i = 0; i < NS; ++i) {
      mbar_init(&s.k_full[i], 1);
      mbar_init(&s.k_empty[i], 1);
      mbar_init(&s.v_full[i], 1);
      mbar_init(&s.v_empty[i], 1);
    }
    mbar_init(&s.s_full[0], 1);
    mbar_init(&s.s_full[1], 1);
    mbar_init(&s.p_full, 128);
    mbar_init(&s.o_ready, 1);
    mbar_init(&s.drain, 1);
    s.abort = 0;
    s.min_lo = LLONG_MAX;
    s.max_hi = LLONG_MIN;
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
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s.tmem_base;

  // Each softmax thread owns one query row: its permitted key interval.
  const bool softmax_role = warp >= 2;
  const int r = (warp & 3) * 32 + lane;
  KeyInterval iv{1, 0};
  if (softmax_role) {
    const int64_t tok = (int64_t)q0 + r;
    if (tok < a.Tq) iv = allowed_interval(a, query_pos(a, tok));
    if (iv.lo <= iv.hi) {
      atomicMin(&s.min_lo, (long long)iv.lo);
      atomicMax(&s.max_hi, (long long)iv.hi);
    }
  }
  __syncthreads();
  const int64_t min_lo = s.min_lo, max_hi = s.max_hi;

  // A KV tile takes part iff its logical key range meets some row's interval.
  auto tile_info = [&](int kt, int64_t& kbase, int& kvalid) -> bool {
    const int64_t j0 = (int64_t)kt * BN;
    kvalid = (int)min((int64_t)BN, (int64_t)a.Tk - j0);
    kbase = logical_pos(a.kv_chunk_map, a.chunk_len, j0);
    return min_lo <= max_hi && kbase <= max_hi && kbase + kvalid - 1 >= min_lo;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int k_issued = 0, v_issued = 0;
      bool q_issued = false;
      for (int kt = 0; kt < p.n_ktiles; ++kt) {
        int64_t kbase;
        int kvalid;
        if (!tile_info(kt, kbase, kvalid)) continue;
        if (!q_issued) {
          mbar_arrive_expect_tx(&s.q_full, kTileBytes);
          tma_load_3d(s.q, &tm_q, &s.q_full, 0, h, q0);
          tma_load_3d(s.q + kHalf, &tm_q, &s.q_full, 64, h, q0);
          q_issued = true;
        }
        const int jt = k_issued, st = jt % NS;
        const uint32_t ph = (jt / NS) & 1;
        if (!mbar_wait(&s.k_empty[st], ph ^ 1, abort_flag)) break;
        mbar_arrive_expect_tx(&s.k_full[st], kTileBytes);
        tma_load_3d(s.k[st], &tm_k, &s.k_full[st], 0, g, kt * BN);
        tma_load_3d(s.k[st] + kHalf, &tm_k, &s.k_full[st], 64, g, kt * BN);
        ++k_issued;
        if (!mbar_wait(&s.v_empty[st], ph ^ 1, abort_flag)) break;
        mbar_arrive_expect_tx(&s.v_full[st], kTileBytes);
        tma_load_3d(s.v[st], &tm_v, &s.v_full[st], 0, g, kt * BN);
        tma_load_3d(s.v[st] + kHalf, &tm_v, &s.v_full[st], 64, g, kt * BN);
        ++v_issued;
      }
      if (*abort_flag) {  // let every copy in flight land before the CTA exits
        int no_abort = 0;
        if (q_issued) mbar_wait(&s.q_full, 0, &no_abort, 200000000ull);
        for (int j = max(0, k_issued - NS); j < k_issued; ++j)
          mbar_wait(&s.k_full[j % NS], (j / NS) & 1, &no_abort, 200000000ull);
        for (int j = max(0, v_issued - NS); j < v_issued; ++j)
          mbar_wait(&s.v_full[j % NS], (j / NS) & 1, &no_abort, 200000000ull);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc_qk = idesc_bf16_f32(BM, BN, 0, 0);   // Q, K both K-major
      const uint32_t idesc_pv = idesc_bf16_f32(BM, HD, 0, 1);   // P K-major, V MN-major
      const uint32_t q_addr = smem_u32(s.q), p_addr = smem_u32(s.p);
      bool ok = true, q_ready = false;
      int jt = 0;
      auto issue_pv = [&](int j) -> bool {
        const int st = j % NS;
        const uint32_t ph = (j / NS) & 1;
        if (!mbar_wait(&s.v_full[st], ph, abort_flag)) return false;
        if (!mbar_wait(&s.p_full, j & 1, abort_flag)) return false;
        tc_fence_after();
        const uint32_t v_addr = smem_u32(s.v[st]);
#pragma unroll
        for (int k = 0; k < BN / 16; ++k) {
          const uint64_t ad = smem_desc(p_addr + (k >> 2) * kHalf + (k & 3) * 32, 16, 1024, kSwizzle128B);
          const uint64_t bd = smem_desc(v_addr + k * 2048, kHalf, 1024, kSwizzle128B);
          umma_bf16_ss(tmem + kColO, ad, bd, idesc_pv, (j > 0 || k > 0) ? 1u : 0u);
        }
        umma_commit(&s.v_empty[st]);
        umma_commit(&s.o_ready);
        return true;
      };
      for (int kt = 0; kt < p.n_ktiles && ok; ++kt) {
        int64_t kbase;
        int kvalid;
        if (!tile_info(kt, kbase, kvalid)) continue;
        if (!q_ready) {
          if (!mbar_wait(&s.q_full, 0, abort_flag)) { ok = false; break; }
          q_ready = true;
        }
        const int st = jt % NS;
        const uint32_t ph = (jt / NS) & 1;
        if (!mbar_wait(&s.k_full[st], ph, abort_flag)) { ok = false; break; }
        tc_fence_after();
        const uint32_t k_addr = smem_u32(s.k[st]);
        const uint32_t d = tmem + kColS0 + (uint32_t)(jt & 1) * BN;
#pragma unroll
        for (int k = 0; k < HD / 16; ++k) {
          const uint32_t off = (k >> 2) * kHalf + (k & 3) * 32;
          const uint64_t ad = smem_desc(q_addr + off, 16, 1024, kSwizzle128B);
          const uint64_t bd = smem_desc(k_addr + off, 16, 1024, kSwizzle128B);
          umma_bf16_ss(d, ad, bd, idesc_qk, k > 0 ? 1u : 0u);
        }
        umma_commit(&s.s_full[jt & 1]);
        umma_commit(&s.k_empty[st]);
        if (jt >= 1 && !issue_pv(jt - 1)) { ok = false; break; }
        ++jt;
      }
      if (ok && jt >= 1) issue_pv(jt - 1);
      // every MMA issued so far must finish before TMEM is released
      umma_commit(&s.drain);
      int no_abort = 0;
      mbar_wait(&s.drain, 0, &no_abort, 1000000000ull);
    }
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const float sl2 = a.scale * 1.4426950408889634f;   // scores in exp2 units
    // l: fp32 sum of the weights (for LSE); lb: sum of the same weights as
    // rounded to bf16 for the PV product, so O = z / lb is a consistent
    // weighted average of V.
    float m2 = -CUDART_INF_F, l = 0.f, lb = 0.f;
    int jt = 0;
    bool ok = true;
    for (int kt = 0; kt < p.n_ktiles; ++kt) {
      int64_t kbase;
      int kvalid;
      if (!tile_info(kt, kbase, kvalid)) continue;
      int lo_c = 1, hi_c = 0;   // permitted columns of this row in this tile
      if (iv.lo <= iv.hi) {
        lo_c = (int)max((int64_t)0, min((int64_t)BN, iv.lo - kbase));
        hi_c = (int)max((int64_t)-1, min((int64_t)kvalid - 1, iv.hi - kbase));
      }
      ok = __all_sync(kFullMask, mbar_wait(&s.s_full[jt & 1], (jt >> 1) & 1, abort_flag));
      if (!ok) break;
      tc_fence_after();
      float sv[BN];
#pragma unroll
      for (int c4 = 0; c4 < BN / 32; ++c4) {
        uint32_t rr[32];
        tmem_ld32_sync(tmem + lane_base + kColS0 + (uint32_t)(jt & 1) * BN + c4 * 32, rr);
#pragma unroll
        for (int i = 0; i < 32; ++i) sv[c4 * 32 + i] = __uint_as_float(rr[i]);
      }
      float mx = -CUDART_INF_F;
      if (lo_c == 0 && hi_c == BN - 1) {
#pragma unroll
        for (int c = 0; c < BN; ++c) {
          sv[c] *= sl2;
          mx = fmaxf(mx, sv[c]);
        }
      } else {
#pragma unroll
        for (int c = 0; c < BN; ++c) {
          sv[c] = (c >= lo_c && c <= hi_c) ? sv[c] * sl2 : -CUDART_INF_F;
          mx = fmaxf(mx, sv[c]);
        }
      }
      float alpha = 1.f;
      bool rescale = false;
      if (mx > m2) {
        if (m2 == -CUDART_INF_F) {
          m2 = mx;                      // nothing accumulated yet for this row
        } else if (mx > m2 + kRescaleThreshold) {
          alpha = exp2f(m2 - mx);
          m2 = mx;
          rescale = true;
        }
      }
      const float mref = (m2 == -CUDART_INF_F) ? 0.f : m2;
      float rs = 0.f, rsb = 0.f;
      uint32_t pk[BN / 2];
#pragma unroll
      for (int c = 0; c < BN / 2; ++c) {
        const float p0 = exp2f(sv[2 * c] - mref);
        const float p1 = exp2f(sv[2 * c + 1] - mref);
        rs += p0 + p1;
        pk[c] = pack_bf16(p0, p1);
        rsb += __uint_as_float(pk[c] << 16) + __uint_as_float(pk[c] & 0xffff0000u);
      }
      l = l * alpha + rs;
      lb = lb * alpha + rsb;
      // O and the P buffer are free once the previous tile's PV has finished.
      if (jt > 0) {
        ok = __all_sync(kFullMask, mbar_wait(&s.o_ready, (jt - 1) & 1, abort_flag));
        if (!ok) break;
        tc_fence_after();
      }
      if (__any_sync(kFullMask, rescale)) {
#pragma unroll
        for (int c4 = 0; c4 < HD / 32; ++c4) {
          uint32_t oo[32];
          const uint32_t addr = tmem + lane_base + kColO + c4 * 32;
          tmem_ld32_sync(addr, oo);
#pragma unroll
          for (int i = 0; i < 32; ++i) oo[i] = __float_as_uint(__uint_as_float(oo[i]) * alpha);
          tmem_st32(addr, oo);
        }
        tmem_wait_st();
      }
      // P row -> shared memory in the 128B-swizzled K-major layout
      // [key block of 64][row][64 keys]: 16-byte chunk c of row r sits at
      // chunk position c ^ (r % 8).
#pragma unroll
      for (int ci = 0; ci < BN / 8; ++ci) {
        const int kb = ci >> 3, c16 = ci & 7;
        uint4 val = make_uint4(pk[ci * 4], pk[ci * 4 + 1], pk[ci * 4 + 2], pk[ci * 4 + 3]);
        *reinterpret_cast<uint4*>(s.p + kb * kHalf + r * 128 + ((c16 ^ (r & 7)) << 4)) = val;
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&s.p_full);
      ++jt;
    }
    if (ok && jt > 0) {
      ok = __all_sync(kFullMask, mbar_wait(&s.o_ready, (jt - 1) & 1, abort_flag));
      if (ok) tc_fence_after();
    }
    // epilogue: O = z / l, LSE = m + ln l (natural log); no key -> (0, -inf)
    const int64_t tok = (int64_t)q0 + r;
    const bool live = ok && jt > 0 && l > 0.f;
    const float inv = (live && lb > 0.f) ? 1.f / lb : 0.f;
    __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(a.o) + tok * a.o_stride_t + (int64_t)h * a.o_stride_h;
#pragma unroll
    for (int c4 = 0; c4 < HD / 32; ++c4) {
      uint32_t oo[32];
      if (ok && jt > 0) {
        tmem_ld32_sync(tmem + lane_base + kColO + c4 * 32, oo);
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

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
  if (threadIdx.x == 0 && s.abort) report_status(a.dev_status, CPATTN_ERR_TIMEOUT);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    cudaDriverEntryPointQueryResult q;
    void* ptr = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// [rows, heads, 128] bf16 with element strides (st_t, st_h); box = 64 x 1 x 128.
bool make_map(CUtensorMap* m, const void* base, int64_t rows, int heads, int64_t st_t,
              int64_t st_h) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[3] = {(cuuint64_t)HD, (cuuint64_t)heads, (cuuint64_t)rows};
  cuuint64_t strides[2] = {(cuuint64_t)st_h * 2, (cuuint64_t)st_t * 2};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)BM};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool dense_tc_supported(const cpattn_attn_args& a) {
  if (a.dtype != CPATTN_BF16 || a.Dqk != HD || a.Dv != HD) return false;
  if (a.kv_chunk_len != 0 || a.Tq <= 0 || a.Tk <= 0) return false;
  if ((a.q_chunk_map || a.kv_chunk_map) && a.chunk_len % BN != 0) return false;
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
  cudaError_t e = cudaFuncSetAttribute(dense_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)p.n_qtiles * (unsigned)a.Hq;
  dense_tc_kernel<<<grid, kThreads, kSmemBytes, stream>>>(tq, tk, tv, p);
  *launched = true;
  return cudaGetLastError();
}

}  // namespace cpattn
