// Pieces shared by the dense tensor-core kernels: tile sizes, TMEM loads,
// the (head, query tile) blocks of a work unit and the TMA descriptors.
#pragma once
#include <cuda.h>

#include <climits>

#include "common.cuh"
#include "internal.h"
#include "sm100.cuh"

namespace cpattn {
namespace {

using namespace sm100;

constexpr int BM = 128, BN = 128, HD = 128;
constexpr int NS = 2;                          // K and V pipeline stages (j & 1 picks one)
constexpr int kThreads = 384;
constexpr uint32_t kTileBytes = BN * HD * 2;   // 32 KiB
constexpr uint32_t kHalf = 16384;              // one 64-column swizzled box
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColO = 256;     // S_X at 128*X, O_X at 256 + 128*X
constexpr float kRescaleThreshold = 8.f;       // log2 units
constexpr int kMaxKTiles = 4096;               // Tk <= 524288 on this path
// Register split: launch budget 168 x 384.  Warpgroup 0 (producer, MMA, two
// idle warps) drops to 64 registers per thread, the two softmax warpgroups
// rise to 216: 128 * 64 + 256 * 216 = 63488 <= 168 * 384 = 64512.
constexpr uint32_t kRegsControl = 64, kRegsSoftmax = 216;
static_assert(128 * kRegsControl + 256 * kRegsSoftmax <= 168 * kThreads, "register split");

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

// 128 TMEM columns of this warp's 32 lanes in one load, complete on return.
__device__ __forceinline__ void tmem_ld128_sync(uint32_t taddr, uint32_t (&r)[128]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x128.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63, %64, %65, %66, %67, %68, %69, %70, %71, %72, %73, %74, %75, %76, %77, %78, %79, %80, %81, %82, %83, %84, %85, %86, %87, %88, %89, %90, %91, %92, %93, %94, %95, %96, %97, %98, %99, %100, %101, %102, %103, %104, %105, %106, %107, %108, %109, %110, %111, %112, %113, %114, %115, %116, %117, %118, %119, %120, %121, %122, %123, %124, %125, %126, %127}, [%128];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]), "=r"(r[64]), "=r"(r[65]), "=r"(r[66]), "=r"(r[67]), "=r"(r[68]), "=r"(r[69]), "=r"(r[70]), "=r"(r[71]), "=r"(r[72]), "=r"(r[73]), "=r"(r[74]), "=r"(r[75]), "=r"(r[76]), "=r"(r[77]), "=r"(r[78]), "=r"(r[79]), "=r"(r[80]), "=r"(r[81]), "=r"(r[82]), "=r"(r[83]), "=r"(r[84]), "=r"(r[85]), "=r"(r[86]), "=r"(r[87]), "=r"(r[88]), "=r"(r[89]), "=r"(r[90]), "=r"(r[91]), "=r"(r[92]), "=r"(r[93]), "=r"(r[94]), "=r"(r[95]), "=r"(r[96]), "=r"(r[97]), "=r"(r[98]), "=r"(r[99]), "=r"(r[100]), "=r"(r[101]), "=r"(r[102]), "=r"(r[103]), "=r"(r[104]), "=r"(r[105]), "=r"(r[106]), "=r"(r[107]), "=r"(r[108]), "=r"(r[109]), "=r"(r[110]), "=r"(r[111]), "=r"(r[112]), "=r"(r[113]), "=r"(r[114]), "=r"(r[115]), "=r"(r[116]), "=r"(r[117]), "=r"(r[118]), "=r"(r[119]), "=r"(r[120]), "=r"(r[121]), "=r"(r[122]), "=r"(r[123]), "=r"(r[124]), "=r"(r[125]), "=r"(r[126]), "=r"(r[127])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 t = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&t);
}

// (head, first query row) of block X of unit u.
struct Block {
  int head, q0;
};
__device__ __forceinline__ Block block_of(int Hq, int head_pairs, int n_qtiles, int u, int X) {
  if (head_pairs) {
    const int hp = Hq / 2;
    const int qt = n_qtiles - 1 - u / hp;   // later query tiles (more keys) first
    return Block{2 * (u % hp) + X, qt * BM};
  }
  const int n_pair = (n_qtiles + 1) / 2;
  const int pi = n_pair - 1 - u / Hq;
  return Block{u % Hq, (2 * pi + X) * BM};
}

// Folded head pairs (even GQA groups, one causal sequence): unit u holds query
// tile t of head 2p and query tile n_qtiles-1-t of head 2p+1.  Under a causal
// mask tile t sees about t + offset/128 key tiles, so every unit carries the
// same total; both heads read the same KV head.
__device__ __forceinline__ Block folded_block_of(int Hq, int n_qtiles, int u, int X) {
  const int hp = Hq / 2;
  const int t = u / hp, pr = u % hp;
  return Block{2 * pr + X, (X ? n_qtiles - 1 - t : t) * BM};
}

// Row-contiguous stores of one warp's rows (lane = row, fp32 values held per
// lane) through a staging slice of shared memory: 32 rows x 16 columns with
// a row stride of 20 floats, so that a lane's four 16-byte writes and the
// eight-lane phases of the reads fall on distinct banks.  Lane L then stores
// columns 4 (L % 4) .. + 3 of row 8 j + L / 4: one store instruction writes
// eight rows' 64 contiguous bytes instead of 32 rows' scattered 16-byte
// pieces.  Every lane of the warp calls these together.
constexpr int kStageStride = 20;
constexpr size_t kStageSliceBytes = 32 * kStageStride * sizeof(float);

struct StagedRows {
  float* dst[4];   // rows 8 j + lane / 4, already offset by 4 (lane % 4) columns
  bool ok[4];
};

__device__ __forceinline__ StagedRows staged_rows(float* row, bool row_ok) {
  const int lane = threadIdx.x & 31;
  StagedRows t;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int src = 8 * j + (lane >> 2);
    t.dst[j] = reinterpret_cast<float*>(
                   __shfl_sync(kFullMask, reinterpret_cast<unsigned long long>(row), src)) +
               4 * (lane & 3);
    t.ok[j] = __shfl_sync(kFullMask, row_ok, src);
  }
  return t;
}

// Columns col0 .. col0 + 31 of the warp's rows: v (this lane's row) x mul.
// Ends with the stage free again; __syncwarp orders the stores for the warp.
__device__ __forceinline__ void store_rows32(float (*stage)[kStageStride], const StagedRows& t,
                                             const uint32_t (&v)[32], float mul, int col0) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
#pragma unroll
    for (int i = 0; i < 16; i += 4)
      *reinterpret_cast<float4*>(&stage[lane][i]) =
          make_float4(__uint_as_float(v[16 * half + i]) * mul,
                      __uint_as_float(v[16 * half + i + 1]) * mul,
                      __uint_as_float(v[16 * half + i + 2]) * mul,
                      __uint_as_float(v[16 * half + i + 3]) * mul);
    __syncwarp();
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float4 x = *reinterpret_cast<const float4*>(&stage[8 * j + (lane >> 2)][4 * (lane & 3)]);
      if (t.ok[j]) *reinterpret_cast<float4*>(t.dst[j] + col0 + 16 * half) = x;
    }
    __syncwarp();
  }
}

// [rows, heads, 128] bf16 with element strides (st_t, st_h); box = 64 x 1 x 128.
bool make_map(CUtensorMap* m, const void* base, int64_t rows, int heads, int64_t st_t,
              int64_t st_h) {
  const uint64_t dims[3] = {(uint64_t)HD, (uint64_t)heads, (uint64_t)rows};
  const uint64_t strides[2] = {(uint64_t)st_h * 2, (uint64_t)st_t * 2};
  const uint32_t box[3] = {64, 1, (uint32_t)BM};
  return encode_bf16_3d(m, base, dims, strides, box);
}

}  // namespace
}  // namespace cpattn
