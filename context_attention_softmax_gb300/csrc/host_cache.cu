// Host-side caches of the launchers, so that a repeated call does no more
// host work than it must before its launch:
//  * TMA tensor maps, encoded once per distinct (base pointer, dims, strides,
//    box) in a small per-thread table and copied out on a hit;
//  * the dynamic shared-memory attribute of each kernel, set once per device
//    (and again only when a larger size is asked for);
//  * the SM count of each device.
// No device memory is involved; nothing here synchronises.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "internal.h"

namespace cpattn {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    PFN_cuTensorMapEncodeTiled_v12000 f = nullptr;
    cudaDriverEntryPointQueryResult q;
    void* ptr = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      f = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    return f;
  }();
  return fn;
}

struct MapKey {
  const void* base;
  uint64_t dims[3];
  uint64_t strides[2];
  uint32_t box[3];
  uint32_t pad;
};

struct MapEntry {
  MapKey key;
  CUtensorMap map;
  bool used;
};

constexpr int kMapSlots = 64;
thread_local MapEntry t_maps[kMapSlots];
thread_local int t_next = 0;

struct AttrEntry {
  int dev;
  const void* func;
  int bytes;
};
constexpr int kAttrSlots = 256;
std::mutex g_attr_mutex;
AttrEntry g_attr[kAttrSlots];
int g_attr_n = 0;

constexpr int kMaxDev = 64;
int g_sm_count[kMaxDev];

}  // namespace

bool encode_bf16_3d(CUtensorMap* out, const void* base, const uint64_t (&dims)[3],
                    const uint64_t (&strides)[2], const uint32_t (&box)[3]) {
  MapKey key;
  std::memset(&key, 0, sizeof(key));
  key.base = base;
  for (int i = 0; i < 3; ++i) key.dims[i] = dims[i], key.box[i] = box[i];
  for (int i = 0; i < 2; ++i) key.strides[i] = strides[i];
  for (int i = 0; i < kMapSlots; ++i) {
    if (t_maps[i].used && std::memcmp(&t_maps[i].key, &key, sizeof(key)) == 0) {
      *out = t_maps[i].map;
      return true;
    }
  }
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t d[3] = {dims[0], dims[1], dims[2]};
  cuuint64_t s[2] = {strides[0], strides[1]};
  cuuint32_t b[3] = {box[0], box[1], box[2]};
  cuuint32_t estr[3] = {1, 1, 1};
  if (fn(out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), d, s, b, estr,
         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  MapEntry& e = t_maps[t_next];
  t_next = (t_next + 1) % kMapSlots;
  e.key = key;
  e.map = *out;
  e.used = true;
  return true;
}

cudaError_t ensure_smem_attr(const void* func, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_attr_mutex);
  for (int i = 0; i < g_attr_n; ++i) {
    if (g_attr[i].dev == dev && g_attr[i].func == func) {
      if (g_attr[i].bytes >= bytes) return cudaSuccess;
      e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
      if (e == cudaSuccess) g_attr[i].bytes = bytes;
      return e;
    }
  }
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && g_attr_n < kAttrSlots) g_attr[g_attr_n++] = AttrEntry{dev, func, bytes};
  return e;
}

int device_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (dev >= 0 && dev < kMaxDev && g_sm_count[dev] > 0) return g_sm_count[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 1;
  if (dev >= 0 && dev < kMaxDev) g_sm_count[dev] = n;
  return n;
}

}  // namespace cpattn
