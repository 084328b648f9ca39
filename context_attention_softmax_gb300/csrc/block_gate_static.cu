// cpattn_block_gate_static: the MoBA block gate with its scratch memory (the
// per-block key means and, for the tensor-core gate, their bf16 split terms)
// held in a fixed array inside this library instead of a caller-supplied
// workspace.
//
// Who needs it: callers that cannot allocate device memory at the point of
// the call - code that runs while a caching allocator must not grow, inside
// a host callback or a custom runtime that owns every allocation, or a
// plugin that receives only the tensors of its inputs and outputs.  They
// pass q, k and sel as usual and never a workspace.
//
// The array is a file-scope __device__ object of kStaticScratchBytes; every
// GPU that loads this library keeps it until the process exits.  Host code
// cannot use the array's name as a device address, so the first call on each
// device (with that device current) looks the address up with
// cudaGetSymbolAddress and caches it; make that first call before any stream
// capture.  All calls on a device share the one array: two calls whose work
// overlaps on the GPU (different streams, no ordering) race and may corrupt
// each other's block means.  Calls in stream order are safe.  Nothing in the
// array needs to start at zero: each call overwrites every block mean it
// reads.  No cudaMalloc, cudaFree or allocating library routine is called.
//
// A shape is accepted only when the whole workspace cpattn_block_gate would
// ask for (cpattn_workspace_size(CPATTN_OP_BLOCK_GATE, ...)) fits the array,
// so this entry always takes the same kernels as cpattn_block_gate given that
// workspace; the MoBA shape of 128 blocks x 32 KV heads x d 128 needs 9.4 MB.
#include <cstdio>
#include <mutex>

#include "cpattn.h"
#include "internal.h"

namespace cpattn {
namespace {

constexpr size_t kStaticScratchBytes = size_t(16) << 20;  // 16 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_gate_scratch[kStaticScratchBytes];

std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the array on the current device (looked up once).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_gate_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace cpattn

extern "C" cpattn_status cpattn_block_gate_static(const cpattn_attn_args* args,
                                                  int32_t block_size, int32_t topk,
                                                  int32_t* sel, void* stream) {
  using namespace cpattn;
  if (args == nullptr || block_size < 1 || args->Tk < 0 || args->Hkv < 1 || args->Dqk < 1)
    // malformed arguments: the regular entry point rejects them with its message
    return cpattn_block_gate(args, block_size, topk, sel, nullptr, 0, stream);
  const size_t need = block_gate_workspace(*args, block_size);
  if (need > kStaticScratchBytes) {
    char msg[256];
    snprintf(msg, sizeof(msg),
             "cpattn_block_gate_static: the gate needs %zu bytes of scratch, more than "
             "its fixed %zu-byte array; use cpattn_block_gate with a workspace",
             need, kStaticScratchBytes);
    return report_error(CPATTN_ERR_UNSUPPORTED, msg);
  }
  void* scratch = nullptr;
  const cudaError_t e = scratch_address(&scratch);
  if (e != cudaSuccess) {
    char msg[256];
    snprintf(msg, sizeof(msg), "cpattn_block_gate_static: cudaGetSymbolAddress failed: %s",
             cudaGetErrorString(e));
    return report_error(CPATTN_ERR_CUDA, msg);
  }
  return cpattn_block_gate(args, block_size, topk, sel, scratch, kStaticScratchBytes, stream);
}
