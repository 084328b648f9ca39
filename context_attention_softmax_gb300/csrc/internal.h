// Host-side declarations shared by the API layer and the kernel launchers.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <string>

#include "cpattn.h"

namespace cpattn {

// Selection of keys for the general (warp-per-row) kernel.
enum KeyMode { kDense = 0, kTokens = 1, kBlocks = 2 };

struct SparseArgs {
  const int32_t* indices;  // [Tq, index_heads, topk]
  int32_t topk;
  int32_t index_heads;
  int32_t block_size;
};

// Sets the calling thread's cpattn_last_error() message and returns s.
cpattn_status report_error(cpattn_status s, const char* msg);

// Host caches (host_cache.cu).  encode_bf16_3d: a 3-D bf16 TMA map with
// 128-byte swizzle (dims innermost first, strides in bytes), reused while
// the pointer, shape, strides and box repeat; false if it cannot be encoded.
// ensure_smem_attr: sets a kernel's dynamic shared-memory limit once per
// device.  device_sm_count: SMs of the current device.
bool encode_bf16_3d(CUtensorMap* out, const void* base, const uint64_t (&dims)[3],
                    const uint64_t (&strides)[2], const uint32_t (&box)[3]);
cudaError_t ensure_smem_attr(const void* func, int bytes);
int device_sm_count();

// Launchers return the cudaError_t of the launch (no synchronisation).
cudaError_t launch_rowwise(const cpattn_attn_args& a, KeyMode mode, const SparseArgs& sp,
                           cudaStream_t stream);
cudaError_t launch_lse_merge(int32_t n_parts, const float* part_o, const float* part_lse,
                             int32_t Tq, int32_t H, int32_t Dv, void* o, int32_t o_dtype,
                             int64_t o_stride_t, int64_t o_stride_h, float* lse,
                             cudaStream_t stream);
// DSA indexer (fp32 qI [Tq, Hq, D], kI [Tk, 1, D]): workspace bytes for a
// given grid, the grid the launcher uses, and the launch (scores, norms,
// per-row certified top-k).
size_t dsa_indexer_workspace(const cpattn_attn_args& a, int grid);
// Tensor-core indexer scores (dsa_indexer_tc.cu): whether the shape takes
// them, their extra workspace, the bound factor c of their error
// (|S - score| <= c a_i ||kI_j||) and the launch (split, tile intervals,
// score GEMM) writing S [Tq, ldS].
bool dsa_indexer_tc_supported(const cpattn_attn_args& a);
size_t dsa_indexer_tc_workspace(const cpattn_attn_args& a);
float dsa_indexer_tc_bound(const cpattn_attn_args& a);
cudaError_t launch_dsa_indexer_scores_tc(const cpattn_attn_args& a, const float* w, float* S,
                                         int64_t ldS, void* tc_ws, cudaStream_t stream);
int dsa_indexer_grid(const cpattn_attn_args& a);
cudaError_t launch_dsa_indexer(const cpattn_attn_args& a, const float* w, int topk, int32_t* out,
                               void* ws, cudaStream_t stream);
// The same merge over bf16 parts (the MoBA slot summaries).
cudaError_t launch_lse_merge_bf16parts(int32_t n_parts, const __nv_bfloat16* part_o,
                                       const float* part_lse, int32_t Tq, int32_t H, int32_t Dv,
                                       void* o, int32_t o_dtype, int64_t o_stride_t,
                                       int64_t o_stride_h, float* lse, cudaStream_t stream);
// tcgen05 dense kernel (bf16, d = 128): supported() says whether the
// arguments fit it; launch sets *launched = false when the layout cannot be
// described by TMA tensor maps (the caller then uses the general kernel).
bool dense_tc_supported(const cpattn_attn_args& a);
cudaError_t launch_dense_tc(const cpattn_attn_args& a, cudaStream_t stream, bool* launched);
// Balanced schedule of the dense tensor-core kernel (no KV chunk map): the
// workspace it needs (0 when it does not apply) and its launch; `launched`
// stays false when the workspace is missing or too small.
size_t dense_tc_bal_workspace(const cpattn_attn_args& a);
cudaError_t launch_dense_tc_bal(const cpattn_attn_args& a, void* ws, size_t ws_bytes,
                                cudaStream_t stream, bool* launched);
// Block-grouped MoBA attention on the tensor cores (bf16, d = 128, block
// size a multiple of 128, keys in logical order).  `sel` is the block list
// [Tq, index_heads, slots]; writes o and lse through partial summaries and
// the LSE merge.
bool moba_tc_supported(const cpattn_attn_args& a, int32_t index_heads, int32_t block_size,
                       int32_t slots);
size_t moba_tc_workspace(const cpattn_attn_args& a, int32_t slots, int32_t block_size);
cudaError_t launch_moba_tc(const cpattn_attn_args& a, const int32_t* sel, int32_t slots,
                           int32_t index_heads, int32_t block_size, void* workspace,
                           cudaStream_t stream);
// DSA token-index attention on the tensor cores for absorbed-MLA shapes:
// bf16, 128 query heads over one KV head, key rows of 576 channels whose
// first 512 are the values (v aliases k), indices shared by all heads.
bool dsa_tc_supported(const cpattn_attn_args& a, int32_t index_heads, int32_t block_size);
cudaError_t launch_dsa_tc(const cpattn_attn_args& a, const int32_t* indices, int32_t topk,
                          cudaStream_t stream, bool* launched);
// Workspace of the block gate: the preferred size (with it, bf16 queries of
// head dim 128 over at most 128 blocks use the tensor-core gate) and the
// minimum (block means only).
size_t block_gate_workspace(const cpattn_attn_args& a, int32_t block_size);
size_t block_gate_workspace_min(const cpattn_attn_args& a, int32_t block_size);
bool gate_tc_supported(const cpattn_attn_args& a, int32_t block_size, int32_t topk);
size_t gate_tc_parts_bytes(const cpattn_attn_args& a, int32_t block_size);
cudaError_t launch_gate_tc(const cpattn_attn_args& a, int32_t block_size, int32_t topk, int32_t* sel,
                           const double* mu64, const float* mu32, void* parts, cudaStream_t stream,
                           bool* launched);
size_t block_gate_smem(int n_blocks, int D);
// Backward of the dense chunk attention on the tensor cores (dense_bwd.cu):
// bf16, d = 128; fp32 gradients; workspace for D, LSE2 and tile intervals.
bool dense_bwd_supported(const cpattn_attn_args& a);
size_t dense_bwd_workspace(const cpattn_attn_args& a);
cudaError_t launch_dense_bwd(const cpattn_attn_args& a, const void* g, int64_t g_st, int64_t g_sh,
                             float* dq, int64_t dq_st, int64_t dq_sh, float* dk, int64_t dk_st,
                             int64_t dk_sh, float* dv, int64_t dv_st, int64_t dv_sh, void* ws,
                             cudaStream_t stream);
// MLA projections on the tensor cores (mla_gemm.cu); arguments validated by
// the caller.
cpattn_status mla_v_up_impl(const void* o_latent, int64_t o_st, int64_t o_sh,
                            const void* up_v_weight, int32_t T, int32_t H, int32_t L, int32_t V,
                            void* out, int64_t out_st, int64_t out_sh, int32_t* dev_status,
                            int64_t wait_limit_ns, cudaStream_t stream);
cpattn_status mla_kv_impl(const void* kv_c, int64_t c_st, const void* k_shared, int64_t ks_st,
                          const void* wkv_b, int32_t T, int32_t L, int32_t H, int32_t N, int32_t R,
                          int32_t V, void* k_out, int64_t k_st, int64_t k_sh, void* v_out,
                          int64_t v_st, int64_t v_sh, int32_t* dev_status, int64_t wait_limit_ns,
                          cudaStream_t stream);
cudaError_t launch_block_gate(const cpattn_attn_args& a, int32_t block_size, int32_t topk,
                              int32_t* sel, void* workspace, size_t workspace_bytes,
                              cudaStream_t stream);

}  // namespace cpattn
