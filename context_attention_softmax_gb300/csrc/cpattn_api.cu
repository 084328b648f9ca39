// C ABI entry points: host-side validation, then dispatch to the kernels.
// Every check runs before anything is launched, so a rejected call leaves the
// stream untouched.  Messages are kept per calling thread.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <string>

#include "cpattn.h"
#include "internal.h"

namespace cpattn {
namespace {

thread_local std::string g_last_error;

cpattn_status fail(cpattn_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

cpattn_status ok() {
  g_last_error.clear();
  return CPATTN_OK;
}

cpattn_status cuda_status(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return ok();
  return fail(CPATTN_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t elem_size(int32_t dtype) { return dtype == CPATTN_BF16 ? 2 : 4; }

#define CHECK(cond, code, ...) \
  do {                         \
    if (!(cond)) return fail(code, __VA_ARGS__); \
  } while (0)

// A [T, H, D] operand: pointer and strides aligned to 16 bytes.
cpattn_status check_tensor(const char* name, const void* p, int64_t st, int64_t sh, int64_t T,
                           size_t es) {
  if (T == 0) return CPATTN_OK;
  CHECK(p != nullptr, CPATTN_ERR_INVALID_ARG, "%s is NULL", name);
  CHECK(aligned16(p), CPATTN_ERR_INVALID_ARG, "%s is not 16-byte aligned", name);
  CHECK(st >= 0 && sh >= 0, CPATTN_ERR_INVALID_ARG, "%s has a negative stride", name);
  CHECK((st * (int64_t)es) % 16 == 0 && (sh * (int64_t)es) % 16 == 0, CPATTN_ERR_INVALID_ARG,
        "%s strides (%lld, %lld elements) are not multiples of 16 bytes", name, (long long)st,
        (long long)sh);
  return CPATTN_OK;
}

#define TRY(expr)                          \
  do {                                     \
    cpattn_status s_ = (expr);             \
    if (s_ != CPATTN_OK) return s_;        \
  } while (0)

// Checks shared by every attention entry point.  need_v: v/Dv used; need_o:
// o written.
cpattn_status check_attn(const cpattn_attn_args* a, bool need_v, bool need_o) {
  CHECK(a != nullptr, CPATTN_ERR_INVALID_ARG, "args is NULL");
  CHECK(a->dtype == CPATTN_BF16 || a->dtype == CPATTN_FP32, CPATTN_ERR_INVALID_ARG,
        "dtype %d is neither CPATTN_BF16 nor CPATTN_FP32", a->dtype);
  CHECK(a->Tq >= 0 && a->Tk >= 0, CPATTN_ERR_INVALID_ARG, "Tq=%d, Tk=%d must be >= 0", a->Tq, a->Tk);
  CHECK(a->Hq >= 1 && a->Hkv >= 1, CPATTN_ERR_INVALID_ARG, "Hq=%d, Hkv=%d must be >= 1", a->Hq, a->Hkv);
  CHECK(a->Hq % a->Hkv == 0, CPATTN_ERR_INVALID_ARG, "Hq=%d is not a multiple of Hkv=%d", a->Hq, a->Hkv);
  CHECK(a->Dqk >= 8 && a->Dqk % 8 == 0, CPATTN_ERR_INVALID_ARG, "Dqk=%d must be a positive multiple of 8", a->Dqk);
  CHECK(a->Dqk <= 1024, CPATTN_ERR_UNSUPPORTED, "Dqk=%d exceeds 1024", a->Dqk);
  const size_t es = elem_size(a->dtype);
  TRY(check_tensor("q", a->q, a->q_stride_t, a->q_stride_h, a->Tq, es));
  TRY(check_tensor("k", a->k, a->k_stride_t, a->k_stride_h, a->Tk, es));
  if (need_v) {
    CHECK(a->Dv >= 8 && a->Dv % 8 == 0, CPATTN_ERR_INVALID_ARG, "Dv=%d must be a positive multiple of 8", a->Dv);
    CHECK(a->Dv <= 512, CPATTN_ERR_UNSUPPORTED, "Dv=%d exceeds 512", a->Dv);
    TRY(check_tensor("v", a->v, a->v_stride_t, a->v_stride_h, a->Tk, es));
  }
  if (need_o) TRY(check_tensor("o", a->o, a->o_stride_t, a->o_stride_h, a->Tq, es));
  CHECK(a->causal == 0 || a->causal == 1, CPATTN_ERR_INVALID_ARG, "causal=%d must be 0 or 1", a->causal);
  CHECK(a->causal_offset >= 0, CPATTN_ERR_INVALID_ARG, "causal_offset=%lld must be >= 0",
        (long long)a->causal_offset);
  CHECK(std::isfinite(a->scale), CPATTN_ERR_INVALID_ARG, "scale is not finite");
  if (a->cu_seqlens != nullptr)
    CHECK(a->num_seqs >= 1, CPATTN_ERR_INVALID_ARG, "num_seqs=%d must be >= 1 with cu_seqlens", a->num_seqs);
  if (a->q_chunk_map != nullptr || a->kv_chunk_map != nullptr)
    CHECK(a->chunk_len > 0, CPATTN_ERR_INVALID_ARG, "a chunk map needs chunk_len > 0");
  if (a->q_chunk_map != nullptr)
    CHECK(a->n_q_chunks >= 1 && (int64_t)a->n_q_chunks * a->chunk_len >= a->Tq,
          CPATTN_ERR_INVALID_ARG, "q_chunk_map: n_q_chunks=%d * chunk_len=%d does not cover Tq=%d",
          a->n_q_chunks, a->chunk_len, a->Tq);
  if (a->kv_chunk_map != nullptr) {
    CHECK((int64_t)a->n_kv_chunks * a->chunk_len == a->Tk, CPATTN_ERR_INVALID_ARG,
          "kv_chunk_map: n_kv_chunks=%d * chunk_len=%d != Tk=%d", a->n_kv_chunks, a->chunk_len, a->Tk);
    CHECK(a->n_kv_chunks <= 4096, CPATTN_ERR_UNSUPPORTED, "n_kv_chunks=%d exceeds 4096", a->n_kv_chunks);
  }
  return CPATTN_OK;
}

}  // namespace

cpattn_status report_error(cpattn_status s, const char* msg) {
  g_last_error = msg;
  return s;
}

}  // namespace cpattn

using namespace cpattn;

extern "C" {

cpattn_status cpattn_chunk_fwd(const cpattn_attn_args* a, void* workspace, size_t workspace_bytes,
                               void* stream) {
  CHECK(a != nullptr, CPATTN_ERR_INVALID_ARG, "args is NULL");
  const bool partials_only = a->kv_chunk_len > 0 && a->o == nullptr;
  TRY(check_attn(a, true, !partials_only));
  CHECK(a->kv_chunk_len >= 0, CPATTN_ERR_INVALID_ARG, "kv_chunk_len=%d must be >= 0", a->kv_chunk_len);
  if (partials_only)
    CHECK(a->lse == nullptr, CPATTN_ERR_INVALID_ARG,
          "with o = NULL (partial summaries only) lse must be NULL too");
  if (a->kv_chunk_len > 0 && a->Tk > 0 && (int64_t)a->Tq * a->Hq > 0)
    CHECK(a->partial_o != nullptr && a->partial_lse != nullptr, CPATTN_ERR_INVALID_ARG,
          "kv_chunk_len > 0 needs partial_o and partial_lse");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (dense_tc_supported(*a)) {
    bool launched = false;
    cudaError_t e = launch_dense_tc_bal(*a, workspace, workspace_bytes, st, &launched);
    if (e != cudaSuccess || launched) return cuda_status(e, "cpattn_chunk_fwd tensor-core launch");
    e = launch_dense_tc(*a, st, &launched);
    if (e != cudaSuccess || launched) return cuda_status(e, "cpattn_chunk_fwd tensor-core launch");
  }
  SparseArgs none{nullptr, 0, 1, 1};
  return cuda_status(launch_rowwise(*a, kDense, none, st), "cpattn_chunk_fwd launch");
}

cpattn_status cpattn_lse_merge(int32_t n_parts, const float* part_o, const float* part_lse,
                               int32_t Tq, int32_t H, int32_t Dv, void* o, int32_t o_dtype,
                               int64_t o_stride_t, int64_t o_stride_h, float* lse, void* stream) {
  CHECK(n_parts >= 0 && Tq >= 0 && H >= 1, CPATTN_ERR_INVALID_ARG,
        "n_parts=%d, Tq=%d must be >= 0 and H=%d >= 1", n_parts, Tq, H);
  CHECK(Dv >= 8 && Dv % 8 == 0, CPATTN_ERR_INVALID_ARG, "Dv=%d must be a positive multiple of 8", Dv);
  CHECK(o_dtype == CPATTN_BF16 || o_dtype == CPATTN_FP32, CPATTN_ERR_INVALID_ARG,
        "o_dtype %d is neither CPATTN_BF16 nor CPATTN_FP32", o_dtype);
  if ((int64_t)Tq * H > 0) {
    if (n_parts > 0) {
      CHECK(part_o != nullptr && part_lse != nullptr, CPATTN_ERR_INVALID_ARG, "part_o/part_lse is NULL");
      CHECK(aligned16(part_o), CPATTN_ERR_INVALID_ARG, "part_o is not 16-byte aligned");
    }
    TRY(check_tensor("o", o, o_stride_t, o_stride_h, Tq, elem_size(o_dtype)));
  }
  return cuda_status(launch_lse_merge(n_parts, part_o, part_lse, Tq, H, Dv, o, o_dtype, o_stride_t,
                                      o_stride_h, lse, reinterpret_cast<cudaStream_t>(stream)),
                     "cpattn_lse_merge launch");
}

cpattn_status cpattn_topk_sparse_fwd(const cpattn_attn_args* a, const int32_t* indices,
                                     int32_t topk, int32_t index_heads, int32_t block_size,
                                     void* workspace, size_t workspace_bytes, void* stream) {
  TRY(check_attn(a, true, true));
  CHECK(topk >= 0, CPATTN_ERR_INVALID_ARG, "topk=%d must be >= 0", topk);
  CHECK(index_heads == 1 || index_heads == a->Hq, CPATTN_ERR_INVALID_ARG,
        "index_heads=%d must be 1 or Hq=%d", index_heads, a->Hq);
  CHECK(block_size >= 1, CPATTN_ERR_INVALID_ARG, "block_size=%d must be >= 1", block_size);
  CHECK(a->kv_chunk_len == 0, CPATTN_ERR_UNSUPPORTED, "partial summaries are not produced by the sparse path");
  if (topk > 0 && a->Tq > 0) CHECK(indices != nullptr, CPATTN_ERR_INVALID_ARG, "indices is NULL");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (block_size > 1 && topk > 0 && moba_tc_supported(*a, index_heads, block_size, topk)) {
    const size_t need = moba_tc_workspace(*a, topk, block_size);
    CHECK(workspace != nullptr && workspace_bytes >= need, CPATTN_ERR_WORKSPACE,
          "workspace of %zu bytes given, %zu needed", workspace_bytes, need);
    return cuda_status(launch_moba_tc(*a, indices, topk, index_heads, block_size, workspace, st),
                       "cpattn_topk_sparse_fwd block-grouped launch");
  }
  if (block_size == 1 && topk > 0 && dsa_tc_supported(*a, index_heads, block_size)) {
    bool launched = false;
    cudaError_t e = launch_dsa_tc(*a, indices, topk, st, &launched);
    if (e != cudaSuccess || launched) return cuda_status(e, "cpattn_topk_sparse_fwd tensor-core launch");
  }
  SparseArgs sp{indices, topk, index_heads, block_size};
  return cuda_status(launch_rowwise(*a, block_size == 1 ? kTokens : kBlocks, sp, st),
                     "cpattn_topk_sparse_fwd launch");
}

cpattn_status cpattn_block_gate(const cpattn_attn_args* a, int32_t block_size, int32_t topk,
                                int32_t* sel, void* workspace, size_t workspace_bytes,
                                void* stream) {
  TRY(check_attn(a, false, false));
  CHECK(block_size >= 1, CPATTN_ERR_INVALID_ARG, "block_size=%d must be >= 1", block_size);
  CHECK(topk >= 0, CPATTN_ERR_INVALID_ARG, "topk=%d must be >= 0", topk);
  CHECK(topk <= 64, CPATTN_ERR_UNSUPPORTED, "topk=%d exceeds 64", topk);
  CHECK(a->cu_seqlens == nullptr && a->kv_chunk_map == nullptr, CPATTN_ERR_UNSUPPORTED,
        "the block gate takes one sequence with keys in logical order (no cu_seqlens, no kv_chunk_map)");
  if ((int64_t)a->Tq * a->Hq > 0) CHECK(sel != nullptr, CPATTN_ERR_INVALID_ARG, "sel is NULL");
  const int n_blocks = a->Tk / block_size;
  CHECK(block_gate_smem(n_blocks, a->Dqk) <= 200 * 1024, CPATTN_ERR_UNSUPPORTED,
        "%d blocks of head dim %d do not fit the gate's shared-memory staging", n_blocks, a->Dqk);
  const size_t need = block_gate_workspace_min(*a, block_size);
  CHECK(workspace_bytes >= need && (need == 0 || workspace != nullptr), CPATTN_ERR_WORKSPACE,
        "workspace of %zu bytes given, %zu needed", workspace_bytes, need);
  if (need > 0) CHECK(aligned16(workspace), CPATTN_ERR_INVALID_ARG, "workspace is not 16-byte aligned");
  return cuda_status(launch_block_gate(*a, block_size, topk, sel, workspace, workspace_bytes,
                                       reinterpret_cast<cudaStream_t>(stream)),
                     "cpattn_block_gate launch");
}

cpattn_status cpattn_dsa_indexer(const cpattn_attn_args* a, const float* w, int32_t topk,
                                 int32_t* indices, void* workspace, size_t workspace_bytes,
                                 void* stream) {
  TRY(check_attn(a, false, false));
  CHECK(a->dtype == CPATTN_FP32, CPATTN_ERR_UNSUPPORTED, "the indexer takes CPATTN_FP32 qI and kI");
  CHECK(a->Hkv == 1, CPATTN_ERR_INVALID_ARG, "the indexer's keys have one head (Hkv=%d)", a->Hkv);
  CHECK(a->Hq <= 16, CPATTN_ERR_UNSUPPORTED, "Hq=%d indexer heads exceed 16", a->Hq);
  CHECK(a->Dqk <= 256, CPATTN_ERR_UNSUPPORTED, "Dqk=%d exceeds 256", a->Dqk);
  CHECK(a->kv_chunk_map == nullptr, CPATTN_ERR_UNSUPPORTED,
        "the indexer takes keys in logical order (kv_chunk_map NULL)");
  CHECK(topk >= 1 && (a->Tk == 0 || topk <= a->Tk), CPATTN_ERR_INVALID_ARG,
        "topk=%d must be in [1, Tk=%d]", topk, a->Tk);
  CHECK(w != nullptr, CPATTN_ERR_INVALID_ARG, "w is NULL");
  if (a->Tq > 0) CHECK(indices != nullptr, CPATTN_ERR_INVALID_ARG, "indices is NULL");
  const size_t need = a->Tq > 0 ? dsa_indexer_workspace(*a, dsa_indexer_grid(*a)) : 0;
  CHECK(workspace_bytes >= need && (need == 0 || workspace != nullptr), CPATTN_ERR_WORKSPACE,
        "workspace of %zu bytes given, %zu needed", workspace_bytes, need);
  if (need > 0) CHECK(aligned16(workspace), CPATTN_ERR_INVALID_ARG, "workspace is not 16-byte aligned");
  return cuda_status(launch_dsa_indexer(*a, w, topk, indices, workspace,
                                        reinterpret_cast<cudaStream_t>(stream)),
                     "cpattn_dsa_indexer launch");
}

cpattn_status cpattn_chunk_bwd(const cpattn_attn_args* a, const void* d_out, int64_t do_stride_t,
                               int64_t do_stride_h, float* dq, int64_t dq_stride_t,
                               int64_t dq_stride_h, float* dk, int64_t dk_stride_t,
                               int64_t dk_stride_h, float* dv, int64_t dv_stride_t,
                               int64_t dv_stride_h, void* workspace, size_t workspace_bytes,
                               void* stream) {
  TRY(check_attn(a, true, true));
  CHECK(a->dtype == CPATTN_BF16 && a->Dqk == 128 && a->Dv == 128, CPATTN_ERR_UNSUPPORTED,
        "the backward takes bf16 q, k, v with head dims 128 (Dqk=%d, Dv=%d)", a->Dqk, a->Dv);
  CHECK(a->kv_chunk_len == 0, CPATTN_ERR_INVALID_ARG, "the backward takes kv_chunk_len = 0");
  CHECK(dense_bwd_supported(*a), CPATTN_ERR_UNSUPPORTED,
        "layout not supported by the backward (chunk_len a multiple of 128, positions < 2^31)");
  if (a->Tq > 0) {
    CHECK(a->lse != nullptr, CPATTN_ERR_INVALID_ARG, "lse (the forward's) is NULL");
    TRY(check_tensor("d_out", d_out, do_stride_t, do_stride_h, a->Tq, 2));
    TRY(check_tensor("dq", dq, dq_stride_t, dq_stride_h, a->Tq, 4));
  }
  if (a->Tk > 0) {
    TRY(check_tensor("dk", dk, dk_stride_t, dk_stride_h, a->Tk, 4));
    TRY(check_tensor("dv", dv, dv_stride_t, dv_stride_h, a->Tk, 4));
  }
  if (a->Tq == 0 && a->Tk == 0) return ok();
  const size_t need = a->Tq > 0 ? dense_bwd_workspace(*a) : 0;
  CHECK(workspace_bytes >= need && (need == 0 || workspace != nullptr), CPATTN_ERR_WORKSPACE,
        "workspace of %zu bytes given, %zu needed", workspace_bytes, need);
  if (need > 0) CHECK(aligned16(workspace), CPATTN_ERR_INVALID_ARG, "workspace is not 16-byte aligned");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (a->Tq == 0 || a->Tk == 0) {   // no pair: every gradient is zero
    for (int64_t t = 0; t < a->Tq; ++t)   // rows may be strided: clear row by row
      if (cudaMemsetAsync(dq + t * dq_stride_t, 0, (size_t)((a->Hq - 1) * dq_stride_h + 128) * 4, st) != cudaSuccess)
        return fail(CPATTN_ERR_CUDA, "cudaMemsetAsync failed");
    for (int64_t t = 0; t < a->Tk; ++t) {
      if (cudaMemsetAsync(dk + t * dk_stride_t, 0, (size_t)((a->Hkv - 1) * dk_stride_h + 128) * 4, st) != cudaSuccess ||
          cudaMemsetAsync(dv + t * dv_stride_t, 0, (size_t)((a->Hkv - 1) * dv_stride_h + 128) * 4, st) != cudaSuccess)
        return fail(CPATTN_ERR_CUDA, "cudaMemsetAsync failed");
    }
    return ok();
  }
  return cuda_status(launch_dense_bwd(*a, d_out, do_stride_t, do_stride_h, dq, dq_stride_t,
                                      dq_stride_h, dk, dk_stride_t, dk_stride_h, dv, dv_stride_t,
                                      dv_stride_h, workspace, st),
                     "cpattn_chunk_bwd launch");
}

cpattn_status cpattn_mla_v_up(const void* o_latent, int64_t o_stride_t, int64_t o_stride_h,
                              const void* up_v_weight, int32_t T, int32_t H, int32_t L, int32_t V,
                              void* out, int64_t out_stride_t, int64_t out_stride_h,
                              int32_t* dev_status, int64_t wait_limit_ns, void* stream) {
  CHECK(T >= 0 && H >= 1, CPATTN_ERR_INVALID_ARG, "T=%d must be >= 0 and H=%d >= 1", T, H);
  CHECK(L >= 64 && L % 64 == 0, CPATTN_ERR_UNSUPPORTED, "L=%d must be a positive multiple of 64", L);
  CHECK(V >= 128 && V % 128 == 0, CPATTN_ERR_UNSUPPORTED, "V=%d must be a positive multiple of 128", V);
  CHECK(wait_limit_ns >= 0, CPATTN_ERR_INVALID_ARG, "wait_limit_ns must be >= 0");
  if (T == 0) return ok();
  TRY(check_tensor("o_latent", o_latent, o_stride_t, o_stride_h, T, 2));
  TRY(check_tensor("out", out, out_stride_t, out_stride_h, T, 2));
  CHECK(up_v_weight != nullptr && aligned16(up_v_weight), CPATTN_ERR_INVALID_ARG,
        "up_v_weight is NULL or not 16-byte aligned");
  const cpattn_status st = mla_v_up_impl(o_latent, o_stride_t, o_stride_h, up_v_weight, T, H, L, V,
                                         out, out_stride_t, out_stride_h, dev_status, wait_limit_ns,
                                         reinterpret_cast<cudaStream_t>(stream));
  return st == CPATTN_OK ? ok() : st;
}

cpattn_status cpattn_mla_kv_materialise(const void* kv_c, int64_t c_stride_t, const void* k_shared,
                                        int64_t ks_stride_t, const void* wkv_b, int32_t T, int32_t L,
                                        int32_t H, int32_t N, int32_t R, int32_t V, void* k_out,
                                        int64_t k_stride_t, int64_t k_stride_h, void* v_out,
                                        int64_t v_stride_t, int64_t v_stride_h, int32_t* dev_status,
                                        int64_t wait_limit_ns, void* stream) {
  CHECK(T >= 0 && H >= 1, CPATTN_ERR_INVALID_ARG, "T=%d must be >= 0 and H=%d >= 1", T, H);
  CHECK(L >= 64 && L % 64 == 0, CPATTN_ERR_UNSUPPORTED, "L=%d must be a positive multiple of 64", L);
  CHECK(N >= 128 && N % 128 == 0 && V >= 128 && V % 128 == 0, CPATTN_ERR_UNSUPPORTED,
        "N=%d and V=%d must be positive multiples of 128", N, V);
  CHECK(R >= 0 && R % 8 == 0, CPATTN_ERR_UNSUPPORTED, "R=%d must be a multiple of 8", R);
  CHECK(wait_limit_ns >= 0, CPATTN_ERR_INVALID_ARG, "wait_limit_ns must be >= 0");
  CHECK((int64_t)H * (N + V) <= (int64_t)1 << 30, CPATTN_ERR_UNSUPPORTED, "H*(N+V) too large");
  if (T == 0) return ok();
  CHECK(kv_c != nullptr && aligned16(kv_c) && c_stride_t >= L && c_stride_t % 8 == 0,
        CPATTN_ERR_INVALID_ARG, "kv_c must be 16-byte aligned with a row stride >= L, a multiple of 8");
  CHECK(wkv_b != nullptr && aligned16(wkv_b), CPATTN_ERR_INVALID_ARG, "wkv_b is NULL or not 16-byte aligned");
  if (R > 0)
    CHECK(k_shared != nullptr && aligned16(k_shared) && ks_stride_t >= R && ks_stride_t % 8 == 0,
          CPATTN_ERR_INVALID_ARG, "k_shared must be 16-byte aligned with a row stride >= R, a multiple of 8");
  TRY(check_tensor("k_out", k_out, k_stride_t, k_stride_h, T, 2));
  TRY(check_tensor("v_out", v_out, v_stride_t, v_stride_h, T, 2));
  const cpattn_status st = mla_kv_impl(kv_c, c_stride_t, k_shared, ks_stride_t, wkv_b, T, L, H, N,
                                       R, V, k_out, k_stride_t, k_stride_h, v_out, v_stride_t,
                                       v_stride_h, dev_status, wait_limit_ns,
                                       reinterpret_cast<cudaStream_t>(stream));
  return st == CPATTN_OK ? ok() : st;
}

size_t cpattn_workspace_size(int32_t op, const cpattn_attn_args* a, int32_t topk, int32_t block_size) {
  if (a == nullptr) return 0;
  if (op == CPATTN_OP_BLOCK_GATE) return block_size > 0 ? block_gate_workspace(*a, block_size) : 0;
  if (op == CPATTN_OP_DSA_INDEXER) return a->Tq > 0 ? dsa_indexer_workspace(*a, dsa_indexer_grid(*a)) : 0;
  if (op == CPATTN_OP_CHUNK_FWD) return a->kv_chunk_len == 0 ? dense_tc_bal_workspace(*a) : 0;
  if (op == CPATTN_OP_CHUNK_BWD) return a->Tq > 0 ? dense_bwd_workspace(*a) : 0;
  if (op == CPATTN_OP_TOPK_SPARSE_FWD && block_size > 1 && topk > 0 &&
      moba_tc_supported(*a, 1, block_size, topk))
    return moba_tc_workspace(*a, topk, block_size);
  return 0;
}

const char* cpattn_last_error(void) { return g_last_error.c_str(); }

int32_t cpattn_version(void) { return CPATTN_VERSION; }

}  // extern "C"
