/*
 * cpattn.h - C ABI of the GB300 context-parallel chunk attention library
 * (libcpattn.so).  One GPU: forward, backward, and the MLA projections
 * around them.
 *
 * What it computes.  A local query chunk placed at a global token offset
 * attends to a gathered global KV sequence:
 *
 *   allowed(i, j) = seq(qpos_i) == seq(kpos_j)  and  (!causal or kpos_j <= qpos_i)
 *   s_ij = scale * <q_i, k_j>
 *   O_i  = sum_{allowed j} exp(s_ij - m_i) v_j / l_i,   LSE_i = m_i + ln l_i
 *
 * computed as per-KV-chunk summaries (m, l, z) merged by rescaling to the
 * larger max, dividing only at the end.  A chunk with no permitted key has the
 * neutral summary (m = -inf, l = 0, z = 0); a query with no permitted key gets
 * O = 0 and LSE = -inf.  Sources, by page and paragraph:
 *   "Context parallel attention: exchange keys and merge softmax globally",
 *     para 1-2 (global-position causal masks, packed-varlen boundaries, GQA),
 *     para 3 (chunk summary m, l, z and its merge), para 4 (neutral summary,
 *     no-key convention), para 5 (zigzag: logical order vs physical chunk).
 *   "[Feature-request] Context Parallel support for DSAttention", "Strategy:
 *     allgather CP mode" (local Q vs gathered KV, causal diagonal shifted by
 *     cp_rank * local_seq, top-k indices in global coordinates).
 *   "[1/2] Enable DSA CP, THD with absorbed MLA - #3674", sequence diagram
 *     (index mask + varlen bounds; QK scores -> top-k -> sparse gather) and
 *     Background (absorbed MLA: key row = [latent | rope], value = latent).
 *   "Question on Implementing Context Parallelism with MoBA Efficient
 *     Attention" (gating scores Q x K^T pick the top-k KV blocks).
 *
 * Conventions shared by every entry point.
 *   Layout: tensors are token-major [T, H, D]; the last dimension is
 *     contiguous; strides are in ELEMENTS; base pointers and every stride
 *     times the element size must be multiples of 16 bytes.
 *   Memory: every pointer is a DEVICE pointer owned by the caller.  The
 *     library never allocates or frees device memory.  Between calls it
 *     keeps per-device caches of kernel attributes and TMA descriptors
 *     (host memory, refreshed whenever a pointer, shape or stride changes)
 *     and one piece of device state: the fixed scratch array of
 *     cpattn_block_gate_static, shared by every call of that entry point.
 *   Execution: every call only enqueues work on `stream` (a cudaStream_t /
 *     CUstream handle; NULL = legacy default stream) and returns; nothing
 *     synchronises.
 *   Errors: the return value is a cpattn_status.  Arguments are validated on
 *     the host before anything is launched, so a rejected call launches
 *     nothing.  cpattn_last_error() gives a message for the calling thread.
 *     Data errors found on the device (an index out of range) are written to
 *     the optional `dev_status` word (set to CPATTN_ERR_BAD_INDEX, first
 *     error wins; the caller zeroes it and reads it after synchronising).
 *     No call traps, asserts or aborts.  The tensor-core kernels wait on
 *     their own pipeline barriers with a bounded wait (wait_limit_ns, 2 s by
 *     default); a wait that runs out makes the kernel drain its copies and
 *     MMAs in flight, release its tensor memory, write CPATTN_ERR_TIMEOUT to
 *     dev_status and return; later calls on the stream are unaffected.
 *   Dtypes: q, k, v and o are all CPATTN_BF16 (fp32 accumulation) or all
 *     CPATTN_FP32.  LSE, partials and scratch are fp32.
 */
#ifndef CPATTN_H
#define CPATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define CPATTN_VERSION 110  /* 1.1.0 */

typedef enum {
  CPATTN_OK = 0,
  CPATTN_ERR_INVALID_ARG = 1,  /* bad shape, stride, alignment, pointer or enum */
  CPATTN_ERR_UNSUPPORTED = 2,  /* valid but not implemented (e.g. head dim too large) */
  CPATTN_ERR_CUDA = 3,         /* a CUDA runtime/driver call failed; see last_error */
  CPATTN_ERR_WORKSPACE = 4,    /* workspace NULL or smaller than cpattn_workspace_size */
  CPATTN_ERR_TIMEOUT = 5,      /* device wait gave up (written to dev_status only) */
  CPATTN_ERR_BAD_INDEX = 6     /* index outside the key range (dev_status only) */
} cpattn_status;

enum { CPATTN_FP32 = 0, CPATTN_BF16 = 1 };

enum { CPATTN_OP_CHUNK_FWD = 0, CPATTN_OP_TOPK_SPARSE_FWD = 1, CPATTN_OP_BLOCK_GATE = 2,
       CPATTN_OP_DSA_INDEXER = 3, CPATTN_OP_CHUNK_BWD = 4 };

/*
 * Arguments of one attention call (shared by chunk_fwd, topk_sparse_fwd and
 * block_gate; fields an entry point does not use are ignored).
 *
 * Positions.  Query row t (0 <= t < Tq) has logical global position
 *   qpos_t = causal_offset + (q_chunk_map ? q_chunk_map[t / chunk_len] * chunk_len
 *                                            + t % chunk_len : t)
 * and KV row j (0 <= j < Tk, the physical row of the gathered buffer) has
 *   kpos_j = kv_chunk_map ? kv_chunk_map[j / chunk_len] * chunk_len + j % chunk_len : j.
 * Physical chunk c holds logical chunk map[c] (zigzag: rank r owns chunks r
 * and 2*cp-1-r).  With a kv_chunk_map, Tk = n_kv_chunks * chunk_len and the
 * map is a permutation of 0..n_kv_chunks-1.  causal_offset = cp_rank *
 * local_seq for a contiguous split ("allgather CP mode").
 *
 * Packed sequences.  cu_seqlens (device, int32[num_seqs + 1], non-decreasing)
 * splits the LOGICAL position stream; seq(p) = s with cu[s] <= p < cu[s+1].  A
 * position outside [cu[0], cu[num_seqs]) belongs to no sequence and attends
 * to nothing.  NULL = one sequence holding every position.  Device metadata
 * is not validated on the host: a malformed cu_seqlens or chunk map gives
 * unspecified values but never an out-of-bounds access.
 *
 * Partial summaries (chunk_fwd only).  kv_chunk_len > 0 also writes, for each
 * KV chunk c of physical rows [c*kv_chunk_len, (c+1)*kv_chunk_len),
 * n_parts = ceil(Tk / kv_chunk_len), the chunk's finalised summary:
 *   partial_o   fp32 [n_parts, Tq, Hq, Dv] contiguous: z_c / l_c (0 if neutral)
 *   partial_lse fp32 [n_parts, Tq, Hq] contiguous:  m_c + ln l_c (-inf if neutral)
 * and o / lse hold the merge of all chunks (cpattn_lse_merge semantics).
 * With kv_chunk_len > 0, o and lse may both be NULL: only the partial
 * summaries are written (a caller that merges them itself, e.g. after
 * exchanging them, skips the in-kernel merge).
 */
typedef struct cpattn_attn_args {
  int32_t dtype;                         /* CPATTN_BF16 or CPATTN_FP32 */
  const void* q;                         /* [Tq, Hq, Dqk] local query chunk */
  int64_t q_stride_t, q_stride_h;
  int32_t Tq, Hq, Dqk;
  const void* k;                         /* [Tk, Hkv, Dqk] gathered keys */
  int64_t k_stride_t, k_stride_h;
  int32_t Tk, Hkv;                       /* Hq % Hkv == 0; head h reads KV head h / (Hq/Hkv) */
  const void* v;                         /* [Tk, Hkv, Dv]; may alias k (absorbed MLA) */
  int64_t v_stride_t, v_stride_h;
  int32_t Dv;
  float scale;                           /* softmax scale applied to q.k */
  int32_t causal;                        /* 0 or 1 */
  int64_t causal_offset;                 /* >= 0 */
  const int32_t* cu_seqlens;             /* device int32[num_seqs+1] or NULL */
  int32_t num_seqs;
  const int32_t* q_chunk_map;            /* device int32[n_q_chunks] or NULL */
  const int32_t* kv_chunk_map;           /* device int32[n_kv_chunks] or NULL */
  int32_t chunk_len, n_q_chunks, n_kv_chunks;
  void* o;                               /* [Tq, Hq, Dv] output, dtype */
  int64_t o_stride_t, o_stride_h;
  float* lse;                            /* fp32 [Tq, Hq] contiguous (natural log), or NULL */
  int32_t kv_chunk_len;                  /* 0 = no partial summaries */
  float* partial_o;                      /* see above, or NULL */
  float* partial_lse;
  int32_t* dev_status;                   /* optional device int32 */
  int64_t wait_limit_ns;                 /* limit of each bounded device wait; 0 = 2 s */
} cpattn_attn_args;

/*
 * cpattn_chunk_fwd - dense CP-chunk attention forward.
 * Source: "Context parallel attention: exchange keys and merge softmax
 * globally" para 1-5; "[Feature-request] Context Parallel support for
 * DSAttention", allgather CP mode (causal_offset).
 * Computes o [Tq, Hq, Dv] and lse [Tq, Hq] (and the partial summaries when
 * kv_chunk_len > 0).  Workspace is optional: with at least
 * cpattn_workspace_size(CPATTN_OP_CHUNK_FWD, ...) bytes (device memory, no
 * initialisation needed, not touched by the host) the KV work of all query
 * blocks is spread evenly over the SMs and blocks cut between CTAs are
 * merged in the kernel; with NULL or fewer bytes every CTA takes whole
 * blocks.  The size is 0 (no workspace used) when the problem's 2-block
 * work units already fill more than 3/4 of the device's SMs.  Both give the same results up to fp32 summation order.  Calls
 * sharing one workspace must be ordered on a stream.
 * Limits: Dqk, Dv multiples of 8, Dqk <= 1024, Dv <= 512; chunk maps need
 * chunk_len > 0.
 */
cpattn_status cpattn_chunk_fwd(const cpattn_attn_args* args, void* workspace,
                               size_t workspace_bytes, void* stream);

/*
 * cpattn_chunk_bwd - gradients of cpattn_chunk_fwd for one query chunk.
 * Source: "Context parallel attention: exchange keys and merge softmax
 * globally" para 2 (backward returns and combines contributions to the
 * owners of K and V) and para 4 (backward intermediates are rebuilt with
 * matching reconstruction rules: here the probabilities come from the
 * forward's LSE).  With P[i, j] = exp(s_ij - LSE_i) on permitted pairs,
 * g = d_out and D_i = <g_i, o_i>:
 *   dv_j = sum_i P_ij g_i,  dS_ij = P_ij (<g_i, v_j> - D_i),
 *   dq_i = scale sum_j dS_ij k_j,  dk_j = scale sum_i dS_ij q_i,
 * dk, dv of a KV head summed over its query heads.  dk and dv cover every
 * gathered KV row and hold this chunk's contribution only; adding the
 * contributions of all chunks (a reduce-scatter to the owners) is the
 * caller's.
 * Inputs: args as given to the forward (q, k, v, positions, cu_seqlens,
 * chunk maps, scale, causal) plus its outputs o (bf16) and lse (fp32);
 * d_out bf16 [Tq, Hq, 128].  Outputs (overwritten, not accumulated): dq fp32
 * [Tq, Hq, 128], dk, dv fp32 [Tk, Hkv, 128], strides in elements.
 * Workspace: cpattn_workspace_size(CPATTN_OP_CHUNK_BWD, ...) bytes.
 * Limits: bf16, Dqk = Dv = 128, kv_chunk_len = 0, chunk maps with chunk_len
 * a multiple of 128, logical positions below 2^31.
 */
cpattn_status cpattn_chunk_bwd(const cpattn_attn_args* args, const void* d_out, int64_t do_stride_t,
                               int64_t do_stride_h, float* dq, int64_t dq_stride_t,
                               int64_t dq_stride_h, float* dk, int64_t dk_stride_t,
                               int64_t dk_stride_h, float* dv, int64_t dv_stride_t,
                               int64_t dv_stride_h, void* workspace, size_t workspace_bytes,
                               void* stream);

/*
 * cpattn_lse_merge - merge finalised per-chunk results into the global one.
 * Source: "Context parallel attention: exchange keys and merge softmax
 * globally" para 3 (rescale to the larger max, add, divide at the end) and
 * para 4 (parts with LSE = -inf are neutral; all neutral -> O = 0, LSE = -inf).
 * part_o fp32 [n_parts, Tq, H, Dv] and part_lse fp32 [n_parts, Tq, H], both
 * contiguous; writes o [Tq, H, Dv] (o_dtype, strides o_stride_t/h in
 * elements) and lse fp32 [Tq, H] contiguous (lse may be NULL).
 *   L = max_c LSE_c,  w_c = exp(LSE_c - L),  LSE = L + ln sum_c w_c,
 *   O = sum_c w_c O_c / sum_c w_c.
 * Limits: Dv a multiple of 8.
 */
cpattn_status cpattn_lse_merge(int32_t n_parts, const float* part_o, const float* part_lse,
                               int32_t Tq, int32_t H, int32_t Dv, void* o, int32_t o_dtype,
                               int64_t o_stride_t, int64_t o_stride_h, float* lse,
                               void* stream);

/*
 * cpattn_topk_sparse_fwd - attention of each query over selected keys only.
 * Source: "[Feature-request] Context Parallel support for DSAttention",
 * allgather CP mode and step 6 (iterate only over the top-k indices, never
 * materialise the score matrix); "[1/2] Enable DSA CP, THD with absorbed MLA
 * - #3674" sequence diagram (QK scores -> top-k -> sparse gather; index mask
 * and varlen bounds) and Background (absorbed MLA shapes, v aliasing k);
 * "Question on Implementing Context Parallelism with MoBA Efficient
 * Attention" (top-k blocks).
 * indices: device int32 [Tq, index_heads, topk] contiguous, index_heads = 1
 * (shared by every query head, DSA) or Hq (one list per head, MoBA).
 *   block_size == 1: each entry is a LOGICAL key position;
 *   block_size  > 1: each entry b names logical keys [b*B, min((b+1)*B, Tk)).
 * -1 marks an unused slot.  The permitted relation is applied again to every
 * selected key (causal + varlen), so a selection never widens attention.  An
 * entry < -1 or beyond the key range is skipped and sets dev_status to
 * CPATTN_ERR_BAD_INDEX.  A repeated entry counts once per occurrence.  No
 * selected permitted key -> O = 0, LSE = -inf.  kv_chunk_len must be 0.
 * Workspace: cpattn_workspace_size(CPATTN_OP_TOPK_SPARSE_FWD, ...) bytes.
 */
cpattn_status cpattn_topk_sparse_fwd(const cpattn_attn_args* args, const int32_t* indices,
                                     int32_t topk, int32_t index_heads, int32_t block_size,
                                     void* workspace, size_t workspace_bytes, void* stream);

/*
 * cpattn_block_gate - MoBA block selection for every (query, head).
 * Source: "Question on Implementing Context Parallelism with MoBA Efficient
 * Attention" (gating scores from Q x K^T choose the top-k KV blocks).  The
 * pooling and tie rule are this library's stated reading:
 *   mean_b = (1/B) sum of the keys of complete block b (per KV head);
 *   gate(i, h, b) = <q_ih, mean_b> (unscaled), over candidate blocks
 *   b < own(i) = qpos_i / B, i.e. blocks that end before the own block;
 *   the `topk` largest gates win, equal gates go to the lower b (all
 *   candidates if fewer); the own block is always added.
 * Output sel: device int32 [Tq, Hq, topk + 1] contiguous, ascending, padded
 * with -1 - directly usable as `indices` of cpattn_topk_sparse_fwd with
 * index_heads = Hq and block_size = B.  The selection equals the one an exact
 * (float64) evaluation of the gates makes: fp32 gates whose error bound
 * reaches the k-th boundary are re-ranked in fp64.
 * Uses args->dtype, q, k (strides, Tq, Hq, Dqk, Tk, Hkv), causal_offset and
 * q_chunk_map/chunk_len for qpos.  cu_seqlens and kv_chunk_map must be NULL.
 * Workspace: cpattn_workspace_size(CPATTN_OP_BLOCK_GATE, ...) bytes (block
 * means).  Limits: topk <= 64; the number of complete blocks Tk / B is
 * limited by the kernel's shared-memory staging (about 370 at Dqk = 128;
 * CPATTN_ERR_UNSUPPORTED beyond).
 */
cpattn_status cpattn_block_gate(const cpattn_attn_args* args, int32_t block_size, int32_t topk,
                                int32_t* sel, void* workspace, size_t workspace_bytes,
                                void* stream);

/*
 * cpattn_block_gate_static - cpattn_block_gate for callers that cannot
 * allocate device memory.  The pages have no counterpart; this is a
 * deployment convenience of this library.
 * Some callers cannot call cudaMalloc or grow a memory pool when they make
 * this call: a plugin handed only its input and output buffers, code running
 * inside a host callback, or a runtime that owns every allocation.  This
 * variant takes no workspace: the block means live in a fixed 16 MiB array
 * compiled into the library, which every GPU that loads the library holds
 * until the process exits.  Arguments, output and selection are those of
 * cpattn_block_gate, and so are the kernels it runs (those that
 * cpattn_block_gate runs with a workspace of cpattn_workspace_size bytes).
 * The call allocates nothing.
 * Limits and behaviour:
 *   - shapes whose workspace (cpattn_workspace_size(CPATTN_OP_BLOCK_GATE,
 *     ...)) exceeds 16 MiB are rejected with CPATTN_ERR_UNSUPPORTED and a
 *     message; nothing is launched;
 *   - the first call on a device, with that device current, looks up the
 *     array's device address (cudaGetSymbolAddress) and caches it; make that
 *     first call before any stream capture;
 *   - every call on a device shares the array and it keeps the last call's
 *     contents (each call rewrites all it reads, so nothing needs clearing);
 *     calls whose work overlaps on the GPU race - keep them in stream order.
 */
cpattn_status cpattn_block_gate_static(const cpattn_attn_args* args, int32_t block_size,
                                       int32_t topk, int32_t* sel, void* stream);

/*
 * cpattn_dsa_indexer - token selection of the DSA indexer for every query.
 * Source: "[1/2] Enable DSA CP, THD with absorbed MLA - #3674", sequence
 * diagram (index mask and varlen bounds, then the indexer's QK scores, then
 * top-k, then the sparse gather); "[Feature-request] Context Parallel
 * support for DSAttention" (indices in global coordinates).  The score is
 * this library's stated reading of the indexer:
 *   score(i, j) = sum_h w[h] * max(0, <qI[i, h], kI[j]>)
 * over the keys the layout permits (allowed(i, j) above).  The `topk` keys
 * with the largest score are chosen, equal scores going to the lower key; a
 * row with fewer permitted keys takes all of them.
 * Output indices: device int32 [Tq, topk] contiguous, each row ascending and
 * padded with -1 - directly usable as `indices` of cpattn_topk_sparse_fwd
 * with index_heads = 1 and block_size = 1.  The selection equals the one an
 * exact (float64) evaluation of the scores makes: the scores (fp32 fmas, or
 * for Dqk = 128 a split bf16 GEMM on the tensor cores) carry a certified
 * error bound, and only keys whose bound reaches the k-th boundary are
 * ranked again (first in fp32 under the tighter fp32 bound when the scores
 * came from the tensor cores, then in float64).
 * Uses args->dtype (CPATTN_FP32), q = qI [Tq, Hq, Dqk] (Hq = indexer heads),
 * k = kI [Tk, 1, Dqk] (Hkv = 1), causal, causal_offset, cu_seqlens and
 * q_chunk_map/chunk_len for positions; keys are in logical order
 * (kv_chunk_map NULL).  w: device fp32 [Hq].  Limits: Dqk <= 256, Hq <= 16,
 * 1 <= topk <= Tk.
 * Workspace: cpattn_workspace_size(CPATTN_OP_DSA_INDEXER, ...) bytes (the
 * fp32 scores of every query and permitted key, key norms, scratch and, for
 * Dqk = 128, the bf16 split operands).
 */
cpattn_status cpattn_dsa_indexer(const cpattn_attn_args* args, const float* w, int32_t topk,
                                 int32_t* indices, void* workspace, size_t workspace_bytes,
                                 void* stream);

/*
 * cpattn_mla_v_up - value up-projection after absorbed attention.
 * Source: "[1/2] Enable DSA CP, THD with absorbed MLA - #3674", sequence
 * diagram (after the sparse gather, an einsum with up_v_weight gives each
 * head's v_channels) and Background (the value up-projection is applied
 * after attention on the latent).
 *   out[t, h, :] = o_latent[t, h, :] @ up_v_weight[h]
 * o_latent: bf16 [T, H, L] (strides in elements, last dim contiguous), e.g.
 * the output of cpattn_topk_sparse_fwd on absorbed-MLA shapes; up_v_weight:
 * bf16 [H, L, V] contiguous; out: bf16 [T, H, V].  fp32 accumulation.
 * Limits: L a multiple of 64, V a multiple of 128.  No workspace.
 * wait_limit_ns: limit of each bounded device wait (0 = 2 s).
 */
cpattn_status cpattn_mla_v_up(const void* o_latent, int64_t o_stride_t, int64_t o_stride_h,
                              const void* up_v_weight, int32_t T, int32_t H, int32_t L, int32_t V,
                              void* out, int64_t out_stride_t, int64_t out_stride_h,
                              int32_t* dev_status, int64_t wait_limit_ns, void* stream);

/*
 * cpattn_mla_kv_materialise - per-head K and V from gathered MLA latents.
 * Source: "[BC][MLA][CP] Optimize MLA all-gather and Ulysses communication
 * for Kimi K3 and dpskV3", "K/V all-gather CP" (gather the compressed
 * latents and the head-shared key, then apply wkv_b and build K/V locally).
 *   kv = kv_c @ wkv_b^T viewed [T, H, N + V];
 *   k_out[t, h] = [kv[t, h, :N] | k_shared[t]],  v_out[t, h] = kv[t, h, N:]
 * kv_c: bf16 [T, L] (row stride c_stride_t); k_shared: bf16 [T, R] (row
 * stride ks_stride_t; unused when R = 0); wkv_b: bf16 [H * (N + V), L]
 * contiguous (a linear layer's weight); k_out: bf16 [T, H, N + R]; v_out:
 * bf16 [T, H, V].  fp32 accumulation.  Limits: L a multiple of 64, N and V
 * multiples of 128, R a multiple of 8.  No workspace.
 */
cpattn_status cpattn_mla_kv_materialise(const void* kv_c, int64_t c_stride_t, const void* k_shared,
                                        int64_t ks_stride_t, const void* wkv_b, int32_t T, int32_t L,
                                        int32_t H, int32_t N, int32_t R, int32_t V, void* k_out,
                                        int64_t k_stride_t, int64_t k_stride_h, void* v_out,
                                        int64_t v_stride_t, int64_t v_stride_h, int32_t* dev_status,
                                        int64_t wait_limit_ns, void* stream);

/* Bytes of device workspace the call needs (0 if none; for
 * CPATTN_OP_CHUNK_FWD the bytes that enable the SM-balanced schedule).
 * `args` supplies the shapes; topk and block_size as passed to the call. */
size_t cpattn_workspace_size(int32_t op, const cpattn_attn_args* args, int32_t topk,
                             int32_t block_size);

/* Message describing the last failed call on this thread ("" if none). */
const char* cpattn_last_error(void);

/* CPATTN_VERSION of the loaded library. */
int32_t cpattn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* CPATTN_H */
