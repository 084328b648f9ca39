"""GPU parity: every entry point through the C ABI against the float64 oracle.

Small cases span several tiles with ragged tails and are compared element by
element on every output; the full-size workloads run in the launch
configuration the bench times and are compared on sampled rows (all heads,
all channels of each sampled row).  Block selections are compared bit-exactly.
"""

import numpy as np
import pytest
import torch

import oracle as orc
import context_attention_softmax_gb300 as pkg
from context_attention_softmax_gb300 import (cpattn_block_gate, cpattn_chunk_fwd, cpattn_dsa_indexer,
                                             cpattn_lse_merge, cpattn_topk_sparse_fwd, inputs)

from helpers import assert_matches, f64, layout_of, sample_rows, to_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from context_attention_softmax_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def _chunk(w, **kw):
    q, k, v = to_gpu(w)
    return cpattn_chunk_fwd(q, k, v, scale=w.scale, causal=w.causal, causal_offset=w.causal_offset,
                            cu_seqlens=w.cu_seqlens, q_chunk_map=w.q_chunk_map,
                            kv_chunk_map=w.kv_chunk_map, chunk_len=w.chunk_len, **kw)


# ---------------------------------------------------------------------------
# dense chunk attention
# ---------------------------------------------------------------------------

def test_tiny_fp32_two_summaries_then_merge():
    w = inputs.tiny_fp32()
    o, lse, po, pl = _chunk(w, kv_chunk_len=w.kv_chunk_len)
    q, k, v = f64(w)
    O, L, PO, PL = orc.summarised_attention(q, k, v, w.scale, layout_of(w), w.kv_chunk_len)
    assert_matches(o, lse, O, L, "fp32", "final")
    for c in range(2):
        assert_matches(po[c], pl[c], PO[c], PL[c], "fp32", f"summary {c}")
    om, lm = cpattn_lse_merge(po, pl, out_dtype=torch.float32)
    assert_matches(om, lm, O, L, "fp32", "lse_merge")
    o2, l2 = _chunk(w)
    assert_matches(o2, l2, O, L, "fp32", "single pass")


@pytest.mark.parametrize("Tq,Tk,off,Hq,Hkv,kvc", [
    (300, 1000, 700, 4, 2, 256),     # ragged tails on both sides
    (257, 1300, 700, 4, 1, 256),     # keys 1000.. never permitted: chunk 4 is neutral
    (128, 640, 0, 2, 2, 0),          # offset 0: the first query sees one key
    (300, 1000, 700, 4, 2, 0),       # single pass (tensor-core path), ragged tails
    (257, 1300, 700, 4, 1, 0),
    (1, 129, 128, 1, 1, 0),          # one query, one key past a tile edge
    (128, 8192, 8064, 2, 2, 0),      # two long units over far more CTAs than tiles each
    (600, 3000, 2500, 8, 2, 0),      # head pairs, units cut across several CTAs
    (300, 1000, 700, 4, 2, 200),     # chunks not a multiple of 128: the row kernel
    (1000, 1100, 300, 2, 1, 128),    # one-tile chunks, folded pairs and their tail
    (640, 4096, 3000, 4, 2, 1024),   # chunks of 8 tiles; chunk 3 reached by few rows
])
def test_dense_gqa_small(Tq, Tk, off, Hq, Hkv, kvc):
    rng_w = inputs.dense_gqa(seed=1, global_seq=Tq, cp_size=1, rank=0, Hq=Hq, Hkv=Hkv, Tk=Tk,
                             kv_chunks=0)
    rng_w.causal_offset = off
    w = rng_w
    q, k, v = f64(w)
    O, L, PO, PL = orc.summarised_attention(q, k, v, w.scale, layout_of(w), kvc or Tk)
    if kvc:
        o, lse, po, pl = _chunk(w, kv_chunk_len=kvc)
        for c in range(po.shape[0]):
            assert_matches(po[c], pl[c], PO[c], PL[c], "bf16", f"summary {c}")
        if Tk == 1300:
            assert torch.isneginf(pl[4]).all() and (po[4] == 0).all()
    else:
        o, lse = _chunk(w)
    assert_matches(o, lse, O, L, "bf16", "final")


def test_dense_gqa_full_size_every_row():
    """The headline workload in the bench's launch configuration: every row,
    head and channel against the oracle; then the four-chunk summary form,
    whose per-chunk summaries are checked on sampled rows and merged by
    cpattn_lse_merge."""
    w = inputs.dense_gqa()
    o, lse = _chunk(w, workspace=torch.empty(64 << 20, dtype=torch.uint8, device="cuda"))
    q, k, v = f64(w)
    O, L = orc.dense_attention(q, k, v, w.scale, layout_of(w))
    assert_matches(o, lse, O, L, "bf16", "cfg full")
    o4, l4, po, pl = _chunk(w, kv_chunk_len=w.kv_chunk_len)
    assert torch.isneginf(pl[3]).all()          # chunk 3 (keys 6144..) is fully masked
    assert_matches(o4, l4, O, L, "bf16", "cfg 4 chunks")
    om, lm = cpattn_lse_merge(po, pl, out_dtype=torch.bfloat16)
    assert_matches(om, lm, O, L, "bf16", "cfg 4 chunks merged")
    # partial summaries only (o = lse = NULL), then the merge: the bench's step
    none_o, none_l, po2, pl2 = _chunk(w, kv_chunk_len=w.kv_chunk_len, merged=False)
    assert none_o is None and none_l is None
    assert torch.equal(po2, po) and torch.equal(pl2, pl)
    rows = sample_rows(w.Tq, 64, edges=(1, 127, 128, 1023, 2047))
    _, _, PO, PL = orc.summarised_attention(q, k, v, w.scale, layout_of(w), w.kv_chunk_len,
                                            rows=rows)
    for c in range(po.shape[0]):
        assert_matches(po[c][rows.tolist()], pl[c][rows.tolist()], PO[c], PL[c], "bf16",
                       f"cfg chunk {c}")


@pytest.mark.parametrize("factor", [3.0, 8.0])
def test_dense_large_logits_rescale(factor):
    # Q and K scaled: a score spread of tens of units, so a row's running max
    # grows by more than 2^8 between tiles and the accumulator is rescaled
    # mid-row.  V stays N(0, 1) so the bf16 output bound keeps its meaning.
    w = inputs.dense_gqa(seed=9, global_seq=512, cp_size=2, rank=1, Hq=2, Hkv=1, Tk=1536,
                         factor=factor, kv_chunks=0, v_factor=1.0)
    q, k, v = f64(w)
    O, L = orc.dense_attention(q, k, v, w.scale, layout_of(w))
    o, lse = _chunk(w)
    assert_matches(o, lse, O, L, "bf16", f"factor {factor}")


def test_noncausal_and_queries_outside_sequences():
    w = inputs.dense_gqa(seed=3, global_seq=200, cp_size=1, rank=0, Hq=2, Hkv=2, Tk=333, kv_chunks=0)
    w.causal = False
    w.causal_offset = 150
    w.cu_seqlens = np.array([0, 100, 160, 290], dtype=np.int32)   # positions >= 290 in no sequence
    q, k, v = f64(w)
    O, L = orc.dense_attention(q, k, v, w.scale, layout_of(w))
    assert np.isneginf(L[140:]).all()
    o, lse = _chunk(w)
    assert_matches(o, lse, O, L, "bf16", "non-causal varlen")


def test_empty_inputs():
    d = torch.device("cuda")
    q = torch.randn(0, 4, 128, device=d, dtype=torch.bfloat16)
    k = torch.randn(64, 2, 128, device=d, dtype=torch.bfloat16)
    o, lse = cpattn_chunk_fwd(q, k, k, causal_offset=3)
    assert o.shape == (0, 4, 128)
    q = torch.randn(16, 4, 128, device=d, dtype=torch.bfloat16)
    k0 = torch.randn(0, 2, 128, device=d, dtype=torch.bfloat16)
    o, lse = cpattn_chunk_fwd(q, k0, k0)
    torch.cuda.synchronize()
    assert (o == 0).all() and torch.isneginf(lse).all()
    o, lse, po, pl = cpattn_chunk_fwd(q, k0, k0, kv_chunk_len=32)
    assert po.shape[0] == 0 and (o == 0).all() and torch.isneginf(lse).all()


# ---------------------------------------------------------------------------
# packed THD varlen + zigzag
# ---------------------------------------------------------------------------

def _zigzag_check(z, rows_per_rank=None, all_rows_ranks=()):
    qg, kg, vg = (inputs.as_f64(t) for t in (z.q_global, z.k_global, z.v_global))
    lay_full = orc.make_layout(qg.shape[0], qg.shape[0], True, 0, z.cu_seqlens)
    L = z.chunk_len
    for r in range(z.cp_size):
        w = z.rank_workload(r)
        o, lse = _chunk(w)
        if rows_per_rank is None or r in all_rows_ranks:
            rows = np.arange(w.Tq)
        else:
            rows = sample_rows(w.Tq, rows_per_rank, seed=r, edges=(L - 1, L, 2 * L - 1))
        logical = np.concatenate([np.arange(c * L, (c + 1) * L) for c in z.rank_chunks(r)])[rows]
        # the oracle's full logical run, rows scattered back by ownership
        O, LSE = orc.dense_attention(qg, kg, vg, z.scale, lay_full, rows=logical)
        assert_matches(o[rows.tolist()], lse[rows.tolist()], O, LSE, "bf16", f"rank {r}")
        # and the oracle on the rank's own physical layout agrees too
        if rows_per_rank is None and r == 0:
            q, k, v = f64(w)
            O2, L2 = orc.dense_attention(q, k, v, w.scale, layout_of(w), rows=rows)
            assert_matches(o, lse, O2, L2, "bf16", "rank 0 physical")


def test_zigzag_partial_summaries_per_physical_chunk():
    """Per-KV-chunk summaries under packed sequences and a zigzag chunk map:
    each partial covers physical rows [c*L, (c+1)*L) of the gathered buffer
    (what one peer contributes), on the tensor-core kernel."""
    z = inputs.zigzag_varlen(seed=4, total=4096, n_seqs=3, len_lo=256, len_hi=2048, cp_size=4, H=4)
    for r in (0, 3):
        w = z.rank_workload(r)
        o, lse, po, pl = _chunk(w, kv_chunk_len=z.chunk_len)
        q, k, v = f64(w)
        O, L, PO, PL = orc.summarised_attention(q, k, v, w.scale, layout_of(w), z.chunk_len)
        assert_matches(o, lse, O, L, "bf16", f"rank {r} final")
        for c in range(po.shape[0]):
            assert_matches(po[c], pl[c], PO[c], PL[c], "bf16", f"rank {r} chunk {c}")


def test_zigzag_varlen_small():
    z = inputs.zigzag_varlen(seed=2, total=2048, n_seqs=4, len_lo=128, len_hi=1024, cp_size=4, H=4)
    _zigzag_check(z)


def _chunk_without_workspace(w):
    """cpattn_chunk_fwd through the C ABI with no workspace: one unit per CTA."""
    import ctypes
    from context_attention_softmax_gb300 import _lib
    q, k, v = to_gpu(w)
    dev = q.device
    cu, qm, km = (pkg._device_i32(x, dev) for x in (w.cu_seqlens, w.q_chunk_map, w.kv_chunk_map))
    o = torch.empty((q.shape[0], q.shape[1], v.shape[2]), dtype=q.dtype, device=dev)
    lse = torch.empty((q.shape[0], q.shape[1]), dtype=torch.float32, device=dev)
    a = pkg._args(q, k, v, w.scale, w.causal, w.causal_offset, cu, qm, km, w.chunk_len, o, lse)
    _lib.check(_lib.load().cpattn_chunk_fwd(ctypes.byref(a), None, 0,
                                            torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    return o, lse


def test_zigzag_schedules_agree():
    """Chunk maps: the SM-balanced schedule and one unit per CTA both match."""
    z = inputs.zigzag_varlen(seed=5, total=4096, n_seqs=3, len_lo=256, len_hi=2048, cp_size=4, H=6)
    w = z.rank_workload(1)
    q, k, v = f64(w)
    O, L = orc.dense_attention(q, k, v, w.scale, layout_of(w))
    o1, l1 = _chunk(w)
    o2, l2 = _chunk_without_workspace(w)
    assert_matches(o1, l1, O, L, "bf16", "balanced")
    assert_matches(o2, l2, O, L, "bf16", "per unit")


def test_zigzag_varlen_full_size():
    """All 8 rank calls of the packed zigzag workload: every row of ranks 0
    and 7 (the earliest and the latest chunk pairs), 64 sampled rows of the
    others."""
    z = inputs.zigzag_varlen()
    _zigzag_check(z, rows_per_rank=64, all_rows_ranks=(0, 7))


def test_zigzag_rank_calls_concurrent_on_separate_streams():
    """The 8 rank calls of the full-size zigzag workload issued on 8 streams at
    once (as the bench issues them) give bit-for-bit the outputs of the same
    calls issued one after another, and 32 sampled rows of each rank match
    the oracle: no call shares device state with another."""
    z = inputs.zigzag_varlen()
    dev = torch.device("cuda")
    k, v = z.k_gathered.to(dev), z.v_gathered.to(dev)
    qs = [z.rank_q(r).to(dev) for r in range(z.cp_size)]

    def run(r, out, lse, stream=None):
        cpattn_chunk_fwd(qs[r], k, v, scale=z.scale, causal=True, cu_seqlens=z.cu_seqlens,
                         q_chunk_map=z.rank_chunks(r), kv_chunk_map=z.kv_chunk_map,
                         chunk_len=z.chunk_len, out=out, lse=lse, stream=stream)

    seq = [(torch.empty_like(q), torch.empty(q.shape[:2], dtype=torch.float32, device=dev))
           for q in qs]
    for r in range(z.cp_size):
        run(r, *seq[r])
    torch.cuda.synchronize()
    par = [(torch.full_like(q, float("nan")),
            torch.full(q.shape[:2], float("nan"), dtype=torch.float32, device=dev)) for q in qs]
    streams = [torch.cuda.Stream(dev) for _ in range(z.cp_size)]
    main = torch.cuda.current_stream()
    start = torch.cuda.Event()
    start.record(main)
    for rep in range(3):
        for r in range(z.cp_size):
            streams[r].wait_event(start)
            run(r, *par[r], stream=streams[r])
    for st in streams:
        main.wait_stream(st)
    torch.cuda.synchronize()
    for r in range(z.cp_size):
        assert torch.equal(par[r][0], seq[r][0]), f"rank {r}: O differs from the sequential call"
        assert torch.equal(par[r][1], seq[r][1]), f"rank {r}: LSE differs from the sequential call"
    T = z.q_global.shape[0]
    lay = orc.make_layout(T, T, True, 0, z.cu_seqlens)
    qg, kg, vg = (inputs.as_f64(t) for t in (z.q_global, z.k_global, z.v_global))
    L = z.chunk_len
    rng = np.random.default_rng(11)
    for r in range(z.cp_size):
        local = np.sort(rng.choice(qs[r].shape[0], size=32, replace=False))
        c = np.asarray(z.rank_chunks(r))[local // L]
        logical = c * L + local % L
        O, LSE = orc.dense_attention(qg, kg, vg, z.scale, lay, rows=logical)
        o, lse = par[r]
        assert_matches(o[local.tolist()], lse[local.tolist()], O, LSE, "bf16", f"rank {r} streams")


# ---------------------------------------------------------------------------
# DSA top-k token indices (absorbed MLA: v aliases the first 512 channels of k)
# ---------------------------------------------------------------------------

def _dsa_run(w, dev_status=None):
    q, k, v = to_gpu(w)
    return cpattn_topk_sparse_fwd(q, k, v, w.indices, block_size=1, scale=w.scale,
                                  causal_offset=w.causal_offset, dev_status=dev_status)


def test_dsa_small_with_padding_and_bad_indices():
    w = inputs.dsa_absorbed(seed=4, Tq=70, Tk=2100, offset=1000, Hq=16, topk=256)
    idx = w.indices.clone()
    idx[3, 0, 100:] = -1                 # fewer than topk selected
    idx[5, 0, :] = -1                    # nothing selected -> (0, -inf)
    idx[7, 0, 10] = 5000                 # out of range: skipped, flagged
    idx[8, 0, 11] = idx[8, 0, 12]        # duplicate counts twice
    idx[9, 0, 20] = 2050                 # in range but after the query: masked again
    w.indices = idx
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, lse = _dsa_run(w, status)
    q, k, v = f64(w)
    O, L, bad = orc.sparse_attention(q, k, v, w.scale, layout_of(w), idx.numpy())
    assert bad == 1
    assert int(status.item()) == 6       # CPATTN_ERR_BAD_INDEX
    assert_matches(o, lse, O, L, "bf16", "dsa small")


def test_dsa_tensor_core_small():
    # 128 heads over one KV head, v = first 512 channels of k: the tensor-core
    # path; top-k 200 leaves a ragged last tile of 64 keys
    w = inputs.dsa_absorbed(seed=10, Tq=24, Tk=3000, offset=1500, Hq=128, topk=200)
    idx = w.indices.clone()
    idx[2, 0, 150:] = -1                 # fewer than topk selected
    idx[4, 0, :] = -1                    # nothing selected -> (0, -inf)
    idx[6, 0, 7] = 4000                  # out of range: skipped, flagged
    idx[8, 0, 11] = idx[8, 0, 12]        # duplicate counts twice
    idx[9, 0, 20] = 2999                 # in range but after the query: masked again
    w.indices = idx
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, lse = _dsa_run(w, status)
    q, k, v = f64(w)
    O, L, bad = orc.sparse_attention(q, k, v, w.scale, layout_of(w), idx.numpy())
    assert bad == 1 and int(status.item()) == 6
    assert_matches(o, lse, O, L, "bf16", "dsa tensor-core small")


def test_dsa_full_size_sampled():
    """The DSA workload: rows 0..79 (their two items are the first items of
    every persistent CTA, one CTA per SM) plus 200 random rows and the last."""
    w = inputs.dsa_absorbed(device="cuda")
    o, lse = _dsa_run(w)
    rows = np.union1d(np.arange(80), sample_rows(w.Tq, 200, edges=(4095,)))
    assert len(rows) >= 256
    q, k, v = f64(w)
    O, L, _ = orc.sparse_attention(q, k, v, w.scale, layout_of(w), w.indices.numpy(), rows=rows)
    assert_matches(o[rows.tolist()], lse[rows.tolist()], O, L, "bf16", "dsa full")


def _dsa_layout_case(seed, Tq, Tk, topk, qpos, cu=None):
    """Absorbed-MLA inputs (128 heads, 576 / 512) whose indices are a mix:
    rows chosen by the float64 indexer under the packed layout (within the
    query's sequence) and rows chosen ignoring the packing (so they name keys
    of other sequences, which the kernel must mask again).

    Some rows attend to one or two keys, so O is close to a single value row.
    KV is N(0, 1) * 0.25 so that |O| stays below 2: a bf16 output of
    magnitude in [2, 4) already carries up to 2^-8 of rounding and one in
    [4, 8) up to 2^-7, beyond the 1e-2 bound that the workloads (outputs
    averaged over thousands of keys, |O| << 1) are held to."""
    rng = np.random.default_rng(seed)
    q = inputs.to_device_dtype((rng.standard_normal((Tq, 128, 576))).astype(np.float32), "bf16")
    kv = inputs.to_device_dtype((rng.standard_normal((Tk, 1, 576)) * 0.25).astype(np.float32),
                                "bf16")
    qI = rng.standard_normal((Tq, 2, 32))
    kI = rng.standard_normal((Tk, 32))
    wI = rng.uniform(0.0, 1.0, 2)
    lay_seq = orc.Layout(np.asarray(qpos, np.int64), np.arange(Tk, dtype=np.int64),
                         orc.sequence_index(qpos, cu), orc.sequence_index(np.arange(Tk), cu),
                         True, cu)
    lay_one = orc.Layout(np.asarray(qpos, np.int64), np.arange(Tk, dtype=np.int64),
                         np.zeros(Tq, np.int64), np.zeros(Tk, np.int64), True, None)
    packed = orc.dsa_indexer_topk(qI, kI, wI, lay_seq, topk)
    crossing = orc.dsa_indexer_topk(qI, kI, wI, lay_one, topk)
    idx = np.where((np.arange(Tq) % 2 == 0)[:, None, None], packed, crossing)
    return q, kv, torch.from_numpy(idx.astype(np.int32))


def test_dsa_tensor_core_packed_sequences():
    """Packed THD sequences on the tensor-core DSA kernel: sequence ends fall
    inside 64-key tiles and inside the index lists; odd rows name keys of
    earlier sequences, which the kernel masks again; query rows past the last
    sequence select nothing; rows just after a sequence start see one or two
    keys."""
    Tq, Tk, topk, off = 40, 2600, 300, 2300
    cu = np.array([0, 1000, 2301, 2333, 2335], dtype=np.int32)
    qpos = off + np.arange(Tq)
    q, kv, idx = _dsa_layout_case(41, Tq, Tk, topk, qpos, cu)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    qd, kd = q.cuda(), kv.cuda()
    o, lse = cpattn_topk_sparse_fwd(qd, kd, kd[:, :, :512], idx, block_size=1,
                                    scale=1 / np.sqrt(576), causal_offset=off,
                                    cu_seqlens=torch.from_numpy(cu), dev_status=status)
    lay = orc.make_layout(Tq, Tk, True, off, cu_seqlens=cu)
    qf, kf = inputs.as_f64(q), inputs.as_f64(kv)
    O, L, bad = orc.sparse_attention(qf, kf, kf[:, :, :512], 1 / np.sqrt(576), lay, idx.numpy())
    assert bad == 0 and int(status.item()) == 0
    assert np.isneginf(L[qpos >= 2335]).all() and np.isfinite(L[qpos < 2335]).any(axis=1).sum() > 20
    assert_matches(o, lse, O, L, "bf16", "dsa tensor-core packed")


def test_dsa_tensor_core_query_chunk_map():
    """A zigzag query chunk map on the tensor-core DSA kernel: local rows
    0..47 hold logical chunk 1 and rows 48..95 logical chunk 6 (chunks of
    48); the indices were chosen for those logical positions."""
    L, Tk, topk = 48, 340, 200
    cmap = np.array([1, 6], dtype=np.int32)
    qpos = np.concatenate([np.arange(c * L, (c + 1) * L) for c in cmap])
    q, kv, idx = _dsa_layout_case(42, 2 * L, Tk, topk, qpos)
    qd, kd = q.cuda(), kv.cuda()
    o, lse = cpattn_topk_sparse_fwd(qd, kd, kd[:, :, :512], idx, block_size=1,
                                    scale=1 / np.sqrt(576), q_chunk_map=torch.from_numpy(cmap),
                                    chunk_len=L)
    lay = orc.make_layout(2 * L, Tk, True, 0, q_chunk_map=cmap, chunk_len=L)
    qf, kf = inputs.as_f64(q), inputs.as_f64(kv)
    O, LS, _ = orc.sparse_attention(qf, kf, kf[:, :, :512], 1 / np.sqrt(576), lay, idx.numpy())
    assert_matches(o, lse, O, LS, "bf16", "dsa tensor-core q chunk map")


# ---------------------------------------------------------------------------
# MoBA block gate + block-sparse attention
# ---------------------------------------------------------------------------

def _moba_gpu(w):
    q, k, v = to_gpu(w)
    sel = cpattn_block_gate(q, k, w.block_size, w.topk, causal_offset=w.causal_offset)
    o, lse = cpattn_topk_sparse_fwd(q, k, v, sel, block_size=w.block_size, scale=w.scale,
                                    causal_offset=w.causal_offset)
    return sel, o, lse


def test_moba_small():
    w = inputs.moba(seed=5, Tq=700, Tk=4096, offset=3300, H=4, block_size=256, topk=3)
    sel, o, lse = _moba_gpu(w)
    q, k, v = f64(w)
    lay = layout_of(w)
    ref_sel = orc.moba_block_gate(q, k, lay.qpos, w.block_size, w.topk)
    np.testing.assert_array_equal(sel.cpu().numpy(), ref_sel)
    O, L = orc.moba_attention(q, k, v, w.scale, lay, ref_sel, w.block_size)
    assert_matches(o, lse, O, L, "bf16", "moba small")


def test_moba_gate_ties_and_few_candidates():
    w = inputs.moba(seed=6, Tq=64, Tk=2048, offset=0, H=2, block_size=128, topk=3)
    k = w.k.clone()
    k[5 * 128:6 * 128] = k[2 * 128:3 * 128]        # blocks 2 and 5 have equal means
    k[9 * 128:10 * 128] = k[2 * 128:3 * 128]       # and block 9
    w.k = k
    w.causal_offset = 2048 - 64                    # own block 15; candidates 0..14
    q = w.q.clone()
    q[:] = (k[2 * 128:3 * 128].float().mean(0) * 50).to(torch.bfloat16)  # favour the tied blocks
    w.q = q
    sel, o, lse = _moba_gpu(w)
    qq, kk, _ = f64(w)
    ref = orc.moba_block_gate(qq, kk, layout_of(w).qpos, w.block_size, w.topk)
    np.testing.assert_array_equal(sel.cpu().numpy(), ref)
    assert (ref[:, :, :3] == [2, 5, 9]).all()
    # a query in block 1 has one candidate: [0, 1, -1, -1]
    w2 = inputs.moba(seed=7, Tq=8, Tk=1024, offset=130, H=2, block_size=128, topk=3)
    sel2, _, _ = _moba_gpu(w2)
    assert sel2[0, 0].tolist() == [0, 1, -1, -1]


def test_moba_attention_slot_patterns():
    """Block-grouped attention on hand-made selections: rows whose every slot
    is empty (-1), rows with only the own block, rows naming a block twice
    (each occurrence counts), and rows naming a block wholly after the query
    (no permitted key there) - equal to the float64 oracle, with O = 0 and
    LSE = -inf where nothing is permitted."""
    w = inputs.moba(seed=9, Tq=384, Tk=2048, offset=1664, H=2, block_size=128, topk=3)
    q, k, v = to_gpu(w)
    rng = np.random.default_rng(9)
    B, S = w.block_size, w.topk + 1
    own = (w.causal_offset + np.arange(w.Tq)) // B
    sel = np.full((w.Tq, 2, S), -1, dtype=np.int32)
    for i in range(w.Tq):
        for h in range(2):
            kind = (i + h) % 5
            if kind == 1:
                sel[i, h, 0] = own[i]
            elif kind == 2:
                b = rng.integers(0, own[i])
                sel[i, h, :3] = [b, b, own[i]]
            elif kind == 3:
                sel[i, h, :2] = [min(own[i] + 1, 15), rng.integers(0, own[i])]
            elif kind == 4:
                sel[i, h] = sorted(rng.choice(own[i], 3, replace=False).tolist()) + [own[i]]
    o, lse = cpattn_topk_sparse_fwd(q, k, v, torch.from_numpy(sel).cuda(), block_size=B,
                                    scale=w.scale, causal_offset=w.causal_offset)
    qf, kf, vf = f64(w)
    O, L, bad = orc.sparse_attention(qf, kf, vf, w.scale, layout_of(w), sel, B)
    assert bad == 0 and np.isneginf(L).sum() >= 150   # the all-empty rows at least
    assert_matches(o, lse, O, L, "bf16", "moba slot patterns")


@pytest.mark.parametrize("dtype,D", [("fp32", 64), ("bf16", 72), ("fp32", 136)])
def test_moba_gate_other_shapes_and_fp32(dtype, D):
    """The SIMT gate over the vectorised block means: fp32 inputs, head dims
    other than 128 (D = 136 leaves 7 row groups of 34 column quads):
    selections equal the float64 oracle's."""
    rng = np.random.default_rng(21 + D)
    Tq, Tk, H, B, topk = 48, 1536, 3, 128, 3
    qf = rng.standard_normal((Tq, H, D)) * 0.5
    kf = rng.standard_normal((Tk, H, D)) * 0.5
    tdt = torch.float32 if dtype == "fp32" else torch.bfloat16
    q = torch.tensor(qf, dtype=torch.float32).to(tdt)
    k = torch.tensor(kf, dtype=torch.float32).to(tdt)
    offset = Tk - Tq
    sel = cpattn_block_gate(q.cuda(), k.cuda(), B, topk, causal_offset=offset)
    qpos = offset + np.arange(Tq)
    ref = orc.moba_block_gate(q.double().numpy(), k.double().numpy(), qpos, B, topk)
    np.testing.assert_array_equal(sel.cpu().numpy(), ref)


def test_moba_full_size():
    w = inputs.moba()
    sel, o, lse = _moba_gpu(w)
    q, k, v = f64(w)
    lay = layout_of(w)
    ref_sel = orc.moba_block_gate(q, k, lay.qpos, w.block_size, w.topk)
    np.testing.assert_array_equal(sel.cpu().numpy(), ref_sel)   # every (query, head), bit-exact
    rows = sample_rows(w.Tq, 256, edges=(511, 512, 8191))
    O, L, _ = orc.sparse_attention(q, k, v, w.scale, lay, ref_sel, w.block_size, rows=rows)
    assert_matches(o[rows.tolist()], lse[rows.tolist()], O, L, "bf16", "moba full")


# ---------------------------------------------------------------------------
# lse_merge on its own
# ---------------------------------------------------------------------------

def test_lse_merge_neutral_parts():
    d = torch.device("cuda")
    rng = np.random.default_rng(8)
    po = rng.standard_normal((3, 37, 5, 64))
    pl = rng.standard_normal((3, 37, 5)) * 3
    pl[1, :10] = -np.inf
    pl[:, 20] = -np.inf                           # every part neutral for row 20
    po[np.isneginf(pl)] = 0
    O, L = orc.lse_merge(po, pl)
    o, lse = cpattn_lse_merge(torch.tensor(po, dtype=torch.float32, device=d),
                              torch.tensor(pl, dtype=torch.float32, device=d),
                              out_dtype=torch.float32)
    assert_matches(o, lse, O, L, "fp32", "lse_merge")
    assert (o[20] == 0).all() and torch.isneginf(lse[20]).all()


@pytest.mark.parametrize("n_parts", [1, 2, 4, 6])
@pytest.mark.parametrize("out", ["fp32", "bf16"])
def test_lse_merge_128_channels_neutral_parts_hold_garbage(n_parts, out):
    """Dv = 128 (the half-warp path up to four parts, the unrolled one beyond):
    a neutral part's channels are never used, whatever they hold."""
    d = torch.device("cuda")
    rng = np.random.default_rng(11 + n_parts)
    po = rng.standard_normal((n_parts, 53, 3, 128)) * 0.5   # the values' scale of the workloads
    pl = rng.standard_normal((n_parts, 53, 3)) * 4
    pl[0, :7] = -np.inf
    pl[:, 30] = -np.inf                           # every part neutral for row 30
    O, L = orc.lse_merge(np.where(np.isneginf(pl)[..., None], 0.0, po), pl)
    po_dev = torch.tensor(po, dtype=torch.float32, device=d)
    po_dev[torch.isneginf(torch.tensor(pl, device=d))] = float("nan")
    o, lse = cpattn_lse_merge(po_dev, torch.tensor(pl, dtype=torch.float32, device=d),
                              out_dtype=torch.float32 if out == "fp32" else torch.bfloat16)
    assert_matches(o, lse, O, L, out, f"lse_merge {n_parts} parts")
    assert (o[30].float() == 0).all() and torch.isneginf(lse[30]).all()


@pytest.mark.parametrize("Tq,Tk,off,Hq,Hkv,cu", [
    (640, 1500, 900, 4, 2, None),      # folded head pairs, odd number of query tiles
    (1000, 1100, 300, 2, 1, None),     # folded, ragged last tile, rows clipped at Tk
    (128, 4000, 3000, 4, 2, None),     # one query tile: both heads at tile 0
    (1000, 1000, 0, 8, 2, None),       # offset 0: tile 0 sees one KV tile, tile 7 eight
    (700, 900, 200, 2, 2, [0, 250, 610, 900]),   # adjacent tiles, packed sequences
    (700, 900, 200, 4, 2, [0, 250, 610, 900]),   # head pairs, packed sequences
])
def test_dense_per_unit_schedule_without_workspace(Tq, Tk, off, Hq, Hkv, cu):
    """Without a workspace the one-unit-per-CTA kernel runs; same answer.  A
    block whose live KV tiles are a prefix of its CTA's list stops early (one
    causal sequence); otherwise it runs the list and masks."""
    import ctypes
    from context_attention_softmax_gb300 import _lib
    w = inputs.dense_gqa(seed=3, global_seq=Tq, cp_size=1, rank=0, Hq=Hq, Hkv=Hkv, Tk=Tk,
                         kv_chunks=0)
    w.causal_offset = off
    if cu is not None:
        w.cu_seqlens = np.array(cu, dtype=np.int32)
    q, k, v = f64(w)
    O, L = orc.dense_attention(q, k, v, w.scale, layout_of(w))
    dev = torch.device("cuda")
    qd, kd, vd = w.q.to(dev), w.k.to(dev), w.v.to(dev)
    o = torch.empty((qd.shape[0], qd.shape[1], vd.shape[2]), dtype=qd.dtype, device=dev)
    lse = torch.empty((qd.shape[0], qd.shape[1]), dtype=torch.float32, device=dev)
    cu_d = None if cu is None else torch.tensor(cu, dtype=torch.int32, device=dev)
    a = pkg._args(qd, kd, vd, w.scale, True, w.causal_offset, cu_d, None, None, 0, o, lse)
    lib = _lib.load()
    _lib.check(lib.cpattn_chunk_fwd(ctypes.byref(a), None, 0, torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    assert_matches(o, lse, O, L, "bf16", "per-unit schedule")


# ---------------------------------------------------------------- DSA indexer
def _indexer_case(seed, Tq, Tk, H, D, offset, dup=None, cu=None):
    rng = np.random.default_rng(seed)
    qI = rng.standard_normal((Tq, H, D)).astype(np.float32)
    kI = rng.standard_normal((Tk, D)).astype(np.float32)
    w = rng.uniform(0.0, 1.0, H).astype(np.float32)
    if dup is not None:                         # equal keys: equal scores
        for j in dup[1:]:
            kI[j] = kI[dup[0]]
        qI[:, :, :] = kI[dup[0]] * 2.0           # and favoured by every query and head
    lay = orc.make_layout(Tq, Tk, True, offset, cu_seqlens=cu)
    return qI, kI, w, lay


@pytest.mark.parametrize("Tq,Tk,H,D,offset,topk", [
    (37, 700, 4, 64, 600, 50),       # every row has more permitted keys than k
    (40, 300, 3, 32, 0, 64),         # early rows: fewer permitted keys than k
    (9, 2000, 4, 128, 1990, 512),    # large k, D = 128
    # D = 128 takes the tensor-core scores (one instantiation per head count)
    (37, 700, 4, 128, 600, 50),
    (40, 300, 8, 128, 0, 64),        # early rows: fewer permitted keys than k
    (70, 900, 1, 128, 850, 100),
    (33, 1000, 2, 128, 960, 300),    # a ragged last query tile, keys not a multiple of 128
])
def test_dsa_indexer_matches_float64_oracle(Tq, Tk, H, D, offset, topk):
    qI, kI, w, lay = _indexer_case(31 + Tq, Tq, Tk, H, D, offset)
    ref = orc.dsa_indexer_topk(qI, kI, w, lay, topk)[:, 0, :]
    got = cpattn_dsa_indexer(torch.from_numpy(qI).cuda(), torch.from_numpy(kI).cuda(),
                             torch.from_numpy(w).cuda(), topk, causal_offset=offset)
    np.testing.assert_array_equal(got.cpu().numpy(), ref)


@pytest.mark.parametrize("D", [32, 128])
def test_dsa_indexer_ties_and_packed_sequences(D):
    """Keys 3, 130, 150, 300 and 390 are equal and favoured by every query: with
    k = 2 the two lowest permitted ones (130, 150) win - key 3 lies in the
    first packed sequence, which the queries of the second never see (D = 32
    scores on the SIMT path, D = 128 on the tensor cores)."""
    cu = np.array([0, 120, 400], dtype=np.int32)
    qI, kI, w, lay = _indexer_case(5, 50, 400, 2, D, 350, dup=(130, 3, 150, 300, 390), cu=cu)
    ref = orc.dsa_indexer_topk(qI, kI, w, lay, 2)[:, 0, :]
    got = cpattn_dsa_indexer(torch.from_numpy(qI).cuda(), torch.from_numpy(kI).cuda(),
                             torch.from_numpy(w).cuda(), 2, causal_offset=350,
                             cu_seqlens=torch.from_numpy(cu))
    np.testing.assert_array_equal(got.cpu().numpy(), ref)
    assert (got.cpu().numpy() == [130, 150]).all()


def test_dsa_indexer_full_size_every_row():
    """The DSA workload's indexer (4096 queries at offset 16384 over 32768
    keys, 4 heads of 128, k = 2048): every row equals the float64 oracle's,
    bit for bit."""
    w = inputs.dsa_absorbed()
    qI, kI, wt = w.extra["qI"], w.extra["kI"], w.extra["w"]
    got = cpattn_dsa_indexer(qI.cuda(), kI.cuda(), wt.cuda(), w.topk, causal_offset=w.causal_offset)
    lay = orc.make_layout(qI.shape[0], kI.shape[0], True, w.causal_offset)
    ref = orc.dsa_indexer_topk(qI.numpy(), kI.numpy(), wt.numpy(), lay, w.topk)[:, 0, :]
    np.testing.assert_array_equal(got.cpu().numpy(), ref)


# ---------------------------------------------------------------- bounded waits
def test_bounded_wait_runs_out_reports_timeout_and_the_stream_stays_usable():
    """A wait limit of 1 ns on the dense tensor-core kernel (one unit per CTA,
    64 KV tiles per CTA, so hundreds of waits): some barrier wait runs out,
    the kernel drains its copies and MMAs, frees tensor memory, writes
    CPATTN_ERR_TIMEOUT to dev_status and returns.  The next call on the same
    stream, with the default limit, is correct."""
    import ctypes
    from context_attention_softmax_gb300 import _lib
    w = inputs.dense_gqa(seed=12, global_seq=256, cp_size=1, rank=0, Hq=2, Hkv=1, Tk=8192,
                         kv_chunks=0)
    w.causal_offset = 8192 - 256
    qd, kd, vd = w.q.cuda(), w.k.cuda(), w.v.cuda()
    o = torch.empty((qd.shape[0], qd.shape[1], 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((qd.shape[0], qd.shape[1]), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib = _lib.load()
    stream = torch.cuda.current_stream().cuda_stream
    a = pkg._args(qd, kd, vd, w.scale, True, w.causal_offset, None, None, None, 0, o, lse,
                  dev_status=status)
    a.wait_limit_ns = 1
    _lib.check(lib.cpattn_chunk_fwd(ctypes.byref(a), None, 0, stream))
    torch.cuda.synchronize()
    assert int(status.item()) == 5               # CPATTN_ERR_TIMEOUT
    status.zero_()
    a.wait_limit_ns = 0                          # default limit
    _lib.check(lib.cpattn_chunk_fwd(ctypes.byref(a), None, 0, stream))
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    q, k, v = f64(w)
    O, L = orc.dense_attention(q, k, v, w.scale, layout_of(w))
    assert_matches(o, lse, O, L, "bf16", "after a timed-out call")
