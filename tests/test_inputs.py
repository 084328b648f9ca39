"""The seeded input recipes (CPU): what the workloads are, checked against
their stated definitions.  The inputs module holds no attention arithmetic;
its one selection routine (the DSA index generator, input synthesis for the
sparse-attention workload) is checked here against the float64 indexer
definition in the oracle."""
import numpy as np
import torch

import oracle as orc
from context_attention_softmax_gb300 import inputs


def test_zigzag_lengths_seed0_and_renormalisation():
    lens = inputs.seeded_lengths(np.random.default_rng(0), 8, 16384, 512, 4096)
    assert lens.tolist() == [4226, 3317, 2782, 1755, 1916, 780, 926, 682]
    assert int(lens.sum()) == 16384
    lens = inputs.seeded_lengths(np.random.default_rng(3), 5, 1000, 50, 400)
    assert int(lens.sum()) == 1000 and len(lens) == 5


def test_zigzag_gathered_kv_is_rank_major():
    z = inputs.zigzag_varlen(seed=1, total=1024, n_seqs=3, len_lo=100, len_hi=600, cp_size=4,
                             H=2, D=16)
    # slot 2r holds logical chunk r, slot 2r+1 holds chunk 2cp-1-r
    assert z.kv_chunk_map.tolist() == [0, 7, 1, 6, 2, 5, 3, 4]
    L = z.chunk_len
    for slot, c in enumerate(z.kv_chunk_map.tolist()):
        assert torch.equal(z.k_gathered[slot * L:(slot + 1) * L], z.k_global[c * L:(c + 1) * L])
    # rank r's local queries are logical chunks r and 2cp-1-r, in that order
    q1 = z.rank_q(1)
    assert torch.equal(q1[:L], z.q_global[L:2 * L]) and torch.equal(q1[L:], z.q_global[6 * L:7 * L])


def test_dense_workload_shapes_offset_and_scale():
    w = inputs.dense_gqa(global_seq=1024, cp_size=4, rank=2, Hq=4, Hkv=2, D=32, kv_chunks=4)
    assert tuple(w.q.shape) == (256, 4, 32) and tuple(w.k.shape) == (1024, 2, 32)
    assert w.q.dtype == torch.bfloat16 and w.causal and w.causal_offset == 512
    assert w.kv_chunk_len == 256 and abs(w.scale - 1 / np.sqrt(32)) < 1e-12
    sd = float(w.k.float().std())
    assert 0.45 < sd < 0.55                     # N(0, 1) * 0.5


def test_index_generator_matches_the_float64_indexer_definition():
    rng = np.random.default_rng(9)
    Tq, Tk, H, D, k, off = 20, 60, 3, 16, 8, 30
    qI = rng.standard_normal((Tq, H, D)).astype(np.float32)
    kI = rng.standard_normal((Tk, D)).astype(np.float32)
    w = rng.uniform(0, 1, H).astype(np.float32)
    got = inputs.indexer_topk(torch.from_numpy(qI), torch.from_numpy(kI), torch.from_numpy(w),
                              torch.arange(Tq) + off, k, row_block=7)
    lay = orc.make_layout(Tq, Tk, causal=True, causal_offset=off)
    ref = orc.dsa_indexer_topk(qI, kI, w, lay, k)
    np.testing.assert_array_equal(got.numpy(), ref)
