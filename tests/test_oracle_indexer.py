"""Pins of the float64 DSA indexer oracle (oracle.dsa_indexer_topk).

Each test fixes the oracle against something other than its own formula:
special cases that reduce to a library sort, an algebraic identity of the
ReLU, constructed ties, the permitted relation, and the row convention for
rows with fewer permitted keys than k.
"""

import numpy as np
import pytest

import oracle as orc

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _sel(qI, kI, w, layout, topk):
    return orc.dsa_indexer_topk(qI, kI, w, layout, topk)[:, 0, :]


def test_one_head_positive_dots_is_a_plain_top_k_of_the_dot_product():
    """H = 1, w = 1 and positive entries: the score is the dot product, so the
    selection is numpy's stable argsort of -q.k (ties to the lower j) cut at k
    and sorted ascending."""
    rng = np.random.default_rng(1)
    qI = rng.random((9, 1, 16))
    kI = rng.random((70, 16))
    lay = orc.make_layout(9, 70, causal=False)
    got = _sel(qI, kI, np.ones(1), lay, 12)
    dots = qI[:, 0, :] @ kI.T
    for i in range(9):
        ref = np.sort(np.argsort(-dots[i], kind="stable")[:12])
        np.testing.assert_array_equal(got[i], ref)


def test_relu_pair_of_opposite_heads_scores_the_absolute_dot():
    """Heads +q and -q with equal weights: relu(x) + relu(-x) = |x|, so the
    selection is the top-k of |q.k|."""
    rng = np.random.default_rng(2)
    q = rng.standard_normal((7, 32))
    qI = np.stack([q, -q], axis=1)
    kI = rng.standard_normal((90, 32))
    lay = orc.make_layout(7, 90, causal=False)
    got = _sel(qI, kI, np.array([0.7, 0.7]), lay, 10)
    absdot = np.abs(q @ kI.T)
    for i in range(7):
        ref = np.sort(np.argsort(-absdot[i], kind="stable")[:10])
        np.testing.assert_array_equal(got[i], ref)


def test_negative_dots_contribute_nothing():
    """A head whose dots are all negative adds zero: the selection equals the
    one computed with that head removed."""
    rng = np.random.default_rng(3)
    kI = rng.random((60, 8))                      # positive keys
    q_pos = rng.random((5, 8))
    q_neg = -rng.random((5, 8))                   # every dot with kI negative
    qI = np.stack([q_pos, q_neg], axis=1)
    lay = orc.make_layout(5, 60, causal=False)
    both = _sel(qI, kI, np.array([0.3, 0.9]), lay, 9)
    alone = _sel(q_pos[:, None, :], kI, np.array([0.3]), lay, 9)
    np.testing.assert_array_equal(both, alone)


def test_equal_scores_go_to_the_lower_key():
    """Keys 4, 17 and 33 are the same vector and score highest; with k = 2 the
    two lowest of them are chosen."""
    rng = np.random.default_rng(4)
    kI = rng.standard_normal((40, 16)) * 0.1
    star = rng.standard_normal(16)
    for j in (4, 17, 33):
        kI[j] = star
    qI = np.stack([star * 3.0, star * 2.0], axis=0)[None, :, :].repeat(3, axis=0)
    lay = orc.make_layout(3, 40, causal=False)
    got = _sel(qI, kI, np.array([0.5, 0.25]), lay, 2)
    np.testing.assert_array_equal(got, [[4, 17]] * 3)


def test_only_permitted_keys_and_fewer_than_k_rows():
    """Causal at offset 3: query i sees keys 0..3+i only; rows with fewer
    permitted keys than k take all of them, ascending, padded with -1."""
    rng = np.random.default_rng(5)
    qI = rng.standard_normal((6, 2, 8))
    kI = rng.standard_normal((30, 8))
    lay = orc.make_layout(6, 30, causal=True, causal_offset=3)
    got = _sel(qI, kI, np.array([1.0, 0.5]), lay, 6)
    for i in range(6):
        n = 4 + i
        if n <= 6:
            np.testing.assert_array_equal(got[i, :n], np.arange(n))
            assert (got[i, n:] == -1).all()
        else:
            assert (got[i] >= 0).all() and (got[i] <= 3 + i).all()
            assert (np.diff(got[i]) > 0).all()


def test_packed_sequences_never_cross():
    """Two packed sequences (cut at 20): a query of the second sequence never
    selects a key of the first, however well it scores."""
    rng = np.random.default_rng(6)
    kI = rng.standard_normal((40, 8))
    kI[:20] *= 10.0                               # first sequence scores far higher
    qI = np.abs(rng.standard_normal((40, 1, 8)))
    kI = np.abs(kI)
    lay = orc.make_layout(40, 40, causal=True, cu_seqlens=np.array([0, 20, 40]))
    got = _sel(qI, kI, np.ones(1), lay, 5)
    for i in range(20, 40):
        row = got[i][got[i] >= 0]
        assert (row >= 20).all() and (row <= i).all()


def test_weight_scale_and_head_order_do_not_change_the_selection():
    rng = np.random.default_rng(7)
    qI = rng.standard_normal((8, 4, 16))
    kI = rng.standard_normal((50, 16))
    w = rng.random(4)
    lay = orc.make_layout(8, 50, causal=True, causal_offset=30)
    base = _sel(qI, kI, w, lay, 7)
    np.testing.assert_array_equal(_sel(qI, kI, w * 4.0, lay, 7), base)   # power-of-two scale is exact
    perm = np.array([2, 0, 3, 1])
    np.testing.assert_array_equal(_sel(qI[:, perm], kI, w[perm], lay, 7), base)


def _brute_topk(qI, kI, w, qpos, kpos, seq_q, seq_k, causal, topk):
    """Scalar loops with math.fsum: the score definition, the permitted
    relation, then a full sort of (score desc, j asc) per row."""
    import math
    Tq, H, D = qI.shape
    out = []
    for i in range(Tq):
        cands = []
        for j in range(kI.shape[0]):
            if seq_q[i] < 0 or seq_q[i] != seq_k[j] or (causal and kpos[j] > qpos[i]):
                continue
            sc = math.fsum(float(w[h]) * max(0.0, math.fsum(float(qI[i, h, d]) * float(kI[j, d])
                                                             for d in range(D)))
                           for h in range(H))
            cands.append((-sc, int(kpos[j])))     # a key is named by its logical position
        cands.sort()
        row = sorted(j for _, j in cands[:topk])
        out.append(row + [-1] * (topk - len(row)))
    return np.array(out)


def test_brute_force_with_mixed_sign_weights_packed_and_offset():
    """A negative head weight turns that head's ReLU into a penalty; two
    packed sequences, a causal offset and a query past the last sequence
    (it selects nothing).  The oracle equals scalar brute force."""
    rng = np.random.default_rng(8)
    Tq, Tk, H, D, k = 14, 40, 3, 6, 5
    qI = rng.standard_normal((Tq, H, D))
    kI = rng.standard_normal((Tk, D))
    w = np.array([0.8, -0.5, 0.3])
    cu = np.array([0, 17, 38])
    lay = orc.make_layout(Tq, Tk, causal=True, causal_offset=25, cu_seqlens=cu)
    got = _sel(qI, kI, w, lay, k)
    qpos = 25 + np.arange(Tq)
    kpos = np.arange(Tk)
    seq = lambda p: np.searchsorted(cu, p, side="right") - 1 if p < cu[-1] else -1
    seq_q = [seq(p) for p in qpos]
    seq_k = [seq(p) for p in kpos]
    ref = _brute_topk(qI, kI, w, qpos, kpos, seq_q, seq_k, True, k)
    np.testing.assert_array_equal(got, ref)
    assert (got[qpos >= 38] == -1).all()            # positions 38.. are in no sequence


def test_brute_force_with_a_kv_chunk_map():
    """Keys stored in zigzag order (physical chunk c holds logical chunk
    map[c]): the oracle names each chosen key by its LOGICAL position, ranks
    equal scores by logical position, and equals scalar brute force over the
    logical positions.  Storing the same keys in logical order gives the same
    selection ([CP] para 5: the layout changes ownership, not the relation)."""
    rng = np.random.default_rng(9)
    L, n_chunks, H, D, k = 8, 6, 2, 5, 7
    Tk, Tq = L * n_chunks, 11
    cmap = np.array([0, 5, 1, 4, 2, 3])
    kI_logical = rng.standard_normal((Tk, D))
    kI_logical[33] = kI_logical[9]                    # equal keys in different chunks
    qI = rng.standard_normal((Tq, H, D))
    qI[4] = np.stack([kI_logical[9] * 4.0, kI_logical[9]])   # favours keys 9 and 33
    w = np.array([0.6, 0.4])
    phys_to_log = (cmap[np.arange(Tk) // L] * L + np.arange(Tk) % L)
    kI_phys = np.empty_like(kI_logical)
    kI_phys[np.arange(Tk)] = kI_logical[phys_to_log]
    lay = orc.make_layout(Tq, Tk, causal=True, causal_offset=36, kv_chunk_map=cmap, chunk_len=L)
    got = _sel(qI, kI_phys, w, lay, k)
    qpos = 36 + np.arange(Tq)
    ref = _brute_topk(qI, kI_phys, w, qpos, lay.kpos, [0] * Tq, [0] * Tk, True, k)
    np.testing.assert_array_equal(got, ref)
    lay_log = orc.make_layout(Tq, Tk, causal=True, causal_offset=36)
    np.testing.assert_array_equal(got, _sel(qI, kI_logical, w, lay_log, k))
    assert {9, 33} <= set(got[4].tolist())
    assert got.max() <= qpos.max()
