"""Pins of the float64 oracle against things other than itself (CPU only).

* brute force on tiny inputs: scalar loops, math.fsum, the plain softmax
  exp(s) / sum exp(s) with no max subtraction, and the permitted relation
  rebuilt from an explicit token -> (sequence, position) table;
* library routines: torch.nn.functional.scaled_dot_product_attention and
  torch.logsumexp in float64 (no mask, causal, block-diagonal varlen mask),
  scipy.special.logsumexp for the overflow case;
* a hand-derived worked example (tests/golden/two_chunk_merge.json);
* the invariants stated on the pages: the chunked merge equals the global
  softmax, a chunk at causal_offset equals the slice of the full run, zigzag
  ownership reassembles the full run, packed equals per-sequence, GQA equals
  repeated-KV MHA, an all-masked chunk is neutral, no key gives (0, -inf).
"""

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------------------
# independent brute force
# ---------------------------------------------------------------------------

def token_table(n_tokens, cu_seqlens):
    """position -> sequence id by walking the packed lengths (None if outside)."""
    seq = [None] * n_tokens
    if cu_seqlens is None:
        return [0] * n_tokens
    for s in range(len(cu_seqlens) - 1):
        for p in range(int(cu_seqlens[s]), int(cu_seqlens[s + 1])):
            if p < n_tokens:
                seq[p] = s
    return seq


def positions_by_listing(n, offset, chunk_map, chunk_len):
    if chunk_map is None:
        return [offset + t for t in range(n)]
    out = []
    for c in chunk_map:
        out.extend(offset + int(c) * chunk_len + t for t in range(chunk_len))
    return out[:n]


def brute_attention(q, k, v, scale, qpos, kpos, seq_of, causal, key_lists=None):
    """Plain softmax over explicit key lists; no max subtraction (small inputs)."""
    Tq, Hq, D = q.shape
    Tk, Hkv, Dv = v.shape
    grp = Hq // Hkv
    O = np.zeros((Tq, Hq, Dv))
    LSE = np.full((Tq, Hq), -np.inf)
    for i in range(Tq):
        for h in range(Hq):
            g = h // grp
            if key_lists is None:
                cand = list(range(Tk))
            else:
                cand = key_lists[i][h]
            keys = []
            for j in cand:
                sq, sk = seq_of(qpos[i]), seq_of(kpos[j])
                if sq is None or sk is None or sq != sk:
                    continue
                if causal and kpos[j] > qpos[i]:
                    continue
                keys.append(j)
            if not keys:
                continue
            w = [math.exp(scale * math.fsum(q[i, h, d] * k[j, g, d] for d in range(D))) for j in keys]
            den = math.fsum(w)
            for d in range(Dv):
                O[i, h, d] = math.fsum(wj * v[j, g, d] for wj, j in zip(w, keys)) / den
            LSE[i, h] = math.log(den)
    return O, LSE


def rnd(rng, *shape, f=0.5):
    return rng.standard_normal(shape) * f


def seq_lookup(n, cu):
    table = token_table(n, cu)
    return lambda p: table[p] if 0 <= p < n else None


CASES = {
    # name: (Tq, Tk, Hq, Hkv, causal, offset, cu, qmap, kvmap, chunk_len)
    "offset_causal": (8, 24, 2, 2, True, 10, None, None, None, 0),
    "non_causal": (8, 24, 2, 1, False, 10, None, None, None, 0),
    "varlen_causal": (12, 24, 2, 2, True, 8, [0, 5, 11, 20, 24], None, None, 0),
    "zigzag_varlen": (8, 24, 2, 2, True, 0, [0, 7, 13, 24], [1, 4], [0, 5, 1, 4, 2, 3], 4),
    "gqa": (6, 16, 4, 2, True, 6, None, None, None, 0),
    "query_outside_sequences": (6, 20, 1, 1, True, 14, [0, 9, 16], None, None, 0),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_dense_matches_brute_force(name):
    Tq, Tk, Hq, Hkv, causal, off, cu, qmap, kvmap, L = CASES[name]
    rng = np.random.default_rng(hash(name) % 2**32)
    q, k, v = rnd(rng, Tq, Hq, 5), rnd(rng, Tk, Hkv, 5), rnd(rng, Tk, Hkv, 3)
    lay = orc.make_layout(Tq, Tk, causal, off, cu, qmap, kvmap, L)
    O, LSE = orc.dense_attention(q, k, v, 0.7, lay)
    qpos = positions_by_listing(Tq, off, qmap, L)
    kpos = positions_by_listing(Tk, 0, kvmap, L)
    Ob, Lb = brute_attention(q, k, v, 0.7, qpos, kpos, seq_lookup(64, cu), causal)
    np.testing.assert_allclose(O, Ob, rtol=0, atol=1e-12)
    np.testing.assert_array_equal(np.isneginf(LSE), np.isneginf(Lb))
    fin = np.isfinite(Lb)
    np.testing.assert_allclose(LSE[fin], Lb[fin], rtol=0, atol=1e-12)
    if name == "query_outside_sequences":
        # positions 16..19 lie in no sequence: no permitted key -> (0, -inf)
        assert np.isneginf(LSE[2:]).all() and (O[2:] == 0).all()


def test_positions_match_listing():
    for Tq, Tk, Hq, Hkv, causal, off, cu, qmap, kvmap, L in CASES.values():
        lay = orc.make_layout(Tq, Tk, causal, off, cu, qmap, kvmap, L)
        assert lay.qpos.tolist() == positions_by_listing(Tq, off, qmap, L)
        assert lay.kpos.tolist() == positions_by_listing(Tk, 0, kvmap, L)


# ---------------------------------------------------------------------------
# library routines
# ---------------------------------------------------------------------------

def _sdpa(q, k, v, scale, **kw):
    tq, tk, tv = (torch.from_numpy(x).permute(1, 0, 2) for x in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, scale=scale, **kw)
    return o.permute(1, 0, 2).numpy()


def _torch_lse(q, k, scale, mask=None):
    s = scale * torch.einsum("ihd,jhd->hij", torch.from_numpy(q), torch.from_numpy(k))
    if mask is not None:
        s = s.masked_fill(~torch.from_numpy(mask)[None], float("-inf"))
    return torch.logsumexp(s, dim=-1).T.numpy()


def test_dense_matches_sdpa_no_mask():
    rng = np.random.default_rng(1)
    q, k, v = rnd(rng, 37, 3, 16, f=1), rnd(rng, 53, 3, 16, f=1), rnd(rng, 53, 3, 8, f=1)
    lay = orc.make_layout(37, 53, causal=False)
    O, LSE = orc.dense_attention(q, k, v, 0.25, lay)
    np.testing.assert_allclose(O, _sdpa(q, k, v, 0.25), atol=1e-12, rtol=0)
    np.testing.assert_allclose(LSE, _torch_lse(q, k, 0.25), atol=1e-12, rtol=0)


def test_dense_matches_sdpa_causal():
    rng = np.random.default_rng(2)
    q, k, v = rnd(rng, 64, 2, 16, f=1), rnd(rng, 64, 2, 16, f=1), rnd(rng, 64, 2, 16, f=1)
    lay = orc.make_layout(64, 64, causal=True)
    O, LSE = orc.dense_attention(q, k, v, 0.25, lay)
    np.testing.assert_allclose(O, _sdpa(q, k, v, 0.25, is_causal=True), atol=1e-12, rtol=0)
    np.testing.assert_allclose(LSE, _torch_lse(q, k, 0.25, np.tril(np.ones((64, 64), bool))),
                               atol=1e-12, rtol=0)


def test_dense_matches_sdpa_block_diagonal_varlen():
    lens = [7, 19, 1, 13]
    T = sum(lens)
    cu = np.concatenate([[0], np.cumsum(lens)])
    mask = torch.block_diag(*[torch.tril(torch.ones(n, n, dtype=torch.bool)) for n in lens]).numpy()
    rng = np.random.default_rng(3)
    q, k, v = rnd(rng, T, 2, 8, f=1), rnd(rng, T, 2, 8, f=1), rnd(rng, T, 2, 8, f=1)
    lay = orc.make_layout(T, T, causal=True, cu_seqlens=cu)
    O, LSE = orc.dense_attention(q, k, v, 0.5, lay)
    np.testing.assert_allclose(O, _sdpa(q, k, v, 0.5, attn_mask=torch.from_numpy(mask)),
                               atol=1e-12, rtol=0)
    np.testing.assert_allclose(LSE, _torch_lse(q, k, 0.5, mask), atol=1e-12, rtol=0)


def test_overflow_safe_softmax_matches_scipy():
    from scipy.special import logsumexp, softmax
    rng = np.random.default_rng(4)
    q, k, v = rnd(rng, 16, 1, 8, f=100.0), rnd(rng, 40, 1, 8, f=1), rnd(rng, 40, 1, 4, f=1)
    lay = orc.make_layout(16, 40, causal=True, causal_offset=24)
    O, LSE = orc.dense_attention(q, k, v, 1.0, lay)
    assert np.isfinite(O).all() and np.isfinite(LSE).all()
    s = q[:, 0] @ k[:, 0].T
    s = np.where(lay.allowed(), s, -np.inf)
    assert np.abs(s[np.isfinite(s)]).max() > 800  # exp(s) alone would overflow float64
    np.testing.assert_allclose(O[:, 0], softmax(s, axis=1) @ v[:, 0], atol=1e-12, rtol=0)
    np.testing.assert_allclose(LSE[:, 0], logsumexp(s, axis=1), atol=1e-9, rtol=1e-15)
    _, _, po, pl = orc.summarised_attention(q, k, v, 1.0, lay, 8)
    assert np.isfinite(po).all() and not np.isnan(pl).any()


# ---------------------------------------------------------------------------
# worked example (closed form)
# ---------------------------------------------------------------------------

def test_golden_two_chunk_merge():
    with open(os.path.join(GOLDEN, "two_chunk_merge.json")) as f:
        g = json.load(f)
    sa = orc.chunk_summary(np.array([g["chunk_a"]["scores"]]), np.ones((1, 2), bool),
                           np.array(g["chunk_a"]["values"]))
    sb = orc.chunk_summary(np.array([g["chunk_b"]["scores"]]), np.ones((1, 1), bool),
                           np.array(g["chunk_b"]["values"]))
    for s, ref in ((sa, g["summary_a"]), (sb, g["summary_b"])):
        assert s[0][0] == pytest.approx(ref["m"], abs=1e-15)
        assert s[1][0] == pytest.approx(ref["l"], abs=1e-15)
        np.testing.assert_allclose(s[2][0], ref["z"], atol=1e-15)
    mg = orc.merge_summaries(sa, sb)
    assert mg[0][0] == pytest.approx(g["merged"]["m"], abs=1e-15)
    assert mg[1][0] == pytest.approx(g["merged"]["l"], abs=1e-15)
    np.testing.assert_allclose(mg[2][0], g["merged"]["z"], atol=1e-14)
    O, LSE = orc.finalise(mg)
    np.testing.assert_allclose(O[0], g["output"]["O"], atol=1e-14)
    assert LSE[0] == pytest.approx(g["output"]["LSE"], abs=1e-14)
    # merge is symmetric and a neutral chunk changes nothing
    O2, L2 = orc.finalise(orc.merge_summaries(orc.merge_summaries(sb, orc.neutral_summary(1, 2)), sa))
    np.testing.assert_allclose(O2, O, atol=1e-14)
    assert L2[0] == pytest.approx(LSE[0], abs=1e-14)
    # the same numbers through the dense definition: D = 1, q = 1, k = scores
    q = np.ones((1, 1, 1))
    k = np.array(g["chunk_a"]["scores"] + g["chunk_b"]["scores"]).reshape(3, 1, 1)
    v = np.array(g["chunk_a"]["values"] + g["chunk_b"]["values"]).reshape(3, 1, 2)
    Od, Ld = orc.dense_attention(q, k, v, 1.0, orc.make_layout(1, 3, causal=False))
    np.testing.assert_allclose(Od[0, 0], g["output"]["O"], atol=1e-14)
    assert Ld[0, 0] == pytest.approx(g["output"]["LSE"], abs=1e-14)
    # the LSE form of the merge
    Oa, La = orc.finalise(sa)
    Ob, Lb = orc.finalise(sb)
    Om, Lm = orc.lse_merge(np.stack([Oa, Ob]), np.stack([La, Lb]))
    np.testing.assert_allclose(Om[0], g["output"]["O"], atol=1e-14)
    assert Lm[0] == pytest.approx(g["output"]["LSE"], abs=1e-14)
    # no permitted key anywhere: (0, -inf), no NaN
    On, Ln = orc.finalise(orc.merge_summaries(orc.neutral_summary(1, 2), orc.neutral_summary(1, 2)))
    assert (On == 0).all() and np.isneginf(Ln).all()


# ---------------------------------------------------------------------------
# invariants from the pages
# ---------------------------------------------------------------------------

def test_two_chunk_merge_equals_global_softmax():
    rng = np.random.default_rng(0)
    q, k, v = rnd(rng, 128, 1, 64, f=1), rnd(rng, 256, 1, 64, f=1), rnd(rng, 256, 1, 64, f=1)
    lay = orc.make_layout(128, 256, True, 128)
    O, LSE = orc.dense_attention(q, k, v, 1 / 8, lay)
    Os, Ls, po, pl = orc.summarised_attention(q, k, v, 1 / 8, lay, 128)
    np.testing.assert_allclose(Os, O, atol=1e-12, rtol=0)
    np.testing.assert_allclose(Ls, LSE, atol=1e-12, rtol=0)
    Om, Lm = orc.lse_merge(po, pl)
    np.testing.assert_allclose(Om, O, atol=1e-12, rtol=0)
    np.testing.assert_allclose(Lm, LSE, atol=1e-12, rtol=0)
    # chunk 0 alone (keys 0..127, all before every query) is plain full attention
    O0, L0 = orc.dense_attention(q, k[:128], v[:128], 1 / 8, orc.make_layout(128, 128, False))
    np.testing.assert_allclose(po[0], O0, atol=1e-12, rtol=0)
    np.testing.assert_allclose(pl[0], L0, atol=1e-12, rtol=0)


def test_fully_masked_chunk_is_neutral():
    rng = np.random.default_rng(5)
    q, k, v = rnd(rng, 64, 4, 16), rnd(rng, 256, 2, 16), rnd(rng, 256, 2, 16)
    lay = orc.make_layout(64, 256, True, 128)          # keys 192..255 are all in the future
    O, LSE = orc.dense_attention(q, k, v, 0.25, lay)
    Os, Ls, po, pl = orc.summarised_attention(q, k, v, 0.25, lay, 64)
    assert (po[3] == 0).all() and np.isneginf(pl[3]).all()
    assert not np.isnan(po).any() and not np.isnan(pl).any()
    np.testing.assert_allclose(Os, O, atol=1e-12, rtol=0)
    np.testing.assert_allclose(Ls, LSE, atol=1e-12, rtol=0)


def test_chunk_at_offset_equals_slice_of_full_run():
    rng = np.random.default_rng(6)
    T, cp = 96, 4
    q, k, v = rnd(rng, T, 2, 16), rnd(rng, T, 2, 16), rnd(rng, T, 2, 16)
    Of, Lf = orc.dense_attention(q, k, v, 0.3, orc.make_layout(T, T, True))
    loc = T // cp
    for r in range(cp):
        O, L = orc.dense_attention(q[r * loc:(r + 1) * loc], k, v, 0.3,
                                   orc.make_layout(loc, T, True, r * loc))
        np.testing.assert_allclose(O, Of[r * loc:(r + 1) * loc], atol=1e-13, rtol=0)
        np.testing.assert_allclose(L, Lf[r * loc:(r + 1) * loc], atol=1e-13, rtol=0)


def test_zigzag_ownership_reassembles_full_run():
    rng = np.random.default_rng(7)
    cp, L = 4, 16
    T = 2 * cp * L
    cu = np.array([0, 21, 50, 51, 100, 128])
    q, k, v = rnd(rng, T, 2, 8), rnd(rng, T, 2, 8), rnd(rng, T, 2, 8)
    Of, Lf = orc.dense_attention(q, k, v, 0.4, orc.make_layout(T, T, True, 0, cu))
    kvmap = [c for r in range(cp) for c in (r, 2 * cp - 1 - r)]
    kphys = np.concatenate([k[c * L:(c + 1) * L] for c in kvmap])
    vphys = np.concatenate([v[c * L:(c + 1) * L] for c in kvmap])
    Oasm = np.zeros_like(Of)
    Lasm = np.zeros_like(Lf)
    for r in range(cp):
        mine = [r, 2 * cp - 1 - r]
        ql = np.concatenate([q[c * L:(c + 1) * L] for c in mine])
        lay = orc.make_layout(2 * L, T, True, 0, cu, mine, kvmap, L)
        O, LSE = orc.dense_attention(ql, kphys, vphys, 0.4, lay)
        for slot, c in enumerate(mine):
            Oasm[c * L:(c + 1) * L] = O[slot * L:(slot + 1) * L]
            Lasm[c * L:(c + 1) * L] = LSE[slot * L:(slot + 1) * L]
    np.testing.assert_allclose(Oasm, Of, atol=1e-13, rtol=0)
    np.testing.assert_allclose(Lasm, Lf, atol=1e-13, rtol=0)


def test_packed_equals_per_sequence_runs():
    rng = np.random.default_rng(8)
    lens = [9, 30, 4, 21]
    cu = np.concatenate([[0], np.cumsum(lens)])
    T = cu[-1]
    q, k, v = rnd(rng, T, 2, 8), rnd(rng, T, 2, 8), rnd(rng, T, 2, 8)
    for causal in (True, False):
        O, LSE = orc.dense_attention(q, k, v, 0.4, orc.make_layout(T, T, causal, 0, cu))
        for s in range(len(lens)):
            a, b = cu[s], cu[s + 1]
            Os, Ls = orc.dense_attention(q[a:b], k[a:b], v[a:b], 0.4,
                                         orc.make_layout(b - a, b - a, causal))
            np.testing.assert_allclose(O[a:b], Os, atol=1e-13, rtol=0)
            np.testing.assert_allclose(LSE[a:b], Ls, atol=1e-13, rtol=0)


def test_gqa_equals_repeated_kv():
    rng = np.random.default_rng(9)
    q, k, v = rnd(rng, 20, 6, 8), rnd(rng, 50, 2, 8), rnd(rng, 50, 2, 4)
    lay = orc.make_layout(20, 50, True, 30)
    O, LSE = orc.dense_attention(q, k, v, 0.3, lay)
    Om, Lm = orc.dense_attention(q, np.repeat(k, 3, axis=1), np.repeat(v, 3, axis=1), 0.3, lay)
    np.testing.assert_allclose(O, Om, atol=1e-14, rtol=0)
    np.testing.assert_allclose(LSE, Lm, atol=1e-14, rtol=0)


def test_rows_subset_matches_full():
    rng = np.random.default_rng(10)
    q, k, v = rnd(rng, 40, 2, 8), rnd(rng, 60, 1, 8), rnd(rng, 60, 1, 8)
    lay = orc.make_layout(40, 60, True, 20)
    O, LSE = orc.dense_attention(q, k, v, 0.3, lay)
    rows = np.array([0, 7, 39, 13])
    Or, Lr = orc.dense_attention(q, k, v, 0.3, lay, rows=rows)
    np.testing.assert_array_equal(Or, O[rows])
    np.testing.assert_array_equal(Lr, LSE[rows])


# ---------------------------------------------------------------------------
# sparse (DSA token indices, MoBA blocks)
# ---------------------------------------------------------------------------

def test_sparse_with_every_permitted_key_equals_dense():
    rng = np.random.default_rng(11)
    Tq, Tk, off = 16, 48, 32
    q, k, v = rnd(rng, Tq, 4, 12), rnd(rng, Tk, 1, 12), rnd(rng, Tk, 1, 8)
    lay = orc.make_layout(Tq, Tk, True, off)
    idx = np.full((Tq, 1, Tk), -1, np.int32)
    for i in range(Tq):
        idx[i, 0, :off + i + 1] = np.arange(off + i + 1)
    O, LSE, bad = orc.sparse_attention(q, k, v, 0.3, lay, idx)
    Od, Ld = orc.dense_attention(q, k, v, 0.3, lay)
    assert bad == 0
    np.testing.assert_allclose(O, Od, atol=1e-13, rtol=0)
    np.testing.assert_allclose(LSE, Ld, atol=1e-13, rtol=0)


def test_sparse_matches_brute_force_with_duplicates_masks_and_bad_indices():
    rng = np.random.default_rng(12)
    Tq, Tk, off, Hq = 6, 30, 10, 2
    cu = [0, 12, 30]
    q, k, v = rnd(rng, Tq, Hq, 6), rnd(rng, Tk, 1, 6), rnd(rng, Tk, 1, 5)
    lay = orc.make_layout(Tq, Tk, True, off, cu)
    idx = rng.integers(0, Tk, (Tq, Hq, 9)).astype(np.int32)
    idx[0, 0, :] = -1                      # nothing selected -> (0, -inf)
    idx[1, 1, 3] = idx[1, 1, 4]           # duplicate counts twice
    idx[2, 0, 0] = Tk + 5                 # out of range -> skipped, counted
    idx[3, 1, 2] = -7                     # below -1 -> skipped, counted
    O, LSE, bad = orc.sparse_attention(q, k, v, 0.5, lay, idx)
    assert bad == 2
    key_lists = [[[int(j) for j in idx[i, h] if 0 <= j < Tk] for h in range(Hq)] for i in range(Tq)]
    qpos = positions_by_listing(Tq, off, None, 0)
    Ob, Lb = brute_attention(q, k, v, 0.5, qpos, list(range(Tk)), seq_lookup(Tk, cu), True, key_lists)
    np.testing.assert_allclose(O, Ob, atol=1e-12, rtol=0)
    np.testing.assert_array_equal(np.isneginf(LSE), np.isneginf(Lb))
    fin = np.isfinite(Lb)
    np.testing.assert_allclose(LSE[fin], Lb[fin], atol=1e-12, rtol=0)
    assert np.isneginf(LSE[0, 0]) and (O[0, 0] == 0).all()


def test_block_indices_select_whole_blocks():
    rng = np.random.default_rng(13)
    Tq, Tk, B, off = 8, 64, 8, 40
    q, k, v = rnd(rng, Tq, 2, 6), rnd(rng, Tk, 2, 6), rnd(rng, Tk, 2, 6)
    lay = orc.make_layout(Tq, Tk, True, off)
    sel = np.tile(np.array([1, 3, 5, -1], np.int32), (Tq, 2, 1))
    O, LSE, _ = orc.sparse_attention(q, k, v, 0.4, lay, sel, block_size=B)
    tok = np.full((Tq, 2, 24), -1, np.int32)
    tok[:, :, :] = np.concatenate([np.arange(8, 16), np.arange(24, 32), np.arange(40, 48)])
    Ot, Lt, _ = orc.sparse_attention(q, k, v, 0.4, lay, tok, block_size=1)
    np.testing.assert_array_equal(O, Ot)
    np.testing.assert_array_equal(LSE, Lt)


# ---------------------------------------------------------------------------
# MoBA gate
# ---------------------------------------------------------------------------

def brute_gate(q, k, qpos, B, topk):
    Tq, Hq, D = q.shape
    Hkv = k.shape[1]
    nb = k.shape[0] // B
    sel = np.full((Tq, Hq, topk + 1), -1, np.int32)
    for i in range(Tq):
        own = qpos[i] // B
        for h in range(Hq):
            g = h // (Hq // Hkv)
            gates = []
            for b in range(min(own, nb)):
                mu = [math.fsum(k[b * B + t, g, d] for t in range(B)) / B for d in range(D)]
                gates.append((-math.fsum(q[i, h, d] * mu[d] for d in range(D)), b))
            chosen = [b for _, b in sorted(gates)[:topk]] + [own]
            chosen.sort()
            sel[i, h, :len(chosen)] = chosen
    return sel


def test_gate_matches_brute_force():
    rng = np.random.default_rng(14)
    B, topk = 4, 3
    q, k = rnd(rng, 10, 4, 6), rnd(rng, 48, 2, 6)
    qpos = np.arange(10) * 5 - 2
    qpos[0] = 0
    sel = orc.moba_block_gate(q, k, qpos, B, topk)
    np.testing.assert_array_equal(sel, brute_gate(q, k, qpos, B, topk))
    # fewer candidates than topk -> all of them plus own, -1 padded
    assert sel[0, 0].tolist() == [0, -1, -1, -1]


def test_gate_ties_go_to_lower_block():
    rng = np.random.default_rng(15)
    B = 4
    k = rnd(rng, 40, 1, 6)
    k[8:12] = k[24:28]          # blocks 2 and 6 equal
    k[4:8] = k[24:28]           # block 1 too
    q = rnd(rng, 3, 1, 6)
    mu6 = k[24:28, 0].mean(0)
    # make blocks 1, 2, 6 the clear winners with equal gates, topk = 2
    for b in (0, 3, 4, 5, 7, 8):
        k[b * B:(b + 1) * B, 0] = -np.sign(q[0, 0]) * np.abs(k[b * B:(b + 1) * B, 0]) - 5 * np.sign(q[0, 0])
    qpos = np.array([38, 38, 38])
    sel = orc.moba_block_gate(q[:1], k, qpos, B, 2)
    assert sel[0, 0].tolist() == [1, 2, 9]
    assert np.allclose(k[4:8, 0].mean(0), mu6)


def test_gate_constant_blocks_closed_form():
    B, D = 8, 4
    nb = 6
    k = np.zeros((nb * B, 1, D))
    for b in range(nb):
        k[b * B:(b + 1) * B, 0, :] = b * np.array([1.0, -1.0, 0.5, 0.0])
    # gate(b) = b * (q . [1, -1, .5, 0]); with q = [1, 0, 0, 0]: gate = b, larger b wins
    q = np.array([[[1.0, 0.0, 0.0, 0.0]], [[-1.0, 0.0, 0.0, 0.0]]])
    qpos = np.array([nb * B - 1, nb * B - 1])            # own block 5, candidates 0..4
    sel = orc.moba_block_gate(q, k, qpos, B, 3)
    assert sel[0, 0].tolist() == [2, 3, 4, 5]
    assert sel[1, 0].tolist() == [0, 1, 2, 5]


def test_moba_with_all_blocks_equals_dense_causal():
    rng = np.random.default_rng(16)
    B, Tk, Tq, off = 8, 64, 16, 48
    q, k, v = rnd(rng, Tq, 2, 6), rnd(rng, Tk, 2, 6), rnd(rng, Tk, 2, 6)
    lay = orc.make_layout(Tq, Tk, True, off)
    sel = orc.moba_block_gate(q, k, lay.qpos, B, topk=Tk // B)
    O, LSE = orc.moba_attention(q, k, v, 0.3, lay, sel, B)
    Od, Ld = orc.dense_attention(q, k, v, 0.3, lay)
    np.testing.assert_allclose(O, Od, atol=1e-13, rtol=0)
    np.testing.assert_allclose(LSE, Ld, atol=1e-13, rtol=0)


def brute_gate_logical(q, k, kpos, qpos, B, topk):
    """Scalar gate whose blocks are runs of LOGICAL key positions: block b
    pools the stored rows j with kpos[j] // B == b (complete blocks only)."""
    Tq, Hq, D = q.shape
    Hkv = k.shape[1]
    nb = len(kpos) // B
    sel = np.full((Tq, Hq, topk + 1), -1, np.int32)
    for i in range(Tq):
        own = qpos[i] // B
        for h in range(Hq):
            g = h // (Hq // Hkv)
            gates = []
            for b in range(min(own, nb)):
                rows = [j for j in range(len(kpos)) if kpos[j] // B == b]
                mu = [math.fsum(k[j, g, d] for j in rows) / B for d in range(D)]
                gates.append((-math.fsum(q[i, h, d] * mu[d] for d in range(D)), b))
            chosen = sorted([b for _, b in sorted(gates)[:topk]] + [own])
            sel[i, h, :len(chosen)] = chosen
    return sel


def test_gate_with_a_kv_chunk_map_pools_logical_blocks():
    """Keys stored in zigzag order with blocks smaller than a chunk: the
    means pool logical blocks, so the selection equals scalar brute force
    over logical positions and equals the gate on the same keys stored in
    logical order ([CP] para 5)."""
    rng = np.random.default_rng(17)
    L, n_chunks, B, topk = 8, 6, 4, 2
    Tk = L * n_chunks
    cmap = np.array([0, 5, 1, 4, 2, 3])
    k_log = rnd(rng, Tk, 2, 5)
    q = rnd(rng, 7, 4, 5)
    phys_to_log = cmap[np.arange(Tk) // L] * L + np.arange(Tk) % L
    k_phys = k_log[phys_to_log]
    lay = orc.make_layout(7, Tk, True, 41, kv_chunk_map=cmap, chunk_len=L)
    sel = orc.moba_block_gate(q, k_phys, lay.qpos, B, topk, kpos=lay.kpos)
    np.testing.assert_array_equal(sel, brute_gate_logical(q, k_phys, lay.kpos, lay.qpos, B, topk))
    np.testing.assert_array_equal(sel, orc.moba_block_gate(q, k_log, lay.qpos, B, topk))
    # pooling physical rows instead would pick other blocks for this seed
    assert not np.array_equal(sel, orc.moba_block_gate(q, k_phys, lay.qpos, B, topk))
