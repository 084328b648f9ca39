"""GPU parity of cpattn_chunk_bwd (dq, dk, dv) against the float64 oracle
(oracle.dense_attention_backward), through the C ABI.

The forward runs on the GPU first (its bf16 O and fp32 LSE are the
backward's inputs, as in training); the oracle differentiates the exact
global softmax of the same bf16 inputs.

Tolerance, elementwise, from the arithmetic of the GPU path (P[i, j] the
exact probabilities, g = d_out):
  * P and dS enter the gradient products rounded to bf16 (2^-9 relative
    each), so dv_j carries at most 2^-9 sum_i P_ij |g_i|, and dq_i, dk_j at
    most scale 2^-9 sum |dS_ij| |k_j| (resp. |q_i|);
  * D_i = <g_i, o_i> uses the forward's bf16 O, whose error per channel is
    at most 2^-9 (|o_id| + sum_j P_ij |v_jd|) (output rounding plus bf16 P
    in the forward), so dS_ij is off by at most P_ij |dD_i|, giving
    scale sum_j P_ij |dD_i| |k_j| in dq and scale sum_i P_ij |dD_i| |q_i| in dk;
  * fp32 accumulation and the exponential add relative errors near 2^-20.
Each bound is doubled (2^-8) and given a floor of 1e-5.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle as orc
import context_attention_softmax_gb300 as pkg
from context_attention_softmax_gb300 import cpattn_chunk_bwd, cpattn_chunk_fwd, inputs

from helpers import f64, layout_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from context_attention_softmax_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def _bounds(q, k, v, g, scale, lay):
    """The elementwise error bounds described in the module docstring."""
    Tq, Hq, _ = q.shape
    Hkv = k.shape[1]
    A = lay.allowed()
    b_dq = np.zeros(q.shape)
    b_dk = np.zeros(k.shape)
    b_dv = np.zeros(v.shape)
    u = 2.0 ** -8
    for h in range(Hq):
        gh = h // (Hq // Hkv)
        S = np.where(A, scale * (q[:, h] @ k[:, gh].T), -np.inf)
        m = np.where(A.any(1), S.max(1), 0.0)
        E = np.where(A, np.exp(S - m[:, None]), 0.0)
        ell = np.where(A.any(1), E.sum(1), 1.0)
        P = E / ell[:, None]
        o = P @ v[:, gh]
        dP = g[:, h] @ v[:, gh].T
        dS = P * (dP - (P * dP).sum(1, keepdims=True))
        dD = u * (np.abs(g[:, h]) * (np.abs(o) + P @ np.abs(v[:, gh]))).sum(1)
        b_dv[:, gh] += u * (P.T @ np.abs(g[:, h]))
        b_dq[:, h] = scale * (u * (np.abs(dS) @ np.abs(k[:, gh])) +
                              (P * dD[:, None]) @ np.abs(k[:, gh]))
        b_dk[:, gh] += scale * (u * (np.abs(dS).T @ np.abs(q[:, h])) +
                                (P * dD[:, None]).T @ np.abs(q[:, h]))
    return b_dq + 1e-5, b_dk + 1e-5, b_dv + 1e-5


def _check(name, got, ref, bound):
    g = got.detach().cpu().numpy()
    assert g.shape == ref.shape, (name, g.shape, ref.shape)
    assert np.isfinite(g).all(), f"{name}: non-finite"
    err = np.abs(g - ref)
    bad = err > bound
    assert not bad.any(), (f"{name}: {bad.sum()} of {bad.size} beyond the bound; worst excess "
                           f"{(err / bound).max():.2f}x, max |d| {err.max():.3e}")


def _run(w, seed=0, d_out_factor=0.5):
    q, k, v = (t.cuda() for t in (w.q, w.k, w.v))
    kw = dict(scale=w.scale, causal=w.causal, causal_offset=w.causal_offset,
              cu_seqlens=w.cu_seqlens, q_chunk_map=w.q_chunk_map, kv_chunk_map=w.kv_chunk_map,
              chunk_len=w.chunk_len)
    o, lse = cpattn_chunk_fwd(q, k, v, **kw)
    rng = np.random.default_rng(seed)
    g = inputs.to_device_dtype((rng.standard_normal(o.shape) * d_out_factor).astype(np.float32),
                               "bf16")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dq, dk, dv = cpattn_chunk_bwd(q, k, v, o, lse, g.cuda(), dev_status=status, **kw)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    qf, kf, vf = f64(w)
    lay = layout_of(w)
    gf = inputs.as_f64(g)
    rq, rk, rv = orc.dense_attention_backward(qf, kf, vf, w.scale, lay, gf)
    bq, bk, bv = _bounds(qf, kf, vf, gf, w.scale, lay)
    _check("dq", dq, rq, bq)
    _check("dk", dk, rk, bk)
    _check("dv", dv, rv, bv)
    return dq, dk, dv, rk, rv


@pytest.mark.parametrize("Tq,Tk,off,Hq,Hkv", [
    (300, 1000, 700, 4, 2),      # ragged tails on both sides, GQA
    (257, 1300, 700, 4, 1),      # keys 957.. never permitted: their dk, dv are zero
    (128, 640, 0, 2, 2),         # offset 0: the first query sees one key
    (600, 3000, 2500, 8, 2),     # several query tiles per key tile, 4 heads per group
])
def test_backward_small(Tq, Tk, off, Hq, Hkv):
    w = inputs.dense_gqa(seed=21, global_seq=Tq, cp_size=1, rank=0, Hq=Hq, Hkv=Hkv, Tk=Tk,
                         kv_chunks=0)
    w.causal_offset = off
    _, dk, dv, rk, rv = _run(w, seed=Tq)
    if Tk == 1300:
        assert (dk[957:] == 0).all() and (dv[957:] == 0).all()


def test_backward_noncausal_packed_with_queries_outside_sequences():
    w = inputs.dense_gqa(seed=22, global_seq=200, cp_size=1, rank=0, Hq=2, Hkv=2, Tk=333,
                         kv_chunks=0)
    w.causal = False
    w.causal_offset = 150
    w.cu_seqlens = np.array([0, 100, 160, 290], dtype=np.int32)   # positions >= 290 in no sequence
    dq, _, _, _, _ = _run(w, seed=5)
    assert (dq[140:] == 0).all()


def test_backward_zigzag_ranks():
    z = inputs.zigzag_varlen(seed=6, total=4096, n_seqs=3, len_lo=256, len_hi=2048, cp_size=4, H=4)
    for r in (0, 3):
        _run(z.rank_workload(r), seed=r)


def test_backward_full_size_headline():
    """The headline forward's workload (2048 queries at offset 4096 over 8192
    keys, GQA 16 / 4): every element of dq, dk and dv."""
    _run(inputs.dense_gqa(), seed=7)


def test_backward_empty_key_set():
    d = torch.device("cuda")
    q = torch.randn(16, 4, 128, device=d, dtype=torch.bfloat16)
    k0 = torch.randn(0, 2, 128, device=d, dtype=torch.bfloat16)
    o, lse = cpattn_chunk_fwd(q, k0, k0)
    g = torch.randn_like(q)
    dq, dk, dv = cpattn_chunk_bwd(q, k0, k0, o, lse, g)
    torch.cuda.synchronize()
    assert (dq == 0).all() and dk.shape == (0, 2, 128)
