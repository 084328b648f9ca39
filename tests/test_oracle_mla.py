"""Pins of the float64 MLA projection oracle (oracle.mla), CPU only.

* scalar brute force with math.fsum, written from the pages' description:
  the value up-projection per (token, head, channel) and the per-head K/V
  built channel by channel from wkv_b's rows;
* library routines in float64: torch.einsum for the per-head up-projection,
  torch.nn.functional.linear + view + split + cat for the materialisation;
* the identity the pages rest on (the absorbed path and the materialised
  path are the same attention): dense attention over materialised K/V
  equals attention over the latent with the key up-projection folded into
  the query, followed by the value up-projection - O and LSE alike.
"""

import math

import numpy as np
import torch

import oracle as orc
from oracle import mla


def test_v_up_matches_scalar_brute_force():
    rng = np.random.default_rng(1)
    T, H, L, V = 5, 3, 7, 4
    o = rng.standard_normal((T, H, L))
    w = rng.standard_normal((H, L, V))
    got = mla.absorbed_v_up(o, w)
    for t in range(T):
        for h in range(H):
            for v in range(V):
                ref = math.fsum(o[t, h, c] * w[h, c, v] for c in range(L))
                assert abs(got[t, h, v] - ref) <= 1e-13


def test_v_up_matches_torch_einsum():
    rng = np.random.default_rng(2)
    o = rng.standard_normal((33, 8, 64))
    w = rng.standard_normal((8, 64, 16))
    ref = torch.einsum("thl,hlv->thv", torch.from_numpy(o), torch.from_numpy(w)).numpy()
    np.testing.assert_allclose(mla.absorbed_v_up(o, w), ref, rtol=0, atol=1e-12)


def test_materialise_matches_scalar_brute_force():
    """Head h's output features are rows h*(N+V) .. (h+1)*(N+V)-1 of wkv_b; the
    first N are the non-positional key, the rest the value; the shared key is
    appended to every head's key."""
    rng = np.random.default_rng(3)
    T, H, L, N, V, R = 4, 3, 6, 2, 3, 2
    c = rng.standard_normal((T, L))
    ks = rng.standard_normal((T, R))
    wb = rng.standard_normal((H * (N + V), L))
    k, v = mla.materialise_kv(c, ks, wb, H, N, V)
    assert k.shape == (T, H, N + R) and v.shape == (T, H, V)
    for t in range(T):
        for h in range(H):
            for j in range(N):
                ref = math.fsum(c[t, x] * wb[h * (N + V) + j, x] for x in range(L))
                assert abs(k[t, h, j] - ref) <= 1e-13
            for j in range(R):
                assert k[t, h, N + j] == ks[t, j]
            for j in range(V):
                ref = math.fsum(c[t, x] * wb[h * (N + V) + N + j, x] for x in range(L))
                assert abs(v[t, h, j] - ref) <= 1e-13


def test_materialise_matches_torch_linear_view_split_cat():
    rng = np.random.default_rng(4)
    T, H, L, N, V, R = 40, 4, 32, 16, 8, 8
    c = torch.from_numpy(rng.standard_normal((T, L)))
    ks = torch.from_numpy(rng.standard_normal((T, R)))
    wb = torch.from_numpy(rng.standard_normal((H * (N + V), L)))
    kv = torch.nn.functional.linear(c, wb).view(T, H, N + V)
    k_nope, v_ref = kv.split([N, V], dim=-1)
    k_ref = torch.cat([k_nope, ks[:, None, :].expand(T, H, R)], dim=-1)
    k, v = mla.materialise_kv(c.numpy(), ks.numpy(), wb.numpy(), H, N, V)
    np.testing.assert_allclose(k, k_ref.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(v, v_ref.numpy(), rtol=0, atol=1e-12)


def test_absorbed_attention_equals_materialised_attention():
    """Causal attention of local queries at an offset: on materialised
    per-head K/V (scores q_nope . k_nope + q_rope . k_shared), and on the
    latent with W_uk folded into the query and W_uv applied after - the same
    O and LSE."""
    rng = np.random.default_rng(5)
    Tk, Tq, off, H, L, N, V, R = 48, 12, 36, 3, 10, 4, 5, 3
    c = rng.standard_normal((Tk, L))
    ks = rng.standard_normal((Tk, R))
    wb = rng.standard_normal((H * (N + V), L)) * 0.5
    q_nope = rng.standard_normal((Tq, H, N))
    q_rope = rng.standard_normal((Tq, H, R))
    scale = 0.3
    lay = orc.make_layout(Tq, Tk, True, off)
    k, v = mla.materialise_kv(c, ks, wb, H, N, V)
    O_mat, L_mat = orc.dense_attention(np.concatenate([q_nope, q_rope], axis=2), k, v, scale, lay)
    q_abs = mla.absorbed_query(q_nope, q_rope, wb, H, N, V)
    k_lat = np.concatenate([c, ks], axis=1)[:, None, :]          # one KV head: [latent | rope]
    v_lat = c[:, None, :]                                          # value = the latent
    O_lat, L_lat = orc.dense_attention(q_abs, k_lat, v_lat, scale, lay)
    O_abs = mla.absorbed_v_up(O_lat, mla.up_v_weight_of(wb, H, N, V))
    np.testing.assert_allclose(L_abs := L_lat, L_mat, rtol=0, atol=1e-12)
    np.testing.assert_allclose(O_abs, O_mat, rtol=0, atol=1e-12)
    assert np.isfinite(L_abs).all()
