"""Float64 CPU oracle for the multi-latent-attention (MLA) projections around
the CP-chunk attention: the value up-projection after absorbed attention and
the local materialisation of per-head K/V from gathered latents.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke check
of ``__graft_entry__`` and the ``cpu_baseline`` / ``--impl reference`` legs of
``bench.py`` may import or run it.  It shares no code with the CUDA library
and imports nothing from it.

Sources, by page title and section:

[DSA-THD] "[1/2] Enable DSA CP, THD with absorbed MLA - #3674", sequence
          diagram (after the sparse gather the attention output of each head
          is multiplied by the value up-projection, ``up_v_weight``, giving
          ``v_channels`` per head) and "Background" (matrix absorption: the
          key up-projection is folded into the query, attention runs on the
          latent, and the value up-projection is applied after attention).
[MLA-CP]  "[BC][MLA][CP] Optimize MLA all-gather and Ulysses communication
          for Kimi K3 and dpskV3", section "K/V all-gather CP": after the
          compressed latents kv_c (T x L) and the head-shared key k_shared
          (T x R) are gathered, each rank applies wkv_b to get T x H x (N + V),
          unpacks it into k_nope (T x H x N) and v (T x H x V), and builds
          k = concat(k_nope, k_shared repeated over the heads) (T x H x (N+R)).
          The page's parity table reports that attention on the materialised
          K/V and the compact (latent) path agree.

Readings taken where the pages are silent:
  * up_v_weight is laid out [H, L, V]: head h maps its L latent channels to
    V value channels, out[t, h, :] = o_latent[t, h, :] @ up_v_weight[h];
  * wkv_b is a linear layer's weight [H * (N + V), L] (output features by
    input features); output feature h * (N + V) + c is channel c of head h,
    the first N of them the non-positional key, the last V the value.
"""

from __future__ import annotations

import numpy as np


def absorbed_v_up(o_latent, up_v_weight):
    """Value up-projection after absorbed attention ([DSA-THD] diagram).

    out[t, h, :] = o_latent[t, h, :] @ up_v_weight[h] for every token t and
    head h.  o_latent: [T, H, L], up_v_weight: [H, L, V] -> [T, H, V] float64.
    """
    o = np.asarray(o_latent, np.float64)
    w = np.asarray(up_v_weight, np.float64)
    T, H, L = o.shape
    out = np.empty((T, H, w.shape[2]))
    for h in range(H):
        out[:, h, :] = o[:, h, :] @ w[h]
    return out


def materialise_kv(kv_c, k_shared, wkv_b, H, N, V):
    """Per-head K and V from gathered latents ([MLA-CP] "K/V all-gather CP").

    kv = kv_c @ wkv_b^T, viewed [T, H, N + V]; k_nope = kv[..., :N],
    v = kv[..., N:]; k = concat(k_nope, k_shared repeated for each head).
    kv_c: [T, L], k_shared: [T, R], wkv_b: [H * (N + V), L].
    Returns k [T, H, N + R], v [T, H, V] float64.
    """
    c = np.asarray(kv_c, np.float64)
    ks = np.asarray(k_shared, np.float64)
    wb = np.asarray(wkv_b, np.float64)
    T = c.shape[0]
    kv = (c @ wb.T).reshape(T, H, N + V)
    k_nope, v = kv[:, :, :N], kv[:, :, N:]
    k = np.concatenate([k_nope, np.broadcast_to(ks[:, None, :], (T, H, ks.shape[1]))], axis=2)
    return k, v.copy()


def absorbed_query(q_nope, q_rope, wkv_b, H, N, V):
    """The query of absorbed attention ([DSA-THD] "Background"): the key
    up-projection of head h (rows h*(N+V) .. h*(N+V)+N-1 of wkv_b, W_uk [N, L])
    folded into the query, q_abs[t, h] = concat(q_nope[t, h] @ W_uk_h, q_rope[t, h]).
    q_nope: [T, H, N], q_rope: [T, H, R] -> [T, H, L + R]."""
    wb = np.asarray(wkv_b, np.float64)
    qn = np.asarray(q_nope, np.float64)
    out = []
    for h in range(H):
        w_uk = wb[h * (N + V): h * (N + V) + N, :]
        out.append(qn[:, h, :] @ w_uk)
    return np.concatenate([np.stack(out, axis=1), np.asarray(q_rope, np.float64)], axis=2)


def up_v_weight_of(wkv_b, H, N, V):
    """up_v_weight [H, L, V] of the value rows of wkv_b: W_uv_h^T, with
    W_uv_h = rows h*(N+V)+N .. (h+1)*(N+V)-1 of wkv_b ([V, L])."""
    wb = np.asarray(wkv_b, np.float64)
    return np.stack([wb[h * (N + V) + N:(h + 1) * (N + V), :].T for h in range(H)], axis=0)
