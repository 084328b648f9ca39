"""GPU parity of the MLA projections (cpattn_mla_v_up, cpattn_mla_kv_materialise)
against the float64 oracle (oracle.mla), through the C ABI.

Small cases span several 128-row tiles with a ragged tail, more than one
128-column tile per head and latent widths of one and of several 64-wide
steps; the full-size workloads run in the bench's launch configuration and
are compared on sampled rows (all heads and channels).  Outputs are bf16
from fp32 accumulation: the tolerance is 2^-8 |ref| + 1e-3 (tests/helpers.py).
"""

import numpy as np
import pytest
import torch

from oracle import mla
from context_attention_softmax_gb300 import (cpattn_chunk_fwd, cpattn_mla_kv_materialise,
                                             cpattn_mla_v_up, cpattn_topk_sparse_fwd, inputs)

from helpers import assert_gemm_close, assert_matches, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from context_attention_softmax_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def f64(t):
    return inputs.as_f64(t)


@pytest.mark.parametrize("T,H,L,V", [
    (300, 3, 128, 128),     # ragged last row tile, two K steps
    (129, 2, 512, 256),     # two column tiles per head, eight K steps
    (64, 5, 64, 128),       # fewer rows than one tile, one K step
])
def test_v_up_small(T, H, L, V):
    w = inputs.mla_v_up(seed=T + H, T=T, H=H, L=L, V=V)
    got = cpattn_mla_v_up(w.o_latent.cuda(), w.up_v_weight.cuda())
    ref = mla.absorbed_v_up(f64(w.o_latent), f64(w.up_v_weight))
    assert_gemm_close(got, ref, f"v_up {T}x{H}x{L}x{V}")


def test_v_up_strided_latent_and_output():
    """o_latent read through row and head strides (a view of a wider buffer)
    and the output written into a strided view."""
    w = inputs.mla_v_up(seed=5, T=200, H=4, L=128, V=128)
    big = torch.zeros((200, 6, 192), dtype=torch.bfloat16, device="cuda")
    big[:, 1:5, 32:160] = w.o_latent.cuda()
    o_view = big[:, 1:5, 32:160]
    out_big = torch.full((200, 4, 256), 7.0, dtype=torch.bfloat16, device="cuda")
    out_view = out_big[:, :, 64:192]
    cpattn_mla_v_up(o_view, w.up_v_weight.cuda(), out=out_view)
    ref = mla.absorbed_v_up(f64(w.o_latent), f64(w.up_v_weight))
    assert_gemm_close(out_view, ref, "v_up strided")
    assert (out_big[:, :, :64] == 7).all() and (out_big[:, :, 192:] == 7).all()


def test_v_up_full_size_sampled():
    w = inputs.mla_v_up()
    got = cpattn_mla_v_up(w.o_latent.cuda(), w.up_v_weight.cuda())
    rows = sample_rows(w.o_latent.shape[0], 96, edges=(127, 128, 4095))
    ref = mla.absorbed_v_up(f64(w.o_latent[rows]), f64(w.up_v_weight))
    assert_gemm_close(got[rows.tolist()], ref, "v_up full")


@pytest.mark.parametrize("T,H,L,N,V,R", [
    (300, 3, 128, 128, 128, 64),    # ragged rows, shared key appended to every head
    (200, 2, 512, 256, 128, 8),     # two key tiles per head, a narrow shared key
    (130, 2, 64, 128, 256, 0),      # no shared key, two value tiles per head
    (100, 1, 128, 128, 256, 16),    # three 128-column halves: the last 256-wide tile half empty
    (150, 2, 576, 128, 128, 64),    # latent wider than 512: the kernel without a resident A block
])
def test_kv_materialise_small(T, H, L, N, V, R):
    w = inputs.mla_kv(seed=T + L, T=T, H=H, L=L, N=N, V=V, R=R)
    k, v = cpattn_mla_kv_materialise(w.kv_c.cuda(), w.k_shared.cuda(), w.wkv_b.cuda(), H, N, V)
    kr, vr = mla.materialise_kv(f64(w.kv_c), f64(w.k_shared), f64(w.wkv_b), H, N, V)
    assert_gemm_close(k, kr, "k")
    assert_gemm_close(v, vr, "v")
    if R:
        assert torch.equal(k[:, :, N:].cpu(), w.k_shared[:, None, :].expand(T, H, R))


def test_kv_materialise_full_size_sampled():
    w = inputs.mla_kv()
    k, v = cpattn_mla_kv_materialise(w.kv_c.cuda(), w.k_shared.cuda(), w.wkv_b.cuda(), w.H, w.N, w.V)
    rows = sample_rows(w.kv_c.shape[0], 64, edges=(127, 128, 32767))
    kr, vr = mla.materialise_kv(f64(w.kv_c[rows]), f64(w.k_shared[rows]), f64(w.wkv_b), w.H, w.N, w.V)
    assert_gemm_close(k[rows.tolist()], kr, "k full")
    assert_gemm_close(v[rows.tolist()], vr, "v full")


def test_absorbed_and_materialised_paths_end_to_end():
    """Both MLA paths on the GPU, each against the oracle on the same inputs:
    attention on the latent with W_uk folded into the query (the DSA kernel's
    absorbed shape, every permitted key selected) followed by cpattn_mla_v_up;
    and dense attention over the K/V that cpattn_mla_kv_materialise builds.
    (That the two paths compute the same attention is pinned on the oracle,
    tests/test_oracle_mla.py.)"""
    import oracle as orc
    rng = np.random.default_rng(3)
    Tk, Tq, off, H, L, N, V, R = 700, 40, 660, 128, 512, 128, 128, 64
    c = inputs.to_device_dtype(rng.standard_normal((Tk, L)).astype(np.float32), "bf16")
    ks = inputs.to_device_dtype(rng.standard_normal((Tk, R)).astype(np.float32), "bf16")
    wb = inputs.to_device_dtype((rng.standard_normal((H * (N + V), L)) / np.sqrt(L) * 0.5)
                                .astype(np.float32), "bf16")
    q_nope = rng.standard_normal((Tq, H, N)) * 0.5
    q_rope = rng.standard_normal((Tq, H, R)) * 0.5
    scale = 1.0 / np.sqrt(N + R)
    # the absorbed query, rounded to bf16 as the kernel receives it
    q_abs = inputs.to_device_dtype(mla.absorbed_query(q_nope, q_rope, f64(wb), H, N, V)
                                   .astype(np.float32), "bf16")
    kv = torch.cat([c, ks], dim=1)[:, None, :].contiguous()          # [Tk, 1, 576]
    idx = torch.full((Tq, 1, 2048), -1, dtype=torch.int32)
    for i in range(Tq):
        idx[i, 0, :off + i + 1] = torch.arange(off + i + 1, dtype=torch.int32)
    kvd = kv.cuda()
    o_lat, lse = cpattn_topk_sparse_fwd(q_abs.cuda(), kvd, kvd[:, :, :L], idx, block_size=1,
                                        scale=scale, causal_offset=off)
    w_uv = inputs.to_device_dtype(mla.up_v_weight_of(f64(wb), H, N, V).astype(np.float32), "bf16")
    out = cpattn_mla_v_up(o_lat, w_uv.cuda())
    # reference: the oracle's attention on materialised K/V from the same
    # bf16 latents and weights, with the query the absorbed one represents
    lay = orc.make_layout(Tq, Tk, True, off)
    k_m, v_m = mla.materialise_kv(f64(c), f64(ks), f64(wb), H, N, V)
    O_lat, L_ref = orc.dense_attention(f64(q_abs), f64(kv), f64(kv)[:, :, :L], scale, lay)
    O_ref = mla.absorbed_v_up(O_lat, f64(w_uv))
    assert_matches(out, lse, O_ref, L_ref, "bf16", "absorbed path end to end")
    # the materialised path on the GPU: K/V from cpattn_mla_kv_materialise,
    # then dense attention of the un-absorbed query over them
    k_g, v_g = cpattn_mla_kv_materialise(c.cuda(), ks.cuda(), wb.cuda(), H, N, V)
    assert_gemm_close(k_g, k_m, "materialised k")
    assert_gemm_close(v_g, v_m, "materialised v")
    q_mat = inputs.to_device_dtype(np.concatenate([q_nope, q_rope], axis=2).astype(np.float32),
                                   "bf16")
    o_m, lse_m = cpattn_chunk_fwd(q_mat.cuda(), k_g, v_g, scale=scale, causal=True,
                                  causal_offset=off)
    O_m, L_m = orc.dense_attention(f64(q_mat), f64(k_g), f64(v_g), scale, lay)
    assert_matches(o_m, lse_m, O_m, L_m, "bf16", "materialised path end to end")
