"""Pins of the float64 backward oracle (oracle.dense_attention_backward), CPU.

* central finite differences of the forward oracle (dense_attention) along
  random directions, for q, k and v, under a causal offset, packed
  sequences (with a query outside every sequence), a zigzag chunk map and
  GQA;
* torch autograd in float64 through scaled_dot_product_attention (no mask,
  and causal with Tq == Tk) with GQA expanded by repeat_interleave;
* invariants: the GQA gradient of a KV head is the sum of the gradients of
  its query heads' copies; a row with no permitted key gets no gradient and
  gives none.
"""

import numpy as np
import pytest
import torch

import oracle as orc


def _rnd(rng, *shape):
    return rng.standard_normal(shape)


def _loss(q, k, v, scale, lay, g):
    O, _ = orc.dense_attention(q, k, v, scale, lay)
    return float((O * g).sum())


@pytest.mark.parametrize("name", ["offset", "packed", "zigzag", "gqa_noncausal"])
def test_gradients_match_central_differences(name):
    rng = np.random.default_rng({"offset": 1, "packed": 2, "zigzag": 3, "gqa_noncausal": 4}[name])
    Hq, Hkv, D, Dv = 4, 2, 5, 3
    if name == "offset":
        Tq, Tk = 6, 14
        lay = orc.make_layout(Tq, Tk, True, 8)
    elif name == "packed":
        Tq, Tk = 9, 16
        lay = orc.make_layout(Tq, Tk, True, 6, cu_seqlens=np.array([0, 5, 11, 14]))
    elif name == "zigzag":
        Tq, Tk = 8, 16
        lay = orc.make_layout(Tq, Tk, True, 0, q_chunk_map=np.array([1, 2]),
                              kv_chunk_map=np.array([0, 3, 1, 2]), chunk_len=4)
    else:
        Tq, Tk = 5, 7
        lay = orc.make_layout(Tq, Tk, False, 0)
    q, k, v = _rnd(rng, Tq, Hq, D), _rnd(rng, Tk, Hkv, D), _rnd(rng, Tk, Hkv, Dv)
    g = _rnd(rng, Tq, Hq, Dv)
    scale = 0.45
    dq, dk, dv = orc.dense_attention_backward(q, k, v, scale, lay, g)
    eps = 1e-5
    for which, x, dx in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        for _ in range(3):
            u = _rnd(rng, *x.shape)
            args = {"q": q, "k": k, "v": v}
            plus = dict(args, **{which: x + eps * u})
            minus = dict(args, **{which: x - eps * u})
            fd = (_loss(plus["q"], plus["k"], plus["v"], scale, lay, g) -
                  _loss(minus["q"], minus["k"], minus["v"], scale, lay, g)) / (2 * eps)
            assert abs(fd - float((dx * u).sum())) <= 1e-7 * (1 + abs(fd)), (name, which)


@pytest.mark.parametrize("causal", [False, True])
def test_gradients_match_torch_autograd_sdpa(causal):
    rng = np.random.default_rng(5 + causal)
    T, Hq, Hkv, D = 11, 4, 2, 6
    q, k, v = _rnd(rng, T, Hq, D), _rnd(rng, T, Hkv, D), _rnd(rng, T, Hkv, D)
    g = _rnd(rng, T, Hq, D)
    scale = 0.37
    lay = orc.make_layout(T, T, causal, 0)
    dq, dk, dv = orc.dense_attention_backward(q, k, v, scale, lay, g)
    tq = torch.tensor(q.transpose(1, 0, 2)[None], requires_grad=True)
    tk = torch.tensor(k.transpose(1, 0, 2)[None], requires_grad=True)
    tv = torch.tensor(v.transpose(1, 0, 2)[None], requires_grad=True)
    rep = Hq // Hkv
    o = torch.nn.functional.scaled_dot_product_attention(
        tq, tk.repeat_interleave(rep, dim=1), tv.repeat_interleave(rep, dim=1),
        is_causal=causal, scale=scale)
    o.backward(torch.tensor(g.transpose(1, 0, 2)[None]))
    np.testing.assert_allclose(dq, tq.grad[0].numpy().transpose(1, 0, 2), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk, tk.grad[0].numpy().transpose(1, 0, 2), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dv, tv.grad[0].numpy().transpose(1, 0, 2), rtol=0, atol=1e-12)


def test_gqa_gradient_is_the_sum_over_the_group():
    rng = np.random.default_rng(9)
    Tq, Tk, Hq, Hkv, D = 5, 9, 4, 2, 4
    lay = orc.make_layout(Tq, Tk, True, 4)
    q, k, v, g = _rnd(rng, Tq, Hq, D), _rnd(rng, Tk, Hkv, D), _rnd(rng, Tk, Hkv, D), _rnd(rng, Tq, Hq, D)
    _, dk, dv = orc.dense_attention_backward(q, k, v, 0.5, lay, g)
    kr, vr = np.repeat(k, 2, axis=1), np.repeat(v, 2, axis=1)
    _, dkr, dvr = orc.dense_attention_backward(q, kr, vr, 0.5, lay, g)
    np.testing.assert_allclose(dk, dkr[:, 0::2] + dkr[:, 1::2], rtol=0, atol=1e-13)
    np.testing.assert_allclose(dv, dvr[:, 0::2] + dvr[:, 1::2], rtol=0, atol=1e-13)


def test_rows_without_keys_get_and_give_no_gradient():
    rng = np.random.default_rng(10)
    Tq, Tk, H, D = 6, 8, 1, 3
    lay = orc.make_layout(Tq, Tk, True, 3, cu_seqlens=np.array([0, 6]))   # qpos 6.. in no sequence
    q, k, v, g = _rnd(rng, Tq, H, D), _rnd(rng, Tk, H, D), _rnd(rng, Tk, H, D), _rnd(rng, Tq, H, D)
    dq, dk, dv = orc.dense_attention_backward(q, k, v, 0.5, lay, g)
    assert (dq[3:] == 0).all()
    g2 = g.copy()
    g2[3:] = 7.0                                     # their upstream gradient changes nothing
    dq2, dk2, dv2 = orc.dense_attention_backward(q, k, v, 0.5, lay, g2)
    np.testing.assert_array_equal(dk, dk2)
    np.testing.assert_array_equal(dv, dv2)
    assert (dk[6:] == 0).all() and (dv[6:] == 0).all()   # keys no query may see
