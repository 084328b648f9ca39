"""Shared test helpers: comparison with tolerances and oracle layouts."""

import numpy as np
import torch

import oracle as orc
from context_attention_softmax_gb300 import inputs

# Tolerances against the float64 oracle.  bf16 inputs/outputs: the stated
# max-abs bounds (O 1e-2, LSE 1e-3).  fp32: 1e-5 on both (fp32 arithmetic over
# a few hundred keys stays far below it; the pages give no fp32 bound).
TOL = {"bf16": (1e-2, 1e-3), "fp32": (1e-5, 1e-5)}


def assert_matches(o_gpu, lse_gpu, o_ref, lse_ref, dtype, what=""):
    tol_o, tol_l = TOL[dtype]
    o = o_gpu.detach().float().cpu().numpy() if isinstance(o_gpu, torch.Tensor) else o_gpu
    ls = lse_gpu.detach().float().cpu().numpy() if isinstance(lse_gpu, torch.Tensor) else lse_gpu
    assert o.shape == o_ref.shape, (what, o.shape, o_ref.shape)
    assert not np.isnan(o).any() and not np.isnan(ls).any(), f"{what}: NaN in GPU output"
    ninf = np.isneginf(lse_ref)
    assert (np.isneginf(ls) == ninf).all(), f"{what}: -inf pattern of LSE differs"
    err_o = np.abs(o - o_ref).max() if o.size else 0.0
    err_l = np.abs(ls[~ninf] - lse_ref[~ninf]).max() if (~ninf).any() else 0.0
    assert err_o <= tol_o, f"{what}: max |dO| = {err_o:.3e} > {tol_o}"
    assert err_l <= tol_l, f"{what}: max |dLSE| = {err_l:.3e} > {tol_l}"
    return err_o, err_l


def layout_of(w: inputs.Workload):
    return orc.make_layout(w.Tq, w.Tk, w.causal, w.causal_offset, w.cu_seqlens, w.q_chunk_map,
                           w.kv_chunk_map, w.chunk_len)


def f64(w: inputs.Workload):
    return inputs.as_f64(w.q), inputs.as_f64(w.k), inputs.as_f64(w.v)


def sample_rows(n, k, seed=0, edges=()):
    rng = np.random.default_rng(seed)
    rows = set(int(x) for x in rng.choice(n, size=min(k, n), replace=False))
    rows.update(int(e) % n for e in edges if n)
    rows.update([0, n - 1])
    return np.array(sorted(rows), dtype=np.int64)


def to_gpu(w: inputs.Workload):
    """q, k, v on the GPU; v stays a view of k when it aliases k (absorbed MLA)."""
    d = torch.device("cuda")
    q, k = w.q.to(d), w.k.to(d)
    if w.v.untyped_storage().data_ptr() == w.k.untyped_storage().data_ptr():
        v = k[:, :, : w.v.shape[2]]
    else:
        v = w.v.to(d)
    return q, k, v


# Outputs of a bf16 GEMM (fp32 accumulation, one bf16 rounding of the result):
# the rounding is at most 2^-9 relative; the fp32 sums of K <= 1024 exact bf16
# products add at most K 2^-24 sum|a b|, far below that.  The bound used:
# |got - ref| <= 2^-8 |ref| + 1e-3 (twice the rounding, plus an absolute floor
# for results near zero).
def assert_gemm_close(got, ref, what=""):
    g = got.detach().float().cpu().numpy() if isinstance(got, torch.Tensor) else got
    assert g.shape == ref.shape, (what, g.shape, ref.shape)
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    bound = 2.0 ** -8 * np.abs(ref) + 1e-3
    bad = np.abs(g - ref) > bound
    assert not bad.any(), (f"{what}: {bad.sum()} elements beyond 2^-8|ref| + 1e-3, worst "
                           f"{np.abs(g - ref)[bad].max():.3e}")
