"""C-ABI checks that need no GPU: the library loads, exports every symbol the
header declares, the ctypes struct matches the C layout, and host-side
validation rejects bad arguments before any launch."""

import ctypes
import os
import re
import subprocess
import tempfile

import pytest

from context_attention_softmax_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "cpattn.h")


@pytest.fixture(scope="module")
def lib():
    from context_attention_softmax_gb300 import build
    build.build()
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(cpattn_\w+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert set(names) == set(_lib.EXPORTS)
    for n in names:
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.LIB_PATH], capture_output=True,
                         text=True).stdout
    exported = set(re.findall(r" T (cpattn_\w+)", out))
    assert set(names) <= exported


def test_struct_layout_matches_c():
    fields = [f for f, _ in _lib.AttnArgs._fields_]
    src = ['#include <stdio.h>', '#include <stddef.h>', '#include "cpattn.h"', 'int main(void){',
           'printf("%zu\\n", sizeof(cpattn_attn_args));']
    src += [f'printf("%zu\\n", offsetof(cpattn_attn_args, {f}));' for f in fields]
    src += ["return 0;}"]
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "layout.c")
        exe = os.path.join(d, "layout")
        open(c, "w").write("\n".join(src))
        subprocess.run(["gcc", "-std=c11", "-I", os.path.dirname(HEADER), c, "-o", exe], check=True)
        vals = [int(x) for x in subprocess.run([exe], capture_output=True, text=True).stdout.split()]
    assert vals[0] == ctypes.sizeof(_lib.AttnArgs)
    assert vals[1:] == [getattr(_lib.AttnArgs, f).offset for f in fields]


def test_version_and_empty_error(lib):
    assert lib.cpattn_version() == 110


def _valid_args():
    a = _lib.AttnArgs()
    a.dtype = _lib.CPATTN_BF16
    a.q, a.q_stride_t, a.q_stride_h, a.Tq, a.Hq, a.Dqk = 0x10000, 16 * 128, 128, 64, 16, 128
    a.k, a.k_stride_t, a.k_stride_h, a.Tk, a.Hkv = 0x20000, 4 * 128, 128, 256, 4
    a.v, a.v_stride_t, a.v_stride_h, a.Dv = 0x30000, 4 * 128, 128, 128
    a.o, a.o_stride_t, a.o_stride_h = 0x40000, 16 * 128, 128
    a.scale, a.causal = 0.088, 1
    return a


def _call(lib, a):
    return lib.cpattn_chunk_fwd(ctypes.byref(a), None, 0, None)


@pytest.mark.parametrize("mutate,status,msg", [
    (lambda a: setattr(a, "dtype", 7), 1, "dtype"),
    (lambda a: setattr(a, "Hkv", 3), 1, "multiple of Hkv"),
    (lambda a: setattr(a, "Dqk", 12), 1, "Dqk"),
    (lambda a: setattr(a, "Dqk", 2048), 2, "exceeds"),
    (lambda a: setattr(a, "Dv", 1024), 2, "Dv"),
    (lambda a: setattr(a, "q", 0x10008), 1, "aligned"),
    (lambda a: setattr(a, "k_stride_h", 4), 1, "16 bytes"),
    (lambda a: setattr(a, "o", None), 1, "o is NULL"),
    (lambda a: setattr(a, "causal", 2), 1, "causal"),
    (lambda a: setattr(a, "causal_offset", -1), 1, "causal_offset"),
    (lambda a: setattr(a, "scale", float("nan")), 1, "scale"),
    (lambda a: (setattr(a, "kv_chunk_map", 0x5000), setattr(a, "chunk_len", 0)), 1, "chunk_len"),
    (lambda a: (setattr(a, "kv_chunk_map", 0x5000), setattr(a, "chunk_len", 100),
                setattr(a, "n_kv_chunks", 2)), 1, "Tk"),
    (lambda a: setattr(a, "kv_chunk_len", 64), 1, "partial"),
    (lambda a: (setattr(a, "cu_seqlens", 0x6000), setattr(a, "num_seqs", 0)), 1, "num_seqs"),
])
def test_chunk_fwd_rejects_bad_arguments(lib, mutate, status, msg):
    a = _valid_args()
    mutate(a)
    assert _call(lib, a) == status
    assert msg in lib.cpattn_last_error().decode()


def test_null_args_rejected(lib):
    assert lib.cpattn_chunk_fwd(None, None, 0, None) == 1
    assert lib.cpattn_topk_sparse_fwd(None, None, 0, 1, 1, None, 0, None) == 1
    assert lib.cpattn_block_gate(None, 512, 3, None, None, 0, None) == 1
    assert lib.cpattn_workspace_size(2, None, 3, 512) == 0


def test_sparse_and_gate_validation(lib):
    a = _valid_args()
    assert lib.cpattn_topk_sparse_fwd(ctypes.byref(a), 0x7000, 8, 3, 1, None, 0, None) == 1
    assert "index_heads" in lib.cpattn_last_error().decode()
    assert lib.cpattn_topk_sparse_fwd(ctypes.byref(a), 0x7000, 8, 1, 0, None, 0, None) == 1
    assert lib.cpattn_topk_sparse_fwd(ctypes.byref(a), None, 8, 1, 1, None, 0, None) == 1
    a.kv_chunk_len = 64
    assert lib.cpattn_topk_sparse_fwd(ctypes.byref(a), 0x7000, 8, 1, 1, None, 0, None) == 2
    g = _valid_args()
    need = lib.cpattn_workspace_size(2, ctypes.byref(g), 3, 64)
    # fp64 + fp32 block means, plus the three bf16 mean terms and the fp32
    # mean norms of the tensor-core gate
    assert need == (256 // 64) * 4 * (128 * (12 + 6) + 4)
    assert lib.cpattn_block_gate(ctypes.byref(g), 64, 3, 0x8000, None, 0, None) == 4
    assert lib.cpattn_block_gate(ctypes.byref(g), 64, 65, 0x8000, 0x9000, need, None) == 2
    g.cu_seqlens, g.num_seqs = 0x6000, 2
    assert lib.cpattn_block_gate(ctypes.byref(g), 64, 3, 0x8000, 0x9000, need, None) == 2
    assert lib.cpattn_lse_merge(2, 0x1000, 0x2000, 4, 2, 12, 0x3000, 1, 24, 12, None, None) == 1
    assert lib.cpattn_lse_merge(2, 0x1000, 0x2000, 4, 2, 16, 0x3000, 5, 32, 16, None, None) == 1


def _indexer_args():
    a = _lib.AttnArgs()
    a.dtype = _lib.CPATTN_FP32
    a.q, a.q_stride_t, a.q_stride_h, a.Tq, a.Hq, a.Dqk = 0x10000, 4 * 128, 128, 64, 4, 128
    a.k, a.k_stride_t, a.k_stride_h, a.Tk, a.Hkv = 0x20000, 128, 128, 256, 1
    a.scale, a.causal = 1.0, 1
    return a


@pytest.mark.parametrize("mutate,topk,status,msg", [
    (lambda a: setattr(a, "dtype", _lib.CPATTN_BF16), 16, 2, "CPATTN_FP32"),
    (lambda a: (setattr(a, "Hq", 4), setattr(a, "Hkv", 2)), 16, 1, "one head"),
    (lambda a: (setattr(a, "Hq", 32), setattr(a, "q_stride_t", 32 * 128)), 16, 2, "exceed 16"),
    (lambda a: (setattr(a, "Dqk", 512), setattr(a, "q_stride_h", 512), setattr(a, "q_stride_t", 4 * 512),
                setattr(a, "k_stride_t", 512), setattr(a, "k_stride_h", 512)), 16, 2, "exceeds 256"),
    (lambda a: (setattr(a, "kv_chunk_map", 0x5000), setattr(a, "chunk_len", 128),
                setattr(a, "n_kv_chunks", 2)), 16, 2, "logical order"),
    (lambda a: None, 0, 1, "topk=0"),
    (lambda a: None, 257, 1, "topk=257"),
])
def test_indexer_rejects_bad_arguments(lib, mutate, topk, status, msg):
    """Host validation of the indexer call: nothing is launched on rejection."""
    a = _indexer_args()
    mutate(a)
    assert lib.cpattn_dsa_indexer(ctypes.byref(a), 0x7000, topk, 0x8000, None, 0, None) == status
    assert msg in lib.cpattn_last_error().decode()


def test_indexer_needs_weights_outputs_and_its_workspace(lib):
    a = _indexer_args()
    assert lib.cpattn_dsa_indexer(ctypes.byref(a), None, 16, 0x8000, None, 0, None) == 1
    assert "w is NULL" in lib.cpattn_last_error().decode()
    assert lib.cpattn_dsa_indexer(ctypes.byref(a), 0x7000, 16, None, None, 0, None) == 1
    assert "indices is NULL" in lib.cpattn_last_error().decode()
    need = lib.cpattn_workspace_size(_lib.OP_DSA_INDEXER, ctypes.byref(a), 16, 1)
    # fp32 scores [Tq, Tk] and the two norm vectors come first
    assert need >= 64 * 256 * 4 + 256 * 4 + 64 * 4
    assert lib.cpattn_dsa_indexer(ctypes.byref(a), 0x7000, 16, 0x8000, None, 0, None) == 4
    assert lib.cpattn_dsa_indexer(ctypes.byref(a), 0x7000, 16, 0x8000, 0x9000, need - 1, None) == 4
    assert lib.cpattn_dsa_indexer(ctypes.byref(a), 0x7000, 16, 0x8000, 0x9008, need, None) == 1
    assert "aligned" in lib.cpattn_last_error().decode()
    a.Tq = 0     # nothing to select: no workspace needed
    assert lib.cpattn_workspace_size(_lib.OP_DSA_INDEXER, ctypes.byref(a), 16, 1) == 0


def test_indexer_workspace_holds_the_tensor_core_operands(lib):
    """D = 128 (the tensor-core scores) needs, beyond what D = 64 needs, the
    bf16 split operands [Tq * H, 256] and [Tk, 256] and one 16-byte key
    interval per 128-row tile, each region 256-byte aligned."""
    def need(D):
        a = _indexer_args()
        a.Dqk, a.q_stride_h, a.q_stride_t, a.k_stride_t, a.k_stride_h = D, D, 4 * D, D, D
        return lib.cpattn_workspace_size(_lib.OP_DSA_INDEXER, ctypes.byref(a), 16, 1)

    up = lambda x: (x + 255) // 256 * 256
    rows, Tk = 64 * 4, 256
    split = up(up(rows * 256 * 2) + Tk * 256 * 2) + (rows + 127) // 128 * 16 + 256
    assert need(128) - need(64) == split


def _bwd_call(lib, a, d_out=0x90000, dq=0xA0000, dk=0xB0000, dv=0xC0000):
    return lib.cpattn_chunk_bwd(ctypes.byref(a), d_out, 16 * 128, 128, dq, 16 * 128, 128,
                                dk, 4 * 128, 128, dv, 4 * 128, 128, None, 0, None)


@pytest.mark.parametrize("mutate,kw,status,msg", [
    (lambda a: setattr(a, "lse", None), {}, 1, "lse (the forward's) is NULL"),
    (lambda a: None, {"dq": None}, 1, "dq"),
    (lambda a: None, {"d_out": None}, 1, "d_out"),
    (lambda a: None, {"dk": None}, 1, "dk"),
    (lambda a: setattr(a, "dtype", _lib.CPATTN_FP32), {}, 2, "bf16"),
    (lambda a: (setattr(a, "Dv", 64), setattr(a, "v_stride_h", 64)), {}, 2, "head dims 128"),
    (lambda a: (setattr(a, "kv_chunk_len", 128), setattr(a, "partial_o", 0x50000),
                setattr(a, "partial_lse", 0x58000)), {}, 1, "kv_chunk_len = 0"),
])
def test_chunk_bwd_rejects_bad_arguments(lib, mutate, kw, status, msg):
    """Host validation of the backward: nothing is launched on rejection."""
    a = _valid_args()
    a.lse = 0x48000
    mutate(a)
    assert _bwd_call(lib, a, **kw) == status
    assert msg in lib.cpattn_last_error().decode()


def test_chunk_bwd_with_no_queries_and_no_keys_is_a_no_op(lib):
    a = _valid_args()
    a.Tq, a.Tk = 0, 0
    assert _bwd_call(lib, a, d_out=None, dq=None, dk=None, dv=None) == 0


def _v_up(lib, o=0x10000, w=0x20000, T=8, H=4, L=512, V=128, out=0x30000, limit=0):
    return lib.cpattn_mla_v_up(o, H * L, L, w, T, H, L, V, out, H * V, V, None, limit, None)


@pytest.mark.parametrize("kw,status,msg", [
    ({"L": 32}, 2, "L=32"),
    ({"V": 64}, 2, "V=64"),
    ({"H": 0}, 1, "H=0"),
    ({"T": -1}, 1, "T=-1"),
    ({"limit": -1}, 1, "wait_limit_ns"),
    ({"w": None}, 1, "up_v_weight"),
    ({"w": 0x20008}, 1, "up_v_weight"),
    ({"o": None}, 1, "o_latent"),
    ({"out": None}, 1, "out"),
])
def test_mla_v_up_rejects_bad_arguments(lib, kw, status, msg):
    assert _v_up(lib, **kw) == status
    assert msg in lib.cpattn_last_error().decode()


def test_mla_v_up_with_no_tokens_is_a_no_op(lib):
    assert _v_up(lib, o=None, w=None, T=0, out=None) == 0


def _kv(lib, c=0x10000, ks=0x20000, wb=0x30000, T=8, L=512, H=4, N=128, R=64, V=128,
        k=0x40000, v=0x50000, c_st=None, limit=0):
    c_st = L if c_st is None else c_st
    return lib.cpattn_mla_kv_materialise(c, c_st, ks, R, wb, T, L, H, N, R, V,
                                         k, H * (N + R), N + R, v, H * V, V, None, limit, None)


@pytest.mark.parametrize("kw,status,msg", [
    ({"R": 4}, 2, "R=4"),
    ({"N": 64}, 2, "N=64"),
    ({"V": 192}, 2, "V=192"),
    ({"L": 96}, 2, "L=96"),
    ({"H": 0}, 1, "H=0"),
    ({"limit": -1}, 1, "wait_limit_ns"),
    ({"c": None}, 1, "kv_c"),
    ({"c_st": 500}, 1, "kv_c"),
    ({"wb": 0x30008}, 1, "wkv_b"),
    ({"ks": None}, 1, "k_shared"),
    ({"k": None}, 1, "k_out"),
    ({"v": None}, 1, "v_out"),
])
def test_mla_kv_materialise_rejects_bad_arguments(lib, kw, status, msg):
    assert _kv(lib, **kw) == status
    assert msg in lib.cpattn_last_error().decode()


def test_mla_kv_materialise_without_shared_key_and_with_no_tokens(lib):
    # R = 0: k_shared is never read, so NULL is valid; T = 0 launches nothing
    assert _kv(lib, c=None, ks=None, wb=None, T=0, k=None, v=None) == 0
    assert _kv(lib, T=0, R=0, ks=None) == 0
