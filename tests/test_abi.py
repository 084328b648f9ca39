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
