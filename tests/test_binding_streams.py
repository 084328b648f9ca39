"""Host logic of the Python binding that needs no GPU: a call given a
`stream` (by keyword or by position) runs with that stream as torch's
current one, and a call without one leaves the current stream alone."""

import contextlib
import inspect

import pytest

import context_attention_softmax_gb300 as pkg


ENTRY_POINTS = ["cpattn_chunk_fwd", "cpattn_chunk_bwd", "cpattn_lse_merge", "cpattn_topk_sparse_fwd",
                "cpattn_block_gate", "cpattn_dsa_indexer", "cpattn_mla_v_up",
                "cpattn_mla_kv_materialise"]


@pytest.fixture
def entered(monkeypatch):
    """Record the streams that torch.cuda.stream is entered with."""
    seen = []

    @contextlib.contextmanager
    def fake_stream(s):
        seen.append(s)
        yield s

    monkeypatch.setattr(pkg.torch.cuda, "stream", fake_stream)
    return seen


def test_every_entry_point_with_a_stream_argument_is_wrapped():
    for name in ENTRY_POINTS:
        fn = getattr(pkg, name)
        assert "stream" in inspect.signature(fn).parameters, name
        assert getattr(fn, "__wrapped__", None) is not None, f"{name} does not switch streams"


def test_stream_by_keyword_and_by_position_is_made_current(entered):
    calls = []

    def body(a, b=None, stream=None):
        calls.append((a, b, stream))
        return a

    wrapped = pkg._on_call_stream(body)
    marker = object()
    assert wrapped(1, stream=marker) == 1
    assert wrapped(2, None, marker) == 2
    assert entered == [marker, marker]
    assert calls == [(1, None, marker), (2, None, marker)]


def test_no_stream_leaves_the_current_stream(entered):
    wrapped = pkg._on_call_stream(lambda a, stream=None: a)
    assert wrapped(3) == 3
    assert wrapped(4, stream=None) == 4
    assert entered == []
