"""attn_partial's argument-struct replay, checked on the host with a fake library.

A call with caller-provided out and lse stores the mslk_attn_args struct it was made with;
a later call with the same buffers and options replays that struct through mslk_attn.
Any difference in pointers, shapes, strides, dtypes or options must miss the cache.
"""

from __future__ import annotations

import ctypes

import pytest
import torch

from attention_fmha_fwd_gb300 import _capi, api


class _FakeLib:
    def __init__(self):
        self.calls = []

    def mslk_attn_partial(self, *args):
        self.calls.append(("partial", args))
        return 0

    def mslk_attn(self, args_ref, stream):
        a = ctypes.cast(args_ref, ctypes.POINTER(_capi.AttnArgs)).contents
        self.calls.append(("attn", a))
        return 0


@pytest.fixture
def fake(monkeypatch):
    lib = _FakeLib()
    monkeypatch.setattr(_capi, "load", lambda path=None: lib)
    monkeypatch.setattr(api, "_check_inputs", lambda q, k, v: None)
    monkeypatch.setattr(api, "_stream_handle", lambda stream, device=None: 0)
    api._PARTIAL_ARGS.clear()
    yield lib
    api._PARTIAL_ARGS.clear()


def _bufs():
    q = torch.zeros(1, 64, 4, 128, dtype=torch.bfloat16)
    k = torch.zeros(1, 512, 4, 128, dtype=torch.bfloat16)
    out = torch.zeros(1, 64, 4, 128)
    lse = torch.zeros(1, 4, 64)
    return q, k, out, lse


def test_same_call_replays_the_struct(fake):
    q, k, out, lse = _bufs()
    kc = k[:, :128]
    api.attn_partial(q, kc, kc, scale=0.1, out=out, lse=lse)
    assert [c[0] for c in fake.calls] == ["partial"]
    api.attn_partial(q, kc, kc, scale=0.1, out=out, lse=lse)
    assert [c[0] for c in fake.calls] == ["partial", "attn"]
    a = fake.calls[1][1]
    assert a.q == q.data_ptr() and a.k == kc.data_ptr() and a.v == kc.data_ptr()
    assert a.out == out.data_ptr() and a.lse == lse.data_ptr()
    assert (a.B, a.M, a.Mkv, a.H, a.Hkv, a.K, a.Kv) == (1, 64, 128, 4, 4, 128, 128)
    assert a.partial == 1 and a.kv_offset == 0 and abs(a.scale - 0.1) < 1e-7
    assert (a.sk.b, a.sk.m, a.sk.h) == tuple(kc.stride()[:3])


@pytest.mark.parametrize("change", ["kv_offset", "chunk", "scale", "mask", "out", "independent"])
def test_any_difference_misses(fake, change):
    q, k, out, lse = _bufs()
    kc = k[:, :128]
    api.attn_partial(q, kc, kc, scale=0.1, out=out, lse=lse)
    kw = dict(scale=0.1, out=out, lse=lse)
    k2 = kc
    if change == "kv_offset":
        kw["kv_offset"] = 128
    elif change == "chunk":
        k2 = k[:, 128:256]
    elif change == "scale":
        kw["scale"] = 0.2
    elif change == "mask":
        kw["mask"] = "causal"
    elif change == "out":
        kw["out"] = torch.zeros(1, 64, 4, 128)
    elif change == "independent":
        kw["independent"] = True
    n = len(fake.calls)
    api.attn_partial(q, k2, k2, **kw)
    kind, a = fake.calls[n]
    if change == "independent":
        # a new struct, built for mslk_attn with the flag, not a replay of the first
        assert kind == "attn" and a.flags == _capi.FLAG_INDEPENDENT
    else:
        assert kind == "partial"
    assert len(api._PARTIAL_ARGS) == 2


def test_cache_is_bounded(fake):
    q, k, out, lse = _bufs()
    for off in range(api._PARTIAL_ARGS_MAX + 5):
        api.attn_partial(q, k[:, :128], k[:, :128], scale=0.1, kv_offset=off, out=out, lse=lse)
    assert len(api._PARTIAL_ARGS) <= api._PARTIAL_ARGS_MAX
