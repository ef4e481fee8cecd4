"""Split-KV in one call, the varargs merge, and the BMGHK layout: CUDA path vs the fp64
oracle, through the C ABI.

* mslk_attn_split_kv: partials over equal key chunks into a caller workspace, then the
  merge ("Attention - Core fMHA" > memory_efficient_attention_partial + merge_attentions).
* mslk_merge_attentions_varargs: separately allocated chunks merged where they lie
  ("Attention - Merge & storage utilities" > fmha_merge_attentions_varargs), with no
  allocation in the binding.
* 5-D BMGHK inputs with K/V expanded over H ("Attention - Core fMHA" >
  memory_efficient_attention layouts; "Operator protocol" > bmghk2bmhk) run on views.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import attention_fmha_fwd_gb300 as fa
import oracle
from attention_fmha_fwd_gb300 import inputs
from tests.gpu_util import compare, f32, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from attention_fmha_fwd_gb300 import build
    build.build()
    fa.set_path_policy(0)
    yield
    fa.set_path_policy(0)
    assert fa.device_status() == 0


def _allocs():
    return torch.cuda.memory_stats().get("allocation.all.allocated", 0)


@pytest.mark.parametrize("n_chunks", [2, 8, 0, 5])
def test_split_kv_workload(n_chunks):
    """The split-KV workload (1 x 128 queries x 1024 keys x 16 heads x 128) in one call."""
    w = inputs.WORKLOADS["split_kv"]
    q, k, v = inputs.qkv(w.B, w.M, w.Mkv, w.H, w.K, seed=0)
    out, lse = fa.attn_split_kv(*to_dev(q, k, v), n_chunks=n_chunks, scale=w.scale)
    ro, rl = oracle.attention(f32(q), f32(k), f32(v), w.scale, oracle.MASK_NONE)
    compare(out.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl, f"split n={n_chunks}")


@pytest.mark.parametrize("mask,kw,M,Mkv,n", [
    ("causal", {}, 300, 700, 4),                              # top-left, chunks past the rows
    ("causal_bottom_right", {}, 200, 1000, 3),                # shift folded into kv_offset
    ("causal", {"window_left": 100}, 333, 333, 6),            # causal local window
    ("none", {"bottom_right": True, "window_left": 64, "window_right": 32}, 129, 900, 7),
    ("none", {}, 5, 4000, 0),                                 # few rows: CUDA-core partials
])
def test_split_kv_masks(mask, kw, M, Mkv, n):
    B, H, D = 2, 4, 128
    q, k, v = inputs.qkv(B, M, Mkv, H, D, seed=41)
    s = D ** -0.5
    out, lse = fa.attn_split_kv(*to_dev(q, k, v), n_chunks=n, mask=mask, scale=s, **kw)
    kind = oracle.MASK_NONE if mask == "none" else oracle.MASK_CAUSAL
    br = mask == "causal_bottom_right" or kw.get("bottom_right", False)
    ro, rl = oracle.attention(f32(q), f32(k), f32(v), s, kind, bottom_right=br,
                              window_left=kw.get("window_left"), window_right=kw.get("window_right"))
    compare(out.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl, f"split {mask} {kw} n={n}")


def test_split_kv_grouped_heads_fp32_out_and_workspace_reuse():
    """Grouped K/V heads, fp32 output, one workspace for two calls in a row."""
    B, M, Mkv, H, Hkv, D = 3, 64, 1500, 8, 2, 64
    g = torch.Generator().manual_seed(5)
    q = torch.randn(B, M, H, D, generator=g).to(torch.bfloat16)
    k = torch.randn(B, Mkv, Hkv, D, generator=g).to(torch.bfloat16)
    v = torch.randn(B, Mkv, Hkv, D, generator=g).to(torch.bfloat16)
    qd, kd, vd = to_dev(q, k, v)
    nb = fa.split_kv_workspace_bytes(qd, kd, vd, n_chunks=4, out_dtype=torch.float32)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    ro, rl = oracle.attention(f32(q), f32(k), f32(v), 0.2, oracle.MASK_NONE)
    for _ in range(2):
        out, lse = fa.attn_split_kv(qd, kd, vd, n_chunks=4, scale=0.2, out_dtype=torch.float32,
                                    workspace=ws)
        compare(out.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl, "split gqa fp32")


def test_split_kv_decode_workload():
    """16 x 1 query x 32768 keys x 8 heads in 16 chunks through the one-call path, every
    (batch, head) pair against the oracle."""
    w = inputs.WORKLOADS["decode_split_kv"]
    q, k, v = inputs.qkv(w.B, w.M, w.Mkv, w.H, w.K, seed=0)
    out, lse = fa.attn_split_kv(*to_dev(q, k, v), n_chunks=16, scale=w.scale)
    out = out.double().cpu().numpy()
    lse = lse.double().cpu().numpy()
    for b in range(w.B):
        qb, kb, vb = f32(q[b:b + 1]), f32(k[b:b + 1]), f32(v[b:b + 1])
        for h in range(w.H):
            ro, rl = oracle.attention_head(qb, kb, vb, 0, h, w.scale, 0)
            compare(out[b, :, h], lse[b, h], ro, rl, f"split decode b{b} h{h}")


def test_varargs_merge_separate_chunks():
    """Chunks from separate allocations merge in place: no allocation in the call, the same
    bits as the stacked merge of copies of them, and the oracle's unsplit attention."""
    B, M, Mkv, H, D = 2, 200, 900, 4, 128
    q, k, v = inputs.qkv(B, M, Mkv, H, D, seed=17)
    qd, kd, vd = to_dev(q, k, v)
    s = D ** -0.5
    bounds = [(0, 100), (100, 450), (450, 451), (451, 900)]
    outs, lses, spacers = [], [], []
    for c, (a, b) in enumerate(bounds):
        o, l_ = fa.attn_partial(qd, kd[:, a:b], vd[:, a:b], mask="causal", kv_offset=a, scale=s)
        outs.append(o)
        lses.append(l_)
        spacers.append(torch.empty(4096 * (c + 1), device="cuda"))  # uneven gaps between chunks
    from attention_fmha_fwd_gb300 import api
    assert api._stacked(outs) is None  # not one strided allocation: the varargs entry runs
    out = torch.empty((B, M, H, D), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H, M), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    n0 = _allocs()
    fa.merge_attentions(outs, lses, out=out, lse=lse)
    assert _allocs() == n0, "the varargs merge allocated device memory"
    so, sl = fa.merge_attentions(torch.stack(outs), torch.stack(lses))
    torch.cuda.synchronize()
    assert torch.equal(out, so) and torch.equal(lse, sl)
    ro, rl = oracle.attention(f32(q), f32(k), f32(v), s, oracle.MASK_CAUSAL)
    compare(out.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl, "varargs merge")


def test_varargs_merge_many_chunks_fp32_out():
    B, M, Mkv, H, D = 1, 16, 1280, 2, 64
    q, k, v = inputs.qkv(B, M, Mkv, H, D, seed=18)
    qd, kd, vd = to_dev(q, k, v)
    outs, lses = [], []
    for c in range(40):
        o, l_ = fa.attn_partial(qd, kd[:, 32 * c:32 * c + 32], vd[:, 32 * c:32 * c + 32], scale=0.125)
        outs.append(o.clone())
        lses.append(l_.clone())
    out, lse = fa.merge_attentions(outs, lses, output_dtype=torch.float32)
    ro, rl = oracle.attention(f32(q), f32(k), f32(v), 0.125, oracle.MASK_NONE)
    compare(out.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl, "varargs 40 chunks")


def test_bmghk_expanded_kv_views():
    """q [B,M,G,H,K] with K/V [B,Mkv,G,1,K] expanded over H (stride 0): no copies (only the
    output and lse are allocated when not given), out [B,M,G,H,K], lse [B,G,H,M]."""
    B, M, Mkv, G, Hg, D = 2, 150, 333, 3, 4, 128
    gen = torch.Generator().manual_seed(23)
    q = torch.randn(B, M, G, Hg, D, generator=gen).to(torch.bfloat16)
    k1 = torch.randn(B, Mkv, G, 1, D, generator=gen).to(torch.bfloat16)
    v1 = torch.randn(B, Mkv, G, 1, D, generator=gen).to(torch.bfloat16)
    qd, kd, vd = to_dev(q, k1, v1)
    ke, ve = kd.expand(B, Mkv, G, Hg, D), vd.expand(B, Mkv, G, Hg, D)
    out = torch.empty((B, M, G, Hg, D), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, G, Hg, M), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    n0 = _allocs()
    fa.attn_fwd(qd, ke, ve, mask="causal", scale=0.1, out=out, lse=lse)
    assert _allocs() == n0, "the BMGHK call copied or allocated"
    qf = f32(q).reshape(B, M, G * Hg, D)
    ro, rl = oracle.attention(qf, f32(k1)[:, :, :, 0], f32(v1)[:, :, :, 0], 0.1, oracle.MASK_CAUSAL)
    compare(out.reshape(B, M, G * Hg, D).double().cpu().numpy(),
            lse.reshape(B, G * Hg, M).double().cpu().numpy(), ro, rl, "bmghk fwd")
    # partials and merge in the same layout
    parts = [fa.attn_partial(qd, ke[:, a:b], ve[:, a:b], mask="causal", kv_offset=a, scale=0.1)
             for a, b in ((0, 111), (111, 333))]
    mo, ml = fa.merge_attentions([p[0] for p in parts], [p[1] for p in parts])
    assert mo.shape == (B, M, G, Hg, D) and ml.shape == (B, G, Hg, M)
    compare(mo.reshape(B, M, G * Hg, D).double().cpu().numpy(),
            ml.reshape(B, G * Hg, M).double().cpu().numpy(), ro, rl, "bmghk split")


def test_partial_repeated_calls_on_the_same_buffers():
    """A second call on the same buffers replays the first call's argument struct: it must
    read the buffers' new contents, and a changed option (key offset, mask, scale) or a
    different chunk must not reuse it."""
    B, M, Mkv, H, D = 1, 70, 300, 4, 128
    q, k, v = inputs.qkv(B, M, Mkv, H, D, seed=31)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    out = torch.empty(B, M, H, D, device="cuda")
    lse = torch.empty(B, H, M, device="cuda")
    s = D ** -0.5
    for step in range(3):
        if step == 2:
            qd.mul_(-0.5)  # same pointer, new contents
        for a0, b0, mask, off in ((0, 128, "none", 0), (128, 300, "causal", 128), (128, 300, "causal", 140)):
            fa.attn_partial(qd, kd[:, a0:b0], vd[:, a0:b0], mask=mask, scale=s, kv_offset=off,
                            out=out, lse=lse)
            torch.cuda.synchronize()
            qh = qd.cpu()
            ro, rl = oracle.attention(qh.float().numpy(), k[:, a0:b0].float().numpy(),
                                      v[:, a0:b0].float().numpy(), s,
                                      oracle.MASK_CAUSAL if mask == "causal" else oracle.MASK_NONE,
                                      kv_offset=off)
            compare(out.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl,
                    f"step {step} chunk {a0}:{b0} {mask} offset {off}")
