"""Grouped-query attention (Hkv K/V heads for H query heads): CUDA path vs the fp64 oracle.

Query head h reads K/V head h // (H / Hkv) (the pages' BMGHK layout flattened group-major).
Few query rows fold a group's query heads into one block of rows (each K/V head streamed
once); the tensor-core path maps heads per unit.  All calls go through the C ABI
(mslk_attn with Hkv set).
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

KIND = {"none": oracle.MASK_NONE, "causal": oracle.MASK_CAUSAL,
        "blockdiag": oracle.MASK_BLOCKDIAG, "blockdiag_causal": oracle.MASK_BLOCKDIAG_CAUSAL}


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


def _i32(x):
    return torch.tensor(x, dtype=torch.int32, device="cuda")


def _np(t):
    return t.numpy() if isinstance(t, torch.Tensor) else np.asarray(t)


@pytest.mark.parametrize("B,M,Mkv,H,Hkv,D,mask,br,wl,policy", [
    (2, 1, 3000, 8, 2, 128, "causal", True, None, 0),     # decode, 4 heads folded per K/V head
    (1, 2, 2500, 8, 2, 128, "causal", True, None, 0),     # 2 positions x 4 heads = 8 rows
    (1, 3, 2000, 8, 2, 64, "causal", True, 100, 0),       # 3 positions: 2 heads folded
    (2, 4, 1500, 6, 3, 128, "none", False, None, 0),      # group 2, 4 positions: 2 heads folded
    (1, 1, 5000, 16, 1, 128, "none", False, None, 0),     # one K/V head for 16 query heads (fold 8)
    (1, 300, 700, 8, 2, 128, "causal", True, None, 0),    # tensor cores
    (2, 260, 260, 6, 2, 64, "causal", False, 50, 0),
    (1, 4, 900, 8, 4, 128, "causal", True, None, 1),      # few rows forced onto the tensor cores
])
def test_gqa_dense(B, M, Mkv, H, Hkv, D, mask, br, wl, policy):
    q, k, v = inputs.qkv(B, M, Mkv, H, D, Hkv=Hkv, seed=M + H + Hkv)
    s = D ** -0.5
    fa.set_path_policy(policy)
    try:
        out, lse = fa.attn_fwd(*to_dev(q, k, v), mask=mask, scale=s, bottom_right=br, window_left=wl)
        torch.cuda.synchronize()
    finally:
        fa.set_path_policy(0)
    ro, rl = oracle.attention(f32(q), f32(k), f32(v), s, KIND[mask], bottom_right=br, window_left=wl)
    compare(out.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl,
            f"gqa B{B} M{M} Mkv{Mkv} H{H}/{Hkv} D{D} {mask} policy{policy}")


@pytest.mark.parametrize("lq", [[1, 1, 1], [2, 1, 2], [100, 7, 300]])
def test_gqa_varlen(lq):
    lk = [900, 64, 1300]
    cu_q, cu_k = inputs.cu_seqlens(lq), inputs.cu_seqlens(lk)
    q, k, v = inputs.qkv(1, sum(lq), sum(lk), 8, 128, Hkv=2, seed=sum(lq))
    s = 128 ** -0.5
    out, lse = fa.attn_fwd(*to_dev(q, k, v), mask="blockdiag_causal", scale=s, cu_seqlens_q=_i32(cu_q),
                           cu_seqlens_k=_i32(cu_k), max_seqlen_q=max(lq), max_seqlen_k=max(lk),
                           bottom_right=True)
    ro, rl = oracle.attention(f32(q), f32(k), f32(v), s, oracle.MASK_BLOCKDIAG_CAUSAL, cu_q, cu_k,
                              bottom_right=True)
    compare(out.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl, f"gqa varlen {lq}")


def test_gqa_paged_decode():
    lq, lk, ps, H, Hkv = [1, 1, 2], [700, 3001, 129], 64, 8, 2
    table, n_pages, _ = inputs.page_table(lk, ps, spare_pages=2, seed=4)
    q, k, v = inputs.qkv(1, sum(lq), n_pages * ps, H, 128, Hkv=Hkv, seed=4)
    s = 128 ** -0.5
    out, lse = fa.attn_fwd_lanes(q.cuda(), k.cuda().view(n_pages, ps, Hkv, 128),
                                 v.cuda().view(n_pages, ps, Hkv, 128), seqlen_k=_i32(lk),
                                 cu_seqlens_q=_i32(inputs.cu_seqlens(lq)), max_seqlen_q=max(lq),
                                 max_seqlen_k=max(lk), block_table=table.cuda(), page_size=ps,
                                 bottom_right=True)
    ro, rl = oracle.attention_lanes(f32(q), f32(k), f32(v), s, oracle.MASK_BLOCKDIAG_CAUSAL,
                                    inputs.cu_seqlens(lq), lk, block_table=table.numpy(),
                                    page_size=ps, bottom_right=True)
    compare(out.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl, "gqa paged decode")


@pytest.mark.parametrize("M", [1, 200])
def test_gqa_split_kv(M):
    q, k, v = inputs.qkv(2, M, 2048, 8, 128, Hkv=2, seed=M)
    s = 128 ** -0.5
    qd, kd, vd = to_dev(q, k, v)
    outs, lses = [], []
    for a, b in inputs.equal_chunks(2048, 4):
        o, l_ = fa.attn_partial(qd, kd[:, a:b], vd[:, a:b], scale=s, kv_offset=a)
        outs.append(o)
        lses.append(l_)
    out, lse = fa.merge_attentions(torch.stack(outs), torch.stack(lses))
    ro, rl = oracle.attention(f32(q), f32(k), f32(v), s, oracle.MASK_NONE)
    compare(out.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl, f"gqa split-KV M{M}")


def test_gqa_fp8_decode():
    q8, dq, k8, dk, v8, dv = inputs.qkv_fp8(2, 1, 4000, 8, 128, Hkv=2, seed=3)
    s = 128 ** -0.5
    out, lse = fa.attn_fwd_fp8(q8.cuda(), k8.cuda(), v8.cuda(), dq.cuda(), dk.cuda(), dv.cuda(),
                               mask="causal", scale=s, bottom_right=True)
    torch.cuda.synchronize()
    ro, rl = oracle.attention_fp8(_np(q8), _np(k8), _np(v8), _np(dq), _np(dk), _np(dv), s,
                                  oracle.MASK_CAUSAL, bottom_right=True)
    compare(out.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl, "gqa fp8 decode")


def test_gqa_equals_expanded_on_tensor_cores():
    """Grouped heads give the same bits as the same K/V repeated per query head (the tensor
    cores process each query head's unit the same way in both)."""
    q, k, v = inputs.qkv(1, 400, 400, 8, 128, Hkv=2, seed=17)
    qd, kd, vd = to_dev(q, k, v)
    a = fa.attn_fwd(qd, kd, vd, mask="causal")
    b = fa.attn_fwd(qd, kd.repeat_interleave(4, dim=2), vd.repeat_interleave(4, dim=2), mask="causal")
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])
