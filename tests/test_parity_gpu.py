"""CUDA path vs the fp64 oracle on seeded inputs, through the C ABI.

Small cases compare every element; the full-size workloads compare sampled heads/rows
that the oracle computes one by one.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import attention_fmha_fwd_gb300 as fa
import oracle
from attention_fmha_fwd_gb300 import inputs
from tests.gpu_util import MASK_IDS, compare, f32, to_dev

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


def _ref(q, k, v, scale, mask, **kw):
    return oracle.attention(f32(q), f32(k), f32(v), scale, MASK_IDS[mask], **kw)


def _fwd_case(B, M, Mkv, H, D, mask, scale=None, seed=0, policy=0):
    q, k, v = inputs.qkv(B, M, Mkv, H, D, seed=seed)
    s = scale if scale is not None else 1 / D ** 0.5
    fa.set_path_policy(policy)
    try:
        out, lse = fa.attn_fwd(*to_dev(q, k, v), mask=mask, scale=s)
        torch.cuda.synchronize()
    finally:
        fa.set_path_policy(0)
    ro, rl = _ref(q, k, v, s, mask)
    return compare(out.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl,
                   f"fwd B{B} M{M} Mkv{Mkv} H{H} D{D} {mask}")


def test_tiny_fwd_workload():
    """1 x 128 x 2 x 64, no mask, scale 1/8, seed 0 (the tiny forward workload)."""
    w = inputs.WORKLOADS["tiny_fwd"]
    _fwd_case(w.B, w.M, w.Mkv, w.H, w.K, w.mask, w.scale)


@pytest.mark.parametrize("mask", ["none", "causal"])
@pytest.mark.parametrize("B,M,Mkv,H,D", [
    (2, 300, 333, 3, 128),    # several tiles, ragged tails on both axes
    (1, 257, 129, 2, 64),
    (1, 640, 640, 2, 128),    # several 256-row units
    (2, 130, 700, 1, 128),    # Mkv > M
    (1, 600, 200, 2, 128),    # Mkv < M (causal rows past the keys)
    (1, 9, 77, 2, 128),       # smallest M on the tensor-core path
    (1, 128, 1, 2, 64),       # a single key
])
def test_fwd_tensor_core(B, M, Mkv, H, D, mask):
    _fwd_case(B, M, Mkv, H, D, mask)


@pytest.mark.parametrize("mask", ["none", "causal"])
@pytest.mark.parametrize("M", [1, 2, 3, 5, 8])
@pytest.mark.parametrize("D", [64, 128])
def test_fwd_decode_rows(M, D, mask):
    """Few query rows: the CUDA-core kernel, and the same problem on the tensor-core kernel."""
    _fwd_case(3, M, 1000, 4, D, mask)
    _fwd_case(3, M, 1000, 4, D, mask, policy=1)


@pytest.mark.parametrize("M", [1, 3, 8])
def test_decode_cluster_split_long_keys(M):
    """Few heads and many keys: the decode kernel splits each head's keys over a cluster
    of CTAs (16 where the device schedules it, else 8) and merges them through distributed
    shared memory."""
    _fwd_case(1, M, 20000, 2, 128, "none", seed=21)
    q, k, v = inputs.qkv(1, M, 20000, 2, 128, seed=22)
    o, l_ = fa.attn_partial(*to_dev(q, k, v), mask="causal", kv_offset=-19990)
    ro, rl = oracle.attention_partial(f32(q), f32(k), f32(v), 1 / 128 ** 0.5, 1, kv_offset=-19990)
    compare(o.double().cpu().numpy(), l_.double().cpu().numpy(), ro, rl, "cluster causal partial")


@pytest.mark.parametrize("B,H,Mkv,D", [(1, 8, 20000, 128), (2, 2, 33000, 128), (1, 4, 40000, 64)])
def test_decode_cluster_sizes(B, H, Mkv, D):
    """Cluster sizes 8 and 16 (and D = 64) over long key ranges, one query row."""
    _fwd_case(B, 1, Mkv, H, D, "none", seed=23)


def test_fwd_strided_views_and_shared_head():
    """q/k/v as views into packed buffers (free strides) and K/V expanded with head stride 0."""
    B, M, Mkv, H, D = 2, 200, 260, 4, 128
    g = torch.Generator().manual_seed(5)
    qkv = torch.randn(B, M, 3, H, D, generator=g).to(torch.bfloat16)
    k1 = torch.randn(B, Mkv, 1, D, generator=g).to(torch.bfloat16)
    v1 = torch.randn(B, Mkv, 1, D, generator=g).to(torch.bfloat16)
    qd = qkv.cuda()[:, :, 0]
    kd = k1.cuda().expand(B, Mkv, H, D)
    vd = v1.cuda().expand(B, Mkv, H, D)
    assert kd.stride(2) == 0
    for mask in ("none", "causal"):
        for policy in (0, 1):
            fa.set_path_policy(policy)
            out, lse = fa.attn_fwd(qd, kd, vd, mask=mask)
            fa.set_path_policy(0)
            ro, rl = oracle.attention(f32(qkv[:, :, 0]), f32(k1), f32(v1), 1 / D ** 0.5,
                                      MASK_IDS[mask])
            compare(out.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl, mask)
    # decode rows through the shared head as well
    out, lse = fa.attn_fwd(qd[:, :4], kd, vd, mask="none")
    ro, rl = oracle.attention(f32(qkv[:, :4, 0]), f32(k1), f32(v1), 1 / D ** 0.5, 0)
    compare(out.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl, "shared decode")


def test_fwd_output_into_strided_view_and_no_lse():
    B, M, Mkv, H, D = 1, 150, 150, 2, 64
    q, k, v = inputs.qkv(B, M, Mkv, H, D, seed=3)
    big = torch.full((B, M, H, 2 * D), 7.0, dtype=torch.bfloat16, device="cuda")
    out_view = big[..., :D]
    out, lse = fa.attn_fwd(*to_dev(q, k, v), mask="causal", out=out_view, lse=False)
    assert lse is None
    ro, _ = _ref(q, k, v, 1 / D ** 0.5, "causal")
    compare(out_view.double().cpu().numpy(), None, ro, None, "strided out")
    assert torch.all(big[..., D:] == 7.0), "wrote outside the output view"


def test_fwd_default_scale_and_empty_keys():
    q, k, v = inputs.qkv(1, 40, 50, 2, 128, seed=4)
    out, lse = fa.attn_fwd(*to_dev(q, k, v), scale=None)
    ro, rl = _ref(q, k, v, 1 / 128 ** 0.5, "none")
    compare(out.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl, "default scale")
    # Mkv = 0: every row is empty
    qd = q.cuda()
    k0 = torch.empty(1, 0, 2, 128, dtype=torch.bfloat16, device="cuda")
    out, lse = fa.attn_fwd(qd, k0, k0)
    torch.cuda.synchronize()
    assert torch.all(out == 0) and torch.all(torch.isneginf(lse))
    # M = 0: nothing happens
    out, lse = fa.attn_fwd(qd[:, :0], k.cuda(), v.cuda())
    assert out.numel() == 0


def test_fwd_deterministic():
    q, k, v = to_dev(*inputs.qkv(2, 500, 500, 4, 128, seed=6))
    o1, l1 = fa.attn_fwd(q, k, v, mask="causal")
    o2, l2 = fa.attn_fwd(q, k, v, mask="causal")
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


# ------------------------------------------------------------------ split-KV


def _split(q, k, v, bounds, mask, scale, out_dtype=torch.float32):
    qd, kd, vd = to_dev(q, k, v)
    outs, lses = [], []
    for a, b in bounds:
        o, l_ = fa.attn_partial(qd, kd[:, a:b], vd[:, a:b], mask=mask, scale=scale,
                                kv_offset=a, out_dtype=out_dtype)
        outs.append(o)
        lses.append(l_)
    return outs, lses


@pytest.mark.parametrize("n", [2, 8])
def test_split_kv_workload(n):
    """1 x 128 queries against 1024 keys, 16 heads, chunks of equal contiguous keys."""
    w = inputs.WORKLOADS["split_kv"]
    q, k, v = inputs.qkv(w.B, w.M, w.Mkv, w.H, w.K, seed=0)
    bounds = inputs.equal_chunks(w.Mkv, n)
    outs, lses = _split(q, k, v, bounds, "none", w.scale)
    # each partial against the oracle's partial
    for (a, b), o, l_ in zip(bounds, outs, lses):
        ro, rl = oracle.attention_partial(f32(q), f32(k[:, a:b]), f32(v[:, a:b]), w.scale, 0)
        compare(o.double().cpu().numpy(), l_.double().cpu().numpy(), ro, rl, f"partial {a}:{b}")
    out, lse = fa.merge_attentions(torch.stack(outs), torch.stack(lses))
    ro, rl = _ref(q, k, v, w.scale, "none")
    compare(out.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl, f"merged n={n}")
    # the merged result also matches the unsplit kernel
    fo, fl = fa.attn_fwd(*to_dev(q, k, v), scale=w.scale)
    torch.cuda.synchronize()
    assert (fo.float() - out.float()).abs().max().item() <= 2e-2
    assert (fl - lse).abs().max().item() <= 1e-3


@pytest.mark.parametrize("mask", ["none", "causal"])
def test_split_kv_unequal_chunks_and_list_merge(mask):
    q, k, v = inputs.qkv(2, 300, 1024, 3, 128, seed=7)
    bounds = [(0, 100), (100, 101), (101, 400), (400, 1024)]
    outs, lses = _split(q, k, v, bounds, mask, 0.1)
    out, lse = fa.merge_attentions(outs, lses)          # a list of separate allocations
    ro, rl = _ref(q, k, v, 0.1, mask)
    compare(out.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl, f"unequal {mask}")
    # permuting chunks changes nothing beyond rounding
    perm = [2, 0, 3, 1]
    out2, lse2 = fa.merge_attentions([outs[i] for i in perm], [lses[i] for i in perm])
    compare(out2.double().cpu().numpy(), lse2.double().cpu().numpy(), ro, rl, "permuted")


def test_causal_partial_empty_rows():
    """A causal chunk that starts past some rows leaves them empty: out 0, lse -inf."""
    q, k, v = inputs.qkv(1, 300, 600, 2, 128, seed=8)
    qd, kd, vd = to_dev(q, k, v)
    for policy in (0, 1):
        fa.set_path_policy(policy)
        o, l_ = fa.attn_partial(qd, kd[:, 200:600], vd[:, 200:600], mask="causal", kv_offset=200)
        fa.set_path_policy(0)
        ro, rl = oracle.attention_partial(f32(q), f32(k[:, 200:600]), f32(v[:, 200:600]),
                                          1 / 128 ** 0.5, 1, kv_offset=200)
        compare(o.double().cpu().numpy(), l_.double().cpu().numpy(), ro, rl, "empty rows")
        assert torch.all(o[:, :200] == 0)
    # decode rows whose chunk is entirely in the future
    o, l_ = fa.attn_partial(qd[:, :4], kd[:, 200:600], vd[:, 200:600], mask="causal", kv_offset=200)
    torch.cuda.synchronize()
    assert torch.all(o == 0) and torch.all(torch.isneginf(l_))


def test_partial_bf16_output():
    q, k, v = inputs.qkv(1, 130, 256, 2, 64, seed=9)
    outs, lses = _split(q, k, v, [(0, 128), (128, 256)], "none", 0.125, out_dtype=torch.bfloat16)
    for (a, b), o, l_ in zip([(0, 128), (128, 256)], outs, lses):
        ro, rl = oracle.attention_partial(f32(q), f32(k[:, a:b]), f32(v[:, a:b]), 0.125, 0)
        compare(o.double().cpu().numpy(), l_.double().cpu().numpy(), ro, rl, "bf16 partial")


def test_decode_split_kv_reduced():
    """The decode split-KV shape at reduced size: 4 x 1 query against 4096 keys, 8 heads,
    K/V drawn as 8 groups of one head, 4 chunks of 1024."""
    q, k, v = inputs.qkv(4, 1, 4096, 8, 128, seed=10)
    bounds = inputs.equal_chunks(4096, 4)
    outs, lses = _split(q, k, v, bounds, "none", 1 / 128 ** 0.5)
    out, lse = fa.merge_attentions(torch.stack(outs), torch.stack(lses))
    ro, rl = _ref(q, k, v, 1 / 128 ** 0.5, "none")
    compare(out.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl, "decode reduced")


# ------------------------------------------------------------------ merge


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
def test_merge_against_oracle_with_empty_chunks(out_dtype):
    g = torch.Generator().manual_seed(11)
    n, B, M, H, Kv = 5, 2, 33, 3, 128
    outs = torch.randn(n, B, M, H, Kv, generator=g)
    lses = torch.randn(n, B, H, M, generator=g) * 4
    lses[1, 0, 1, 2] = float("-inf")
    lses[:, 1, 0, 5] = float("-inf")                     # every chunk empty for one row
    out, lse = fa.merge_attentions(outs.cuda(), lses.cuda(), output_dtype=out_dtype)
    ro, rl = oracle.merge_attentions(outs.numpy(), lses.numpy())
    compare(out.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl, "merge")
    assert torch.all(out[1, 5, 0] == 0)
    out2, lse2 = fa.merge_attentions(outs.cuda(), lses.cuda(), write_lse=False)
    assert lse2 is None
    compare(out2.double().cpu().numpy(), None, ro, None, "merge no lse")


def test_merge_many_chunks_and_head_dim_64():
    g = torch.Generator().manual_seed(12)
    n, B, M, H, Kv = 40, 1, 17, 2, 64
    outs = torch.randn(n, B, M, H, Kv, generator=g)
    lses = torch.randn(n, B, H, M, generator=g)
    out, lse = fa.merge_attentions(outs.cuda(), lses.cuda())
    ro, rl = oracle.merge_attentions(outs.numpy(), lses.numpy())
    compare(out.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl, "merge n=40")


# ------------------------------------------------------------------ varlen


@pytest.mark.parametrize("mask", ["blockdiag", "blockdiag_causal"])
def test_varlen_small(mask):
    lq = [1, 127, 129, 300, 5, 256]
    lk = [3, 127, 129, 300, 260, 1] if mask == "blockdiag" else lq
    cq, ck = inputs.cu_seqlens(lq), inputs.cu_seqlens(lk)
    q, k, v = inputs.qkv(1, cq[-1], ck[-1], 3, 128, seed=13)
    cqd = torch.tensor(cq, dtype=torch.int32, device="cuda")
    ckd = torch.tensor(ck, dtype=torch.int32, device="cuda")
    out, lse = fa.attn_fwd(*to_dev(q, k, v), mask=mask, cu_seqlens_q=cqd, cu_seqlens_k=ckd,
                           max_seqlen_q=max(lq), max_seqlen_k=max(lk))
    ro, rl = _ref(q, k, v, 1 / 128 ** 0.5, mask, cu_seqlens_q=cq, cu_seqlens_k=ck)
    compare(out.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl, f"varlen {mask}")


@pytest.mark.parametrize("n_seqs", [12, 128, 140])
def test_varlen_many_sequences(n_seqs):
    """Many packed sequences of mixed lengths (one empty, two equal) against the oracle: most
    slots of the unit grid (longest sequence x heads x sequences) are empty and skipped."""
    g = torch.Generator().manual_seed(40 + n_seqs)
    lq = torch.randint(1, 700, (n_seqs,), generator=g).tolist()
    lq[3] = 0
    lq[7] = lq[8] = 256  # equal unit counts
    cq = inputs.cu_seqlens(lq)
    q, k, v = inputs.qkv(1, cq[-1], cq[-1], 2, 64, seed=41)
    cqd = torch.tensor(cq, dtype=torch.int32, device="cuda")
    out, lse = fa.attn_fwd(*to_dev(q, k, v), mask="blockdiag_causal", cu_seqlens_q=cqd,
                           cu_seqlens_k=cqd, max_seqlen_q=max(lq), max_seqlen_k=max(lq))
    ro, rl = _ref(q, k, v, 1 / 64 ** 0.5, "blockdiag_causal", cu_seqlens_q=cq, cu_seqlens_k=cq)
    compare(out.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl, f"varlen x{n_seqs}")


def test_varlen_partial_merge():
    """Block-diagonal causal split per sequence: chunk c holds keys [c*64, c*64+64) of
    every sequence (kv_offset = c*64), merged == the unsplit packed attention."""
    lens = [70, 200, 129]
    cu = inputs.cu_seqlens(lens)
    q, k, v = inputs.qkv(1, cu[-1], cu[-1], 2, 64, seed=14)
    qd, kd, vd = to_dev(q, k, v)
    cqd = torch.tensor(cu, dtype=torch.int32, device="cuda")
    outs, lses = [], []
    for c in range(4):
        idx, cuc = [], [0]
        for s, L in enumerate(lens):
            sel = list(range(cu[s] + 64 * c, cu[s] + min(L, 64 * c + 64)))
            idx += sel
            cuc.append(cuc[-1] + len(sel))
        it = torch.tensor(idx, dtype=torch.long, device="cuda")
        kc, vc = kd[:, it].contiguous(), vd[:, it].contiguous()
        ckd = torch.tensor(cuc, dtype=torch.int32, device="cuda")
        max_k = max(b - a for a, b in zip(cuc[:-1], cuc[1:]))
        o, l_ = fa.attn_partial(qd, kc, vc, mask="blockdiag_causal", kv_offset=64 * c,
                                cu_seqlens_q=cqd, cu_seqlens_k=ckd, max_seqlen_q=max(lens),
                                max_seqlen_k=max_k)
        outs.append(o)
        lses.append(l_)
    out, lse = fa.merge_attentions(outs, lses)
    ro, rl = _ref(q, k, v, 1 / 64 ** 0.5, "blockdiag_causal", cu_seqlens_q=cu, cu_seqlens_k=cu)
    compare(out.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl, "varlen split")


# ------------------------------------------------------------------ full-size workloads


def test_causal_fwd_workload_sampled():
    """2 x 2048 x 32 x 128 causal at full size, in the launch configuration the benchmark
    times.  Every (batch, head) pair is checked against the oracle on the first and last
    row of every 128-row tile plus 16 random rows: a fault confined to one persistent
    CTA's units, one scheduling round or one Q tile of a unit shows up in some pair."""
    w = inputs.WORKLOADS["causal_fwd"]
    q, k, v = inputs.qkv(w.B, w.M, w.Mkv, w.H, w.K, seed=0)
    out, lse = fa.attn_fwd(*to_dev(q, k, v), mask="causal", scale=w.scale)
    out = out.double().cpu().numpy()
    lse = lse.double().cpu().numpy()
    rng = np.random.default_rng(0)
    edges = np.concatenate([np.arange(0, w.M, 128), np.arange(127, w.M, 128)])
    qf, kf, vf = f32(q), f32(k), f32(v)
    for b in range(w.B):
        for h in range(w.H):
            rows = np.unique(np.concatenate([edges, rng.integers(0, w.M, 16)]))
            ro, rl = oracle.attention_head(qf, kf, vf, b, h, w.scale, oracle.MASK_CAUSAL, rows=rows)
            compare(out[b, rows, h], lse[b, h, rows], ro, rl, f"causal b{b} h{h}")


def test_decode_split_kv_workload_sampled():
    """16 x 1 query against 32768 keys, 8 heads, 16 chunks of 2048 + merge, at full size;
    every (batch, head) pair against the oracle's unsplit attention."""
    w = inputs.WORKLOADS["decode_split_kv"]
    q, k, v = inputs.qkv(w.B, w.M, w.Mkv, w.H, w.K, seed=0)
    bounds = inputs.equal_chunks(w.Mkv, 16)
    outs, lses = _split(q, k, v, bounds, "none", w.scale)
    out, lse = fa.merge_attentions(torch.stack(outs), torch.stack(lses))
    out = out.double().cpu().numpy()
    lse = lse.double().cpu().numpy()
    for b in range(w.B):
        qb, kb, vb = f32(q[b:b + 1]), f32(k[b:b + 1]), f32(v[b:b + 1])
        for h in range(w.H):
            ro, rl = oracle.attention_head(qb, kb, vb, 0, h, w.scale, 0)
            compare(out[b, :, h], lse[b, h], ro, rl, f"decode b{b} h{h}")


def test_varlen_workload_sampled():
    """12 packed sequences (seeded lengths in [128, 4096], total 16384), 32 heads, 128,
    block-diagonal causal; every head against the oracle (all rows)."""
    w = inputs.WORKLOADS["varlen_packed"]
    lens = inputs.varlen_seqlens(w.n_seqs, w.M, seed=0)
    cu = inputs.cu_seqlens(lens)
    q, k, v = inputs.qkv(1, w.M, w.Mkv, w.H, w.K, seed=0)
    cud = torch.tensor(cu, dtype=torch.int32, device="cuda")
    out, lse = fa.attn_fwd(*to_dev(q, k, v), mask="blockdiag_causal", scale=w.scale,
                           cu_seqlens_q=cud, cu_seqlens_k=cud, max_seqlen_q=max(lens),
                           max_seqlen_k=max(lens))
    out = out.double().cpu().numpy()
    lse = lse.double().cpu().numpy()
    qf, kf, vf = f32(q), f32(k), f32(v)
    for h in range(w.H):
        ro, rl = oracle.attention_head(qf, kf, vf, 0, h, w.scale, oracle.MASK_BLOCKDIAG_CAUSAL,
                                       cu_seqlens_q=cu, cu_seqlens_k=cu)
        compare(out[0, :, h], lse[0, h], ro, rl, f"varlen h{h}")


def test_independent_partials_overlap():
    """Back-to-back chunk partials declared independent (programmatic dependent launch),
    eager and captured in a CUDA graph, then merged: equal to the oracle and bit-equal to
    the same partials in plain stream order."""
    B, M, Mkv, H, D = 16, 1, 8192, 8, 128
    q, k, v = inputs.qkv(B, M, Mkv, H, D, seed=31)
    s = D ** -0.5
    qd, kd, vd = to_dev(q, k, v)
    bounds = inputs.equal_chunks(Mkv, 8)
    po = torch.empty((8, B, M, H, D), dtype=torch.float32, device="cuda")
    pl = torch.empty((8, B, H, M), dtype=torch.float32, device="cuda")

    def parts(independent):
        for c, (a, b) in enumerate(bounds):
            fa.attn_partial(qd, kd[:, a:b], vd[:, a:b], scale=s, out=po[c], lse=pl[c],
                            independent=independent and c > 0)

    parts(False)
    ref_o, ref_l = po.clone(), pl.clone()
    parts(True)
    torch.cuda.synchronize()
    assert torch.equal(po, ref_o) and torch.equal(pl, ref_l)
    po.zero_()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        parts(True)
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        parts(True)
    po.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(po, ref_o) and torch.equal(pl, ref_l)
    out, lse = fa.merge_attentions(po, pl)
    ro, rl = oracle.attention(f32(q), f32(k), f32(v), s, oracle.MASK_NONE)
    compare(out.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl, "independent partials")


def test_independent_partials_tensor_cores():
    """The same on the tensor-core path (128 query rows per chunk)."""
    w = inputs.WORKLOADS["split_kv"]
    q, k, v = inputs.qkv(w.B, w.M, w.Mkv, w.H, w.K, seed=0)
    qd, kd, vd = to_dev(q, k, v)
    bounds = inputs.equal_chunks(w.Mkv, 8)
    outs = {}
    for ind in (False, True):
        po = torch.empty((8, w.B, w.M, w.H, w.Kv), dtype=torch.float32, device="cuda")
        pl = torch.empty((8, w.B, w.H, w.M), dtype=torch.float32, device="cuda")
        for c, (a, b) in enumerate(bounds):
            fa.attn_partial(qd, kd[:, a:b], vd[:, a:b], scale=w.scale, out=po[c], lse=pl[c],
                            independent=ind and c > 0)
        torch.cuda.synchronize()
        outs[ind] = (po, pl)
    assert torch.equal(outs[False][0], outs[True][0]) and torch.equal(outs[False][1], outs[True][1])
    out, lse = fa.merge_attentions(*outs[True])
    ro, rl = oracle.attention(f32(q), f32(k), f32(v), w.scale, oracle.MASK_NONE)
    compare(out.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl, "independent tc partials")
