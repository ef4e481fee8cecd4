"""Numerical and shape edge cases on both kernels, vs the fp64 oracle through the C ABI.

* large logits (scale x 30: scores hundreds apart), so the lazy rescale and the empty
  -inf handling work at the extremes of fp32 exponents;
* a key late in the row that dominates it (the running max jumps after many tiles);
* many key tiles per row (accumulation over 512 tiles, sampled rows);
* unit counts that do not divide the SM count, and many heads on the decode path;
* tensors of more than 2^31 elements (64-bit offsets): built on the device by repeating a
  host-generated block, so the oracle sees the block (closed form for repeated keys).
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

KIND = {"none": oracle.MASK_NONE, "causal": oracle.MASK_CAUSAL}


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


def _run(q, k, v, scale, mask, policy=0):
    fa.set_path_policy(policy)
    try:
        out, lse = fa.attn_fwd(*to_dev(q, k, v), mask=mask, scale=scale)
        torch.cuda.synchronize()
    finally:
        fa.set_path_policy(0)
    return out.double().cpu().numpy(), lse.double().cpu().numpy()


@pytest.mark.parametrize("M,Mkv,mask,policy", [
    (300, 900, "none", 0), (300, 300, "causal", 0), (4, 3000, "none", 0), (4, 3000, "none", 1)])
def test_large_logits(M, Mkv, mask, policy):
    """scale 30/sqrt(D): logits span hundreds; softmax is near one-hot per row."""
    q, k, v = inputs.qkv(1, M, Mkv, 2, 128, seed=M + Mkv)
    s = 30.0 / 128 ** 0.5
    out, lse = _run(q, k, v, s, mask, policy)
    ro, rl = oracle.attention(f32(q), f32(k), f32(v), s, KIND[mask])
    compare(out, lse, ro, rl, f"large logits M{M} Mkv{Mkv} {mask} policy{policy}")


@pytest.mark.parametrize("M,policy", [(256, 0), (2, 0), (2, 1)])
def test_late_dominant_key(M, policy):
    """Key Mkv - 5 has a large dot product with every query: the running max jumps by far
    more than the lazy threshold in the last tile, after many tiles of small scores."""
    Mkv, H, D = 4000, 2, 128
    q, k, v = inputs.qkv(1, M, Mkv, H, D, seed=41)
    k = k.clone()
    qm = q.float().mean(dim=1, keepdim=True)            # [1, 1, H, D]
    k[:, Mkv - 5] = (qm[:, 0] * 40.0).to(torch.bfloat16)  # aligned with the average query
    s = D ** -0.5
    out, lse = _run(q, k, v, s, "none", policy)
    ro, rl = oracle.attention(f32(q), f32(k), f32(v), s, oracle.MASK_NONE)
    compare(out, lse, ro, rl, f"late dominant key M{M} policy{policy}")


def test_many_key_tiles_sampled():
    """256 queries against 65536 keys (512 key tiles per row), rows sampled for the oracle."""
    M, Mkv, H, D = 256, 65536, 2, 128
    q, k, v = inputs.qkv(1, M, Mkv, H, D, seed=8)
    s = D ** -0.5
    out, lse = _run(q, k, v, s, "causal")  # top-left causal: row i sees keys 0..i
    out2, lse2 = fa.attn_fwd(*to_dev(q, k, v), mask="none", scale=s)
    out2, lse2 = out2.double().cpu().numpy(), lse2.double().cpu().numpy()
    rows = [0, 1, 77, 128, 255]
    qs = q[:, rows]
    ro, rl = oracle.attention(f32(qs), f32(k), f32(v), s, oracle.MASK_NONE)
    compare(out2[:, rows], lse2[:, :, rows], ro, rl, "65536 keys, sampled rows")
    # causal: row i against its own prefix
    for i in (0, 77, 255):
        ro, rl = oracle.attention(f32(q[:, i:i + 1]), f32(k[:, :i + 1]), f32(v[:, :i + 1]), s,
                                  oracle.MASK_NONE)
        compare(out[:, i:i + 1], lse[:, :, i:i + 1], ro, rl, f"causal row {i}")


@pytest.mark.parametrize("mask", ["causal", "none"])
def test_more_than_32_rounds_per_cta(mask):
    """16 x 2560 rows x 32 heads = 5120 units of 256 rows: 34 per CTA on 152 SMs, so the MMA
    warp decodes its units in two batches of 32 rounds.  The last rounds hold the lightest
    units (the first rows of each sequence under a causal mask): sampled rows from every
    256-row block of several heads, and rows 0-255 of every head of one batch."""
    B, M, H, D = 16, 2560, 32, 64
    q, k, v = inputs.qkv(B, M, M, H, D, seed=77)
    s = D ** -0.5
    out, lse = _run(q, k, v, s, mask)
    qf, kf, vf = f32(q), f32(k), f32(v)
    rng = np.random.default_rng(5)
    for b, h in ((0, 0), (7, 13), (15, 31), (11, 2)):
        rows = np.unique(np.concatenate([np.arange(0, M, 256), np.arange(255, M, 256),
                                         rng.integers(0, M, 24)]))
        ro, rl = oracle.attention_head(qf, kf, vf, b, h, s, KIND[mask], rows=rows)
        compare(out[b, rows, h], lse[b, h, rows], ro, rl, f"b{b} h{h}")
    rows = np.arange(0, 256)
    for h in range(H):
        ro, rl = oracle.attention_head(qf, kf, vf, 3, h, s, KIND[mask], rows=rows)
        compare(out[3, rows, h], lse[3, h, rows], ro, rl, f"b3 h{h} rows 0-255")


@pytest.mark.parametrize("B,M,Mkv,H,D,mask", [
    (3, 300, 300, 40, 64, "causal"),     # 3 x 40 x 2 = 240 units on 152 SMs
    (5, 1, 1000, 96, 128, "none"),       # 480 decode CTAs
    (1, 7, 513, 128, 64, "causal"),      # 128 heads, 7 rows
])
def test_odd_unit_counts(B, M, Mkv, H, D, mask):
    q, k, v = inputs.qkv(B, M, Mkv, H, D, seed=B * H + M)
    s = D ** -0.5
    out, lse = _run(q, k, v, s, mask)
    ro, rl = oracle.attention(f32(q), f32(k), f32(v), s, KIND[mask])
    compare(out, lse, ro, rl, f"B{B} M{M} Mkv{Mkv} H{H} D{D} {mask}")


@pytest.mark.parametrize("M,policy", [(4, 0), (4, 2), (8, 0), (2, 0)])
def test_few_rows_many_heads_dispatch(M, policy):
    """Few query rows over 16 x 8 (batch, head) units: the automatic choice sends 2+ rows to
    the tensor cores (policy 0), policy 2 keeps the CUDA-core kernel; both match the oracle."""
    B, Mkv, H, D = 16, 3000, 8, 128
    q, k, v = inputs.qkv(B, M, Mkv, H, D, seed=M + 100)
    s = D ** -0.5
    fa.set_path_policy(policy)
    try:
        out, lse = fa.attn_fwd(*to_dev(q, k, v), mask="causal", scale=s, bottom_right=True)
        torch.cuda.synchronize()
    finally:
        fa.set_path_policy(0)
    ro, rl = oracle.attention(f32(q), f32(k), f32(v), s, oracle.MASK_CAUSAL, bottom_right=True)
    compare(out.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl, f"M{M} policy{policy}")


# ------------------------------------------------------------------ head dim 96
# Runs on the 128-wide kernels: the tensor maps zero-fill columns 96..127; padding lanes of
# the CUDA-core kernel neither load q nor store out.

@pytest.mark.parametrize("B,M,Mkv,H,Hkv,mask,policy", [
    (2, 300, 700, 2, 2, "causal", 0),    # tensor cores
    (2, 1, 3000, 4, 4, "causal", 0),     # CUDA cores
    (2, 5, 2000, 4, 4, "none", 2),
    (16, 1, 900, 16, 4, "causal", 0),    # folded grouped heads on the tensor cores
])
def test_head_dim_96(B, M, Mkv, H, Hkv, mask, policy):
    q, k, v = inputs.qkv(B, M, Mkv, H, 96, Hkv=Hkv, seed=M + 96)
    s = 96 ** -0.5
    fa.set_path_policy(policy)
    try:
        out, lse = fa.attn_fwd(*to_dev(q, k, v), mask=mask, scale=s, bottom_right=True)
        torch.cuda.synchronize()
    finally:
        fa.set_path_policy(0)
    ro, rl = oracle.attention(f32(q), f32(k), f32(v), s, KIND[mask], bottom_right=True)
    compare(out.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl, f"d96 B{B} M{M} {mask}")


def test_head_dim_96_split_kv_and_fp8():
    q, k, v = inputs.qkv(1, 200, 1500, 2, 96, seed=96)
    s = 96 ** -0.5
    qd, kd, vd = to_dev(q, k, v)
    outs, lses = [], []
    for a, b in inputs.equal_chunks(1500, 3):
        o, l_ = fa.attn_partial(qd, kd[:, a:b], vd[:, a:b], scale=s)
        outs.append(o)
        lses.append(l_)
    out, lse = fa.merge_attentions(torch.stack(outs), torch.stack(lses))
    ro, rl = oracle.attention(f32(q), f32(k), f32(v), s, oracle.MASK_NONE)
    compare(out.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl, "d96 split-KV")
    # E4M3 at head dim 96: decode rows (CUDA cores) and a prefill block (tensor cores)
    from tests.test_fp8_gpu import _check_lse, _deq, _np, _p_rounding_check
    for M in (3, 300):
        q8, dq, k8, dk, v8, dv = inputs.qkv_fp8(1, M, 1200, 2, 96, seed=M)
        o, l_ = fa.attn_fwd_fp8(q8.cuda(), k8.cuda(), v8.cuda(), dq.cuda(), dk.cuda(), dv.cuda(),
                                mask="causal", scale=s, bottom_right=True)
        torch.cuda.synchronize()
        ro, rl = oracle.attention_fp8(_np(q8), _np(k8), _np(v8), _np(dq), _np(dk), _np(dv), s,
                                      oracle.MASK_CAUSAL, bottom_right=True)
        o, l_ = o.double().cpu().numpy(), l_.double().cpu().numpy()
        if M <= 8:
            compare(o, l_, ro, rl, "d96 fp8 decode")
        else:
            _check_lse(l_, rl, "d96 fp8 tc")
            _p_rounding_check(o, ro, _deq(q8, dq), _deq(k8, dk), _deq(v8, dv), s, "causal",
                              "d96 fp8 tc", br=True)


BIG = 2 ** 31


def _repeat_rows(block, rows):
    """Host [1, n, H, D] block -> device [1, rows, H, D] view whose row i is block row i % n."""
    n = block.shape[1]
    return block.cuda().repeat(1, -(-rows // n), 1, 1)[:, :rows]


def _big_memory_ok(gib):
    return torch.cuda.mem_get_info()[0] >= gib << 30


def test_queries_past_2g_elements():
    """q and out with more than 2^31 elements (2,097,452 rows x 8 heads x 128) on the tensor
    cores: rows sampled at the start, middle and ragged end against the oracle."""
    if not _big_memory_ok(24):
        pytest.skip("needs ~9 GB of free device memory")
    H, D, n = 8, 128, 4096
    s = D ** -0.5
    Mq = BIG // (H * D) + 300
    qb, k, v = inputs.qkv(1, n, 256, H, D, seed=21)
    q = _repeat_rows(qb, Mq)
    assert q.numel() > BIG
    out, lse = fa.attn_fwd(q, k.cuda(), v.cuda(), scale=s)
    torch.cuda.synchronize()
    rows = [0, 1, n - 1, Mq // 2, Mq - 300, Mq - 129, Mq - 44, Mq - 1]
    ro, rl = oracle.attention(f32(qb[:, [r % n for r in rows]]), f32(k), f32(v), s, oracle.MASK_NONE)
    compare(out[:, rows].double().cpu().numpy(), lse[:, :, rows].double().cpu().numpy(), ro, rl,
            "queries past 2^31 elements")


@pytest.mark.parametrize("policy", [2, 1])
def test_keys_past_2g_elements(policy):
    """K and V of 513 copies of a 4096-key block (2,101,248 keys x 8 heads x 128, more than
    2^31 elements each): every key appears 513 times, so out equals attention over the block
    and lse is the block's plus ln 513.  CUDA-core decode (cluster split) and tensor cores."""
    if not _big_memory_ok(24):
        pytest.skip("needs ~9 GB of free device memory")
    H, D, n = 8, 128, 4096
    s = D ** -0.5
    R = BIG // (H * D * n) + 1
    q, kb, vb = inputs.qkv(1, 1, n, H, D, seed=22)
    k, v = _repeat_rows(kb, R * n), _repeat_rows(vb, R * n)
    assert k.numel() > BIG
    ro, rl = oracle.attention(f32(q), f32(kb), f32(vb), s, oracle.MASK_NONE)
    fa.set_path_policy(policy)
    try:
        out, lse = fa.attn_fwd(q.cuda(), k, v, scale=s)
        torch.cuda.synchronize()
    finally:
        fa.set_path_policy(0)
    compare(out.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl + np.log(R),
            f"keys past 2^31 elements, policy {policy}")


def test_merge_past_2g_elements():
    """Two chunk results of [1, 2,097,216 rows, 8, 128] fp32 (more than 2^31 elements in the
    stack): sampled rows against the oracle's merge of the block they repeat."""
    if not _big_memory_ok(32):
        pytest.skip("needs ~13 GB of free device memory")
    H, D, n = 8, 128, 4096
    M = BIG // (2 * H * D) + 64
    g = torch.Generator().manual_seed(23)
    ob = torch.randn(2, 1, n, H, D, generator=g)
    lb = torch.randn(2, 1, H, n, generator=g) * 4
    reps = -(-M // n)
    outs = ob.cuda().repeat(1, 1, reps, 1, 1)[:, :, :M]
    lses = lb.cuda().repeat(1, 1, 1, reps)[..., :M].contiguous()
    assert outs.numel() > BIG
    out, lse = fa.merge_attentions(outs, lses)
    torch.cuda.synchronize()
    rows = [0, n - 1, M // 2, M - 65, M - 1]
    ro, rl = oracle.merge_attentions(ob[:, :, [r % n for r in rows]].numpy(),
                                     lb[..., [r % n for r in rows]].numpy())
    compare(out[:, rows].double().cpu().numpy(), lse[..., rows].double().cpu().numpy(), ro, rl,
            "merge past 2^31 elements")


@pytest.mark.parametrize("B,Mkv,H,Hkv,D,mask,br,wl", [
    (64, 256, 8, 1, 128, "none", False, None),      # exactly two key tiles: one per Q tile
    (64, 300, 16, 2, 64, "causal", True, None),     # three key tiles (odd count), head dim 64
    (4, 1000, 128, 1, 128, "none", False, None),    # 128 folded rows: the largest split unit
    (8, 700, 32, 4, 128, "causal", True, 200),      # window: each tile masks its own key tiles
    (16, 129, 8, 2, 128, "none", False, None),      # second key tile holds a single key
])
def test_split_units(B, Mkv, H, Hkv, D, mask, br, wl):
    """Folded decode units (rows fit one Q tile) give both Q tiles the same rows and
    alternate key tiles, merged by log-sum-exp at the epilogue: forward (bf16 out) and
    partial (fp32 out) against the oracle."""
    q, k, v = inputs.qkv(B, 1, Mkv, H, D, Hkv=Hkv, seed=B + Mkv + H)
    s = D ** -0.5
    ro, rl = oracle.attention(f32(q), f32(k), f32(v), s, KIND[mask], bottom_right=br,
                              window_left=wl)
    fa.set_path_policy(1)
    try:
        out, lse = fa.attn_fwd(*to_dev(q, k, v), mask=mask, scale=s, bottom_right=br,
                               window_left=wl)
        shift = (Mkv - 1) if br else 0
        po, pl = fa.attn_partial(*to_dev(q, k, v), mask=mask, scale=s, kv_offset=-shift,
                                 window_left=wl)
        torch.cuda.synchronize()
    finally:
        fa.set_path_policy(0)
    what = f"split B{B} Mkv{Mkv} H{H}/{Hkv} D{D} {mask}"
    compare(out.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl, what)
    compare(po.double().cpu().numpy(), pl.double().cpu().numpy(), ro, rl, what + " partial")
