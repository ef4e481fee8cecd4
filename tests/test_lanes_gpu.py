"""Key lanes (padded and paged K/V): CUDA path vs the fp64 oracle, through the C ABI.

The padded-keys and paged block-diagonal masks of "Attention - Biases & masks"
(BlockDiagonalPaddedKeysMask, BlockDiagonalCausalWithOffsetPaddedKeysMask,
PagedBlockDiagonalPaddedKeysMask and the local variants), in the reading the oracle
documents: sequence s sees seqlen_k[s] keys of its lane; rows past them are never used.
Every row or page no lane owns is filled with NaN here, so reading one shows up.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import attention_fmha_fwd_gb300 as fa
import oracle
from attention_fmha_fwd_gb300 import inputs
from tests.gpu_util import compare, f32

pytestmark = pytest.mark.gpu

KINDS = {"blockdiag": oracle.MASK_BLOCKDIAG, "blockdiag_causal": oracle.MASK_BLOCKDIAG_CAUSAL}


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


def _paged(lq, lk, page_size, H=4, D=128, mask="blockdiag_causal", br=True, wl=None, hkv=None,
           seed=0, policy=0):
    hkv = H if hkv is None else hkv
    total_q = sum(lq)
    table, n_pages, spare = inputs.page_table(lk, page_size, spare_pages=2, seed=seed)
    q, k, v = inputs.qkv(1, total_q, n_pages * page_size, H, D, Hkv=hkv, seed=seed)
    # poison: the spare pages and every lane's rows past its last key
    k = k.clone()
    v = v.clone()
    own = np.zeros(n_pages * page_size, dtype=bool)
    for s, n in enumerate(lk):
        own[oracle.lane_rows(s, lk, block_table=table.numpy(), page_size=page_size)] = True
    k[0, torch.from_numpy(~own)] = float("nan")
    v[0, torch.from_numpy(~own)] = float("nan")
    scale = 1 / D ** 0.5
    kd = k.cuda().view(n_pages, page_size, hkv, D)  # the pool as [pages, page_size, H, D]
    vd = v.cuda().view(n_pages, page_size, hkv, D)
    if hkv == 1 and H > 1:
        kd, vd = kd.expand(-1, -1, H, -1), vd.expand(-1, -1, H, -1)
    fa.set_path_policy(policy)
    try:
        out, lse = fa.attn_fwd_lanes(q.cuda(), kd, vd, seqlen_k=_i32(lk),
                                     cu_seqlens_q=_i32(inputs.cu_seqlens(lq)),
                                     max_seqlen_q=max(lq), max_seqlen_k=max(lk),
                                     block_table=table.cuda(), page_size=page_size, mask=mask,
                                     scale=scale, bottom_right=br, window_left=wl)
        torch.cuda.synchronize()
    finally:
        fa.set_path_policy(0)
    ro, rl = oracle.attention_lanes(f32(q), f32(k), f32(v), scale, KINDS[mask],
                                    inputs.cu_seqlens(lq), lk, block_table=table.numpy(),
                                    page_size=page_size, bottom_right=br, window_left=wl)
    compare(out.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl,
            f"paged lq{lq} lk{lk} ps{page_size} {mask} br{br} wl{wl} hkv{hkv} policy{policy}")


@pytest.mark.parametrize("page_size", [64, 128, 256])
def test_paged_decode(page_size):
    """One query per sequence (decode kernel), lanes ragged against pages and tiles."""
    lk = [1, 63, 64, 700, 3001, 0, 129]
    _paged([1] * len(lk), lk, page_size, seed=page_size)


@pytest.mark.parametrize("lq,mask,br,wl", [
    ([1, 3, 8, 0, 5], "blockdiag_causal", True, None),   # a few queries per sequence
    ([2, 8, 4, 1, 7], "blockdiag", False, None),
    ([8, 1, 6, 3, 2], "blockdiag_causal", True, 200),    # local window on a lane
])
def test_paged_few_queries(lq, mask, br, wl):
    _paged(lq, [1500, 90, 2049, 64, 333], 64, mask=mask, br=br, wl=wl, seed=len(lq) + (wl or 0))


@pytest.mark.parametrize("hkv,rows", [(8, 4), (2, 1)])
def test_paged_small_pages_many_units(hkv, rows):
    """64-key pages (accepted for a few queries per sequence) with enough (sequence, head)
    units that the tensor cores would be the faster choice (up to 4 queries per sequence;
    or one query with the 4 query heads of each K/V head folded): the dispatch keeps such
    pages on the CUDA-core kernel, since a 128-key tile would straddle pages."""
    g = torch.Generator().manual_seed(17)
    lk = torch.randint(100, 2500, (40,), generator=g).tolist()
    lq = [rows if i % 3 else 1 for i in range(40)]
    _paged(lq, lk, 64, H=8, hkv=hkv, seed=17 + hkv)


def test_paged_shared_kv_head():
    """Multi-query: one K/V head in the pool (head stride 0) serves every query head."""
    _paged([1, 4, 2], [1000, 77, 4100], 128, H=8, hkv=1, seed=3)


@pytest.mark.parametrize("lq,lk,page_size,D,mask,br,wl", [
    ([100, 257, 1, 130], [300, 257, 900, 129], 128, 128, "blockdiag_causal", True, None),
    ([300, 64, 129], [300, 1000, 129], 256, 64, "blockdiag", False, None),
    ([200, 513], [700, 513], 128, 128, "blockdiag_causal", True, 150),
])
def test_paged_prefill_tensor_core(lq, lk, page_size, D, mask, br, wl):
    """Sequences of more than 8 queries (tensor-core kernel, 128-key tiles in pages)."""
    _paged(lq, lk, page_size, D=D, mask=mask, br=br, wl=wl, seed=sum(lq))


def test_paged_decode_on_tensor_core_path():
    """The same few-query lanes forced onto the tensor-core kernel."""
    _paged([1, 5, 2], [800, 129, 2000], 128, policy=1, seed=11)


@pytest.mark.parametrize("lq,pad,mask,br,policy", [
    ([1, 1, 1, 1], 1024, "blockdiag_causal", True, 0),
    ([3, 8, 1], 2048, "blockdiag", False, 0),
    ([100, 300, 7], 1024, "blockdiag_causal", True, 0),
    ([1, 2, 6], 1024, "blockdiag_causal", True, 1),
])
def test_padded_lanes(lq, pad, mask, br, policy):
    """Lanes at seqstart_k = s * pad, with seqlen_k[s] <= pad valid keys each."""
    n = len(lq)
    lk = [pad - 1 - 37 * s for s in range(n)]
    lk[-1] = max(1, pad // 3)
    start = [s * pad for s in range(n)]
    H, D = 4, 128
    q, k, v = inputs.qkv(1, sum(lq), n * pad, H, D, seed=pad + n)
    k, v = k.clone(), v.clone()
    for s in range(n):
        k[0, start[s] + lk[s]:start[s] + pad] = float("nan")
        v[0, start[s] + lk[s]:start[s] + pad] = float("nan")
    scale = 1 / D ** 0.5
    fa.set_path_policy(policy)
    try:
        out, lse = fa.attn_fwd_lanes(q.cuda(), k.cuda(), v.cuda(), seqlen_k=_i32(lk),
                                     seqstart_k=_i32(start),
                                     cu_seqlens_q=_i32(inputs.cu_seqlens(lq)),
                                     max_seqlen_q=max(lq), max_seqlen_k=max(lk), mask=mask,
                                     scale=scale, bottom_right=br)
        torch.cuda.synchronize()
    finally:
        fa.set_path_policy(0)
    ro, rl = oracle.attention_lanes(f32(q), f32(k), f32(v), scale, KINDS[mask],
                                    inputs.cu_seqlens(lq), lk, seqstart_k=start, bottom_right=br)
    compare(out.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl,
            f"padded lq{lq} pad{pad} {mask} br{br} policy{policy}")


def test_paged_equals_contiguous():
    """A paged pool gives the same bits as the same keys laid out contiguously (cu_seqlens_k)."""
    lq, lk, ps = [1, 1, 1], [1000, 3000, 257], 128
    table, n_pages, _ = inputs.page_table(lk, ps, seed=2)
    q, k, v = inputs.qkv(1, 3, n_pages * ps, 4, 128, seed=2)
    rows = np.concatenate([oracle.lane_rows(s, lk, block_table=table.numpy(), page_size=ps)
                           for s in range(3)])
    kc, vc = k[:, rows].contiguous().cuda(), v[:, rows].contiguous().cuda()
    cq, ck = _i32(inputs.cu_seqlens(lq)), _i32(inputs.cu_seqlens(lk))
    a = fa.attn_fwd(q.cuda(), kc, vc, mask="blockdiag_causal", cu_seqlens_q=cq, cu_seqlens_k=ck,
                    max_seqlen_q=1, max_seqlen_k=max(lk), bottom_right=True)
    b = fa.attn_fwd_lanes(q.cuda(), k.cuda(), v.cuda(), seqlen_k=_i32(lk), cu_seqlens_q=cq,
                          max_seqlen_q=1, max_seqlen_k=max(lk), block_table=table.cuda(),
                          page_size=ps, bottom_right=True)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_paged_full_size_sampled():
    """128 decode lanes of up to 16384 keys in 256-key pages (the paged-decode benchmark
    shape), checked on a sample of lanes against the oracle."""
    n, ps, H, D = 128, 256, 8, 128
    g = torch.Generator().manual_seed(21)
    lk = torch.randint(1, 16385, (n,), generator=g).tolist()
    lq = [1] * n
    table, n_pages, _ = inputs.page_table(lk, ps, seed=21)
    q, k, v = inputs.qkv(1, n, n_pages * ps, H, D, seed=21)
    scale = 1 / D ** 0.5
    out, lse = fa.attn_fwd_lanes(q.cuda(), k.cuda(), v.cuda(), seqlen_k=_i32(lk),
                                 cu_seqlens_q=_i32(inputs.cu_seqlens(lq)), max_seqlen_q=1,
                                 max_seqlen_k=max(lk), block_table=table.cuda(), page_size=ps,
                                 bottom_right=True)
    out, lse = out.double().cpu().numpy(), lse.double().cpu().numpy()
    kf, vf = f32(k), f32(v)
    for s in (0, 17, 64, 127):
        ro, rl = oracle.attention_lanes(f32(q[:, s:s + 1]), kf, vf, scale,
                                        oracle.MASK_BLOCKDIAG_CAUSAL, [0, 1], [lk[s]],
                                        block_table=table[s:s + 1].numpy(), page_size=ps,
                                        bottom_right=True)
        compare(out[:, s:s + 1], lse[:, :, s:s + 1], ro, rl, f"lane {s} of {n} (Lk {lk[s]})")
