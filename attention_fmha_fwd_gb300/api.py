"""PyTorch-facing calls over the C ABI: marshal tensors into pointers, strides and sizes.

PyTorch supplies device memory and the stream; every step of the computation runs in
libmslk_attn.so's CUDA kernels.  The calls mirror MSLK's fMHA API ("Attention - Core
fMHA"): forward with optional LSE, partial attention over one K/V chunk, and the exact
LSE merge.
"""

from __future__ import annotations

import ctypes
from typing import Sequence

import torch

from . import _capi
from ._capi import MslkError, Seqlens, Strides, check

MASKS = {
    "none": _capi.MASK_NONE,
    "causal": _capi.MASK_CAUSAL,
    "blockdiag": _capi.MASK_BLOCKDIAG,
    "blockdiag_causal": _capi.MASK_BLOCKDIAG_CAUSAL,
    "causal_bottom_right": _capi.MASK_CAUSAL_BOTTOM_RIGHT,
    "blockdiag_causal_bottom_right": _capi.MASK_BLOCKDIAG_CAUSAL_BOTTOM_RIGHT,
}
_BLOCKDIAG = (_capi.MASK_BLOCKDIAG, _capi.MASK_BLOCKDIAG_CAUSAL, _capi.MASK_BLOCKDIAG_CAUSAL_BOTTOM_RIGHT)
_DTYPES = {torch.bfloat16: _capi.DTYPE_BF16, torch.float32: _capi.DTYPE_FP32}


def _mask_kind(mask) -> int:
    if isinstance(mask, str):
        if mask not in MASKS:
            raise ValueError(f"unknown mask {mask!r}; expected one of {sorted(MASKS)}")
        return MASKS[mask]
    return int(mask)


def _ptr(t):
    return None if t is None else t.data_ptr()


# The raw handle of the current stream without building a torch.cuda.Stream object
# (a few microseconds per call); torch.cuda.current_stream() where that is unavailable.
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream_handle(stream, device=None) -> int:
    if stream is not None:
        return stream.cuda_stream
    index = device.index if device is not None else None
    if index is None:
        index = torch.cuda.current_device()
    if _raw_stream is not None:
        return _raw_stream(index)
    return torch.cuda.current_stream(index).cuda_stream


def _bmhk_strides(t: torch.Tensor, name: str) -> Strides:
    st = t.stride()
    if len(st) != 4:
        raise ValueError(f"{name} must be [B, M, H, D], got shape {tuple(t.shape)}")
    if st[3] != 1 and t.shape[3] > 1:
        raise ValueError(f"{name}: the last dimension must have stride 1")
    return Strides(st[0], st[1], st[2])


def _as_bmhk(t: torch.Tensor) -> torch.Tensor:
    """BMK -> BM1K (a view); BMHK unchanged."""
    if t.dim() == 3:
        return t.unsqueeze(2)
    return t


def _merge_heads(t: torch.Tensor, name: str) -> torch.Tensor:
    """[B, M, G, H, D] -> a [B, M, G * H, D] view (group-major head index g * H + h).

    Raises instead of copying when the (G, H) axes cannot be viewed as one."""
    B, M, G, H, D = t.shape
    if G > 1 and H > 1 and t.stride(2) != H * t.stride(3):
        raise ValueError(f"{name}: the G and H axes of a BMGHK tensor must be adjacent in memory "
                         f"(stride(2) == H * stride(3)) to flatten without a copy")
    return t.as_strided((B, M, G * H, D),
                        (t.stride(0), t.stride(1), t.stride(3) if H > 1 else t.stride(2), t.stride(4)))


def _bmghk(q, k, v):
    """The pages' 5-D BMGHK layout flattened to BMHK views (bmghk2bmhk), no copies.

    q [B, M, G, H, K]; k, v [B, Mkv, G, H or 1, K].  K/V that hold one head per group, or are
    expanded over H with stride 0 (the pages' way of sharing K/V within a group), become
    G K/V heads (grouped-query attention: query head g * H + h reads K/V head g); K/V with
    H distinct heads per group become G * H heads.  Returns (q4, k4, v4, G, H).
    """
    if k.dim() != 5 or v.dim() != 5:
        raise ValueError("a 5-D (BMGHK) q needs 5-D k and v")
    B, M, G, H, K = q.shape
    if k.shape[2] != G or v.shape[2] != G:
        raise ValueError(f"k/v have {k.shape[2]}/{v.shape[2]} groups, q has {G}")

    def kv_view(t, name):
        if t.shape[3] == 1 or t.stride(3) == 0:  # one K/V head per group
            return t.select(3, 0)
        if t.shape[3] != H:
            raise ValueError(f"{name} must have 1 or {H} heads per group (got {t.shape[3]})")
        return _merge_heads(t, name)

    return _merge_heads(q, "q"), kv_view(k, "k"), kv_view(v, "v"), G, H


def _check_inputs(q, k, v):
    bf16 = torch.bfloat16
    if q.dtype is bf16 and k.dtype is bf16 and v.dtype is bf16 and q.is_cuda and k.is_cuda and v.is_cuda:
        return
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor (the library reads device memory)")
        if t.dtype != torch.bfloat16:
            raise ValueError(f"{name} must be bfloat16, got {t.dtype}")


def _kv_heads(q, k, v) -> int:
    """K/V head count, checked against q: equal batch, key count and head dims, and a number
    of K/V heads dividing the query heads (query head h reads K/V head h // (H // Hkv))."""
    qs, ks, vs = q.shape, k.shape, v.shape  # (each .shape builds a new Size: read once)
    H = qs[2]
    if ks[0] != qs[0] or vs[0] != qs[0]:
        raise ValueError("q, k and v must have the same batch size")
    if ks[1] != vs[1] or ks[2] != vs[2]:
        raise ValueError("k and v must have the same number of keys and heads")
    if ks[3] != qs[3]:
        raise ValueError("q and k head dims differ")
    Hkv = ks[2]
    if Hkv < 1 or H % Hkv:
        raise ValueError(f"k/v heads ({Hkv}) must divide the query heads ({H})")
    return Hkv


def _addr(x):
    """Address of a ctypes struct, or of the struct behind ctypes.byref(...); None stays None."""
    if x is None:
        return None
    return ctypes.addressof(x if isinstance(x, ctypes.Structure) else x._obj)


def _args(q, k, v, Hkv, mk, scale, sl, band, out, out_dtype, lse, *, lanes=None, fp8=None,
          partial=0, kv_offset=0, flags=0, ptrs=True):
    """The mslk_attn_args struct of a call (ptrs=False: sizes only, null pointers)."""
    B, M, H, K = q.shape
    a = _capi.AttnArgs()
    if ptrs:
        a.q, a.k, a.v = q.data_ptr(), k.data_ptr(), v.data_ptr()
        a.out, a.lse = out.data_ptr(), _ptr(lse)
    a.sq, a.sk, a.sv = _bmhk_strides(q, "q"), _bmhk_strides(k, "k"), _bmhk_strides(v, "v")
    a.so = _bmhk_strides(out, "out")
    a.B, a.M, a.Mkv, a.H, a.Hkv, a.K, a.Kv = B, M, k.shape[1], H, Hkv, K, v.shape[3]
    a.scale = 0.0 if scale is None else float(scale)
    a.mask_kind = mk
    a.seqlens, a.band, a.lanes, a.fp8 = _addr(sl), _addr(band), _addr(lanes), _addr(fp8)
    a.partial, a.kv_offset = int(partial), int(kv_offset)
    a.out_dtype = _DTYPES[out_dtype]
    a.flags = int(flags)
    a._keep = (band, lanes, fp8)  # the structs the pointers above refer to
    return a


def _general(q, k, v, Hkv, mk, scale, sl, band, out, out_dtype, lse, stream, *, lanes=None,
             fp8=None, partial=0, kv_offset=0, flags=0):
    """mslk_attn with every option in one argument struct (grouped K/V heads)."""
    a = _args(q, k, v, Hkv, mk, scale, sl, band, out, out_dtype, lse, lanes=lanes, fp8=fp8,
              partial=partial, kv_offset=kv_offset, flags=flags)
    check(_capi.load().mslk_attn(ctypes.byref(a), _stream_handle(stream, q.device)))


def _band(bottom_right, window_left, window_right):
    """mslk_band for the *_band entry points, or None when the plain call suffices."""
    if not bottom_right and window_left is None and window_right is None:
        return None
    return _capi.Band(1 if bottom_right else 0, -1 if window_left is None else int(window_left),
                      -1 if window_right is None else int(window_right))


def _seqlens(mask_kind, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k):
    if mask_kind not in _BLOCKDIAG:
        return None, ()
    if cu_seqlens_q is None or cu_seqlens_k is None:
        raise ValueError("block-diagonal masks need cu_seqlens_q and cu_seqlens_k")
    keep = []
    cq, ck = cu_seqlens_q, cu_seqlens_k
    if cq.dtype != torch.int32 or not cq.is_cuda or not cq.is_contiguous():
        raise ValueError("cu_seqlens_q must be a contiguous int32 CUDA tensor")
    if ck.dtype != torch.int32 or not ck.is_cuda or not ck.is_contiguous():
        raise ValueError("cu_seqlens_k must be a contiguous int32 CUDA tensor")
    if max_seqlen_q is None or max_seqlen_k is None:
        raise ValueError("block-diagonal masks need max_seqlen_q and max_seqlen_k (host ints)")
    sl = Seqlens(cq.data_ptr(), ck.data_ptr(), cq.numel() - 1, int(max_seqlen_q), int(max_seqlen_k))
    keep.append(sl)
    return ctypes.byref(sl), keep


def attn_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, *, mask="none", scale=None,
             cu_seqlens_q=None, cu_seqlens_k=None, max_seqlen_q=None, max_seqlen_k=None,
             out=None, lse=True, stream=None, bottom_right=False, window_left=None,
             window_right=None, independent=False):
    """Fused attention forward; returns (out, lse) with lse None when ``lse=False``.

    q [B,M,H,K], k [B,Mkv,Hkv,K], v [B,Mkv,Hkv,Kv] bf16 CUDA tensors (Hkv dividing H:
    grouped K/V heads; BMK inputs are viewed as one head), or the 5-D BMGHK layout
    q [B,M,G,H,K], k/v [B,Mkv,G,H or 1,K] (K/V expanded over H share one head per group),
    which returns out [B,M,G,H,Kv] and lse [B,G,H,M].  ``lse`` may be True (allocate),
    False (skip) or an fp32 [B,H,M] tensor.
    ``bottom_right`` / ``window_left`` / ``window_right`` (keys before / after the paired
    key; None = unbounded) select a bottom-right alignment and a local window (the pages'
    ``...FromBottomRight...`` and ``...LocalAttention...`` masks; a causal window of
    ``window_size`` w keys is ``window_left=w - 1``).
    """
    if q.dim() == 5:  # BMGHK: run on flattened views, return out [B,M,G,H,Kv], lse [B,G,H,M]
        q4, k4, v4, G, Hg = _bmghk(q, k, v)
        B, M = q.shape[0], q.shape[1]
        Kv = v.shape[4]
        if out is None:
            out = torch.empty((B, M, G, Hg, Kv), dtype=torch.bfloat16, device=q.device)
        if lse is True:
            lse = torch.empty((B, G, Hg, M), dtype=torch.float32, device=q.device)
        elif lse is False:
            lse = None
        attn_fwd(q4, k4, v4, mask=mask, scale=scale, cu_seqlens_q=cu_seqlens_q,
                 cu_seqlens_k=cu_seqlens_k, max_seqlen_q=max_seqlen_q, max_seqlen_k=max_seqlen_k,
                 out=_merge_heads(out, "out"), lse=False if lse is None else lse.view(B, G * Hg, M),
                 stream=stream, bottom_right=bottom_right, window_left=window_left,
                 window_right=window_right, independent=independent)
        return out, lse
    q, k, v = _as_bmhk(q), _as_bmhk(k), _as_bmhk(v)
    _check_inputs(q, k, v)
    Hkv = _kv_heads(q, k, v)
    B, M, H, K = q.shape
    Mkv, Kv = k.shape[1], v.shape[3]
    mk = _mask_kind(mask)
    if out is None:
        out = torch.empty((B, M, H, Kv), dtype=torch.bfloat16, device=q.device)
    if lse is True:
        lse = torch.empty((B, H, M), dtype=torch.float32, device=q.device)
    elif lse is False:
        lse = None
    sl, _keep = _seqlens(mk, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k)
    band = _band(bottom_right, window_left, window_right)
    if Hkv != H or independent:  # grouped K/V heads, or a launch that may overlap the previous
        _general(q, k, v, Hkv, mk, scale, sl, band, out, torch.bfloat16, lse, stream,
                 flags=_capi.FLAG_INDEPENDENT if independent else 0)
        return out, lse
    sq, sk, sv = _bmhk_strides(q, "q"), _bmhk_strides(k, "k"), _bmhk_strides(v, "v")
    so = _bmhk_strides(out, "out")
    lib = _capi.load()
    sc = 0.0 if scale is None else float(scale)
    if band is None:
        check(lib.mslk_attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), ctypes.byref(sq),
                                ctypes.byref(sk), ctypes.byref(sv), ctypes.byref(so), B, M, Mkv, H,
                                K, Kv, sc, mk, sl, out.data_ptr(), _ptr(lse),
                                _stream_handle(stream, q.device)))
    else:
        check(lib.mslk_attn_fwd_band(q.data_ptr(), k.data_ptr(), v.data_ptr(), ctypes.byref(sq),
                                     ctypes.byref(sk), ctypes.byref(sv), ctypes.byref(so), B, M,
                                     Mkv, H, K, Kv, sc, mk, sl, ctypes.byref(band), out.data_ptr(),
                                     _ptr(lse), _stream_handle(stream, q.device)))
    return out, lse


def _i32_dev(t, name):
    if t is None:
        return None
    if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous int32 CUDA tensor")
    return t


def _pool_rows(t: torch.Tensor, name: str) -> torch.Tensor:
    """[n_pages, page_size, H, D] -> a [1, n_pages * page_size, H, D] view (pages adjacent)."""
    if t.dim() == 4 and t.shape[0] > 1:
        if t.stride(0) != t.shape[1] * t.stride(1):
            raise ValueError(f"{name}: pages must be adjacent rows (stride(0) == page_size * stride(1))")
        return t.as_strided((1, t.shape[0] * t.shape[1], t.shape[2], t.shape[3]),
                            (t.shape[0] * t.stride(0), t.stride(1), t.stride(2), t.stride(3)))
    return t


def attn_fwd_lanes(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, *, seqlen_k, cu_seqlens_q,
                   max_seqlen_q, max_seqlen_k, seqstart_k=None, block_table=None, page_size=None,
                   mask="blockdiag_causal", scale=None, out=None, lse=True, stream=None,
                   bottom_right=False, window_left=None, window_right=None):
    """Forward over per-sequence key lanes: padded (``seqstart_k``) or paged (``block_table``).

    The padded-keys and paged block-diagonal masks of "Attention - Biases & masks": queries
    packed [1, total_q, H, K] with ``cu_seqlens_q``; sequence s sees ``seqlen_k[s]`` keys,
    logical key p at K/V row ``seqstart_k[s] + p`` or, paged, at row
    ``block_table[s, p // page_size] * page_size + p % page_size`` of the pool.  k, v are
    [1, rows, H, K] or a page pool [n_pages, page_size, H, K].  ``mask`` is a block-diagonal
    kind; ``bottom_right=True`` (or "blockdiag_causal_bottom_right") is the causal-with-offset
    alignment (query i of a sequence pairs with key i + seqlen_k - seqlen_q).  Returns
    (out [1, total_q, H, Kv], lse [1, H, total_q] or None).
    """
    q, k, v = _as_bmhk(q), _as_bmhk(k), _as_bmhk(v)
    k, v = _pool_rows(k, "k"), _pool_rows(v, "v")
    _check_inputs(q, k, v)
    Hkv = _kv_heads(q, k, v)
    B, M, H, K = q.shape
    if B != 1:
        raise ValueError("attn_fwd_lanes takes packed queries [1, total_q, H, K]")
    Mkv, Kv = k.shape[1], v.shape[3]
    mk = _mask_kind(mask)
    if mk not in _BLOCKDIAG:
        raise ValueError("key lanes need a block-diagonal mask kind")
    sk_len = _i32_dev(seqlen_k, "seqlen_k")
    start = _i32_dev(seqstart_k, "seqstart_k")
    table = _i32_dev(block_table, "block_table")
    if sk_len is None or (start is None and table is None):
        raise ValueError("attn_fwd_lanes needs seqlen_k and either seqstart_k or block_table")
    max_pages = 0
    if table is not None:
        if table.dim() != 2 or page_size is None:
            raise ValueError("block_table must be [n_seqs, max_pages] with page_size given")
        max_pages = table.shape[1]
    cq = _i32_dev(cu_seqlens_q, "cu_seqlens_q")
    if cq is None:
        raise ValueError("attn_fwd_lanes needs cu_seqlens_q")
    sl = Seqlens(cq.data_ptr(), sk_len.data_ptr(), cq.numel() - 1, int(max_seqlen_q), int(max_seqlen_k))
    lanes = _capi.KvLanes(sk_len.data_ptr(), _ptr(start), _ptr(table),
                          0 if page_size is None else int(page_size), max_pages)
    if out is None:
        out = torch.empty((1, M, H, Kv), dtype=torch.bfloat16, device=q.device)
    if lse is True:
        lse = torch.empty((1, H, M), dtype=torch.float32, device=q.device)
    elif lse is False:
        lse = None
    sq, sk, sv = _bmhk_strides(q, "q"), _bmhk_strides(k, "k"), _bmhk_strides(v, "v")
    so = _bmhk_strides(out, "out")
    band = _band(bottom_right, window_left, window_right)
    if Hkv != H:  # grouped K/V heads
        _general(q, k, v, Hkv, mk, scale, sl, band, out, torch.bfloat16, lse, stream, lanes=lanes)
        return out, lse
    lib = _capi.load()
    check(lib.mslk_attn_fwd_lanes(q.data_ptr(), k.data_ptr(), v.data_ptr(), ctypes.byref(sq),
                                  ctypes.byref(sk), ctypes.byref(sv), ctypes.byref(so), M, Mkv, H, K,
                                  Kv, 0.0 if scale is None else float(scale), mk, ctypes.byref(sl),
                                  ctypes.byref(lanes), None if band is None else ctypes.byref(band),
                                  out.data_ptr(), _ptr(lse), _stream_handle(stream, q.device)))
    return out, lse


_FP8_DTYPES = tuple(d for d in (torch.uint8, getattr(torch, "float8_e4m3fn", None)) if d is not None)


def _descale(x, name, device):
    """A descale argument as a contiguous fp32 device tensor (a Python float -> one value)."""
    if isinstance(x, torch.Tensor):
        if x.dtype != torch.float32 or not x.is_cuda or not x.is_contiguous():
            raise ValueError(f"{name} must be a contiguous float32 CUDA tensor (or a float)")
        return x.reshape(-1)
    return torch.full((1,), float(x), dtype=torch.float32, device=device)


def attn_fwd_fp8(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, descale_q, descale_k, descale_v,
                 *, mask="none", scale=None, cu_seqlens_q=None, cu_seqlens_k=None, max_seqlen_q=None,
                 max_seqlen_k=None, seqlen_k=None, seqstart_k=None, block_table=None, page_size=None,
                 out=None, lse=True, stream=None, bottom_right=False, window_left=None,
                 window_right=None):
    """Forward on FP8 E4M3 q, k, v (uint8 codes or float8_e4m3fn tensors, [B, M, H, K]).

    Element x of head h stands for x * descale[h]: each descale is a float (tensorwise) or
    a float32 CUDA tensor of one value or one per head ([H] for q; [H], or [1] for a shared
    k/v head, for k and v) — the FP8 E4M3 inputs of the pages' Blackwell / FlashAttention-3
    forward backends.  Masks, windows and packed sequences as ``attn_fwd``; key lanes
    (``seqlen_k`` with ``seqstart_k`` or ``block_table`` + ``page_size``) as
    ``attn_fwd_lanes``.  Returns (out bf16 [B, M, H, Kv], lse fp32 [B, H, M] or None).
    """
    q, k, v = _as_bmhk(q), _as_bmhk(k), _as_bmhk(v)
    lanes_mode = seqlen_k is not None
    if lanes_mode:
        k, v = _pool_rows(k, "k"), _pool_rows(v, "v")
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor (the library reads device memory)")
        if t.dtype not in _FP8_DTYPES:
            raise ValueError(f"{name} must hold E4M3 codes (uint8 or float8_e4m3fn), got {t.dtype}")
    Hkv = _kv_heads(q, k, v)
    B, M, H, K = q.shape
    Mkv, Kv = k.shape[1], v.shape[3]
    mk = _mask_kind(mask)
    dq, dk, dv = (_descale(x, n, q.device) for x, n in ((descale_q, "descale_q"),
                                                       (descale_k, "descale_k"),
                                                       (descale_v, "descale_v")))
    sizes = {dq.numel(), dk.numel(), dv.numel()}
    per_tensor = 1 if sizes == {1} else 0
    if not per_tensor:
        hk = 1 if (k.stride(2) == 0 and H > 1) else Hkv
        if dq.numel() != H or dk.numel() != hk or dv.numel() != hk:
            raise ValueError(f"per-head descales need {H} (q) and {hk} (k, v) entries, or one each")
    scales = _capi.Fp8Scales(dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), per_tensor)
    lanes = None
    keep = []
    if lanes_mode:
        sk_len = _i32_dev(seqlen_k, "seqlen_k")
        start = _i32_dev(seqstart_k, "seqstart_k")
        table = _i32_dev(block_table, "block_table")
        if start is None and table is None:
            raise ValueError("key lanes need seqstart_k or block_table")
        max_pages = 0
        if table is not None:
            if table.dim() != 2 or page_size is None:
                raise ValueError("block_table must be [n_seqs, max_pages] with page_size given")
            max_pages = table.shape[1]
        cq = _i32_dev(cu_seqlens_q, "cu_seqlens_q")
        if cq is None or max_seqlen_q is None or max_seqlen_k is None:
            raise ValueError("key lanes need cu_seqlens_q, max_seqlen_q and max_seqlen_k")
        sl_struct = Seqlens(cq.data_ptr(), sk_len.data_ptr(), cq.numel() - 1, int(max_seqlen_q),
                            int(max_seqlen_k))
        keep.append(sl_struct)
        sl = ctypes.byref(sl_struct)
        lanes = _capi.KvLanes(sk_len.data_ptr(), _ptr(start), _ptr(table),
                              0 if page_size is None else int(page_size), max_pages)
    else:
        sl, keep = _seqlens(mk, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k)
    if out is None:
        out = torch.empty((B, M, H, Kv), dtype=torch.bfloat16, device=q.device)
    if lse is True:
        lse = torch.empty((B, H, M), dtype=torch.float32, device=q.device)
    elif lse is False:
        lse = None
    sq, sk, sv = _bmhk_strides(q, "q"), _bmhk_strides(k, "k"), _bmhk_strides(v, "v")
    so = _bmhk_strides(out, "out")
    band = _band(bottom_right, window_left, window_right)
    if Hkv != H:  # grouped K/V heads
        _general(q, k, v, Hkv, mk, scale, sl, band, out, torch.bfloat16, lse, stream, lanes=lanes,
                 fp8=scales)
        return out, lse
    lib = _capi.load()
    check(lib.mslk_attn_fwd_fp8(q.data_ptr(), k.data_ptr(), v.data_ptr(), ctypes.byref(sq),
                                ctypes.byref(sk), ctypes.byref(sv), ctypes.byref(so), B, M, Mkv, H, K,
                                Kv, 0.0 if scale is None else float(scale), mk, sl,
                                None if band is None else ctypes.byref(band),
                                None if lanes is None else ctypes.byref(lanes), ctypes.byref(scales),
                                out.data_ptr(), _ptr(lse), _stream_handle(stream, q.device)))
    return out, lse


# Argument structs of earlier attn_partial calls with caller-provided out and lse, keyed by
# everything they hold (pointers, shapes, strides, dtypes and options): a loop over the same
# buffers (the chunks of a split, a decode step) replays the struct through mslk_attn
# instead of rebuilding 21 ctypes arguments.  The library validates every call either way.
_PARTIAL_ARGS: dict = {}
_PARTIAL_ARGS_MAX = 256


def _partial_key(q, k, v, out, lse, mask, scale, kv_offset, out_dtype, independent):
    return (q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
            q.shape, k.shape, v.shape, out.shape, lse.shape, q.stride(), k.stride(), v.stride(),
            out.stride(), lse.stride(), q.dtype, k.dtype, v.dtype, out.dtype, lse.dtype,
            q.get_device(), mask, scale, kv_offset, out_dtype, independent)


def _remember_partial(key, a):
    if key is None:
        return
    if len(_PARTIAL_ARGS) >= _PARTIAL_ARGS_MAX:
        _PARTIAL_ARGS.clear()
    _PARTIAL_ARGS[key] = a


def attn_partial(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, *, mask="none",
                 scale=None, kv_offset: int = 0, cu_seqlens_q=None, cu_seqlens_k=None,
                 max_seqlen_q=None, max_seqlen_k=None, out_dtype=torch.float32, out=None,
                 lse=None, stream=None, window_left=None, window_right=None, independent=False):
    """Attention over one disjoint K/V chunk; returns (out, lse) for merge_attentions.

    ``kv_offset`` is the position of the chunk's first key (read by causal masks and
    windows; a bottom-right alignment over the full keys is folded into it).
    ``independent=True`` states that q, k and v are not written by the launch just before
    this one on the stream (e.g. the previous chunk of the same split): the call may then
    start while that launch finishes.
    """
    if q.dim() == 5:  # BMGHK: out [B,M,G,H,Kv], lse [B,G,H,M] over flattened views
        q4, k4, v4, G, Hg = _bmghk(q, k, v)
        B, M = q.shape[0], q.shape[1]
        if out is None:
            out = torch.empty((B, M, G, Hg, v.shape[4]), dtype=out_dtype, device=q.device)
        if lse is None:
            lse = torch.empty((B, G, Hg, M), dtype=torch.float32, device=q.device)
        attn_partial(q4, k4, v4, mask=mask, scale=scale, kv_offset=kv_offset,
                     cu_seqlens_q=cu_seqlens_q, cu_seqlens_k=cu_seqlens_k,
                     max_seqlen_q=max_seqlen_q, max_seqlen_k=max_seqlen_k, out_dtype=out_dtype,
                     out=_merge_heads(out, "out"), lse=lse.view(B, G * Hg, M), stream=stream,
                     window_left=window_left, window_right=window_right, independent=independent)
        return out, lse
    q, k, v = _as_bmhk(q), _as_bmhk(k), _as_bmhk(v)
    key = None
    if (out is not None and lse is not None and cu_seqlens_q is None and cu_seqlens_k is None
            and window_left is None and window_right is None):
        key = _partial_key(q, k, v, out, lse, mask, scale, kv_offset, out_dtype, independent)
        a = _PARTIAL_ARGS.get(key)
        if a is not None:
            check(_capi.load().mslk_attn(ctypes.byref(a), _stream_handle(stream, q.device)))
            return out, lse
    _check_inputs(q, k, v)
    Hkv = _kv_heads(q, k, v)
    B, M, H, K = q.shape
    Mkv, Kv = k.shape[1], v.shape[3]
    mk = _mask_kind(mask)
    if out_dtype not in _DTYPES:
        raise ValueError("out_dtype must be torch.float32 or torch.bfloat16")
    if out is None:
        out = torch.empty((B, M, H, Kv), dtype=out_dtype, device=q.device)
    elif out.dtype != out_dtype:
        raise ValueError("out dtype does not match out_dtype")
    if lse is None:
        lse = torch.empty((B, H, M), dtype=torch.float32, device=q.device)
    sl, _keep = _seqlens(mk, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, max_seqlen_k)
    band = _band(False, window_left, window_right)
    if Hkv != H or independent:  # grouped K/V heads, or a launch that may overlap the previous
        a = _args(q, k, v, Hkv, mk, scale, sl, band, out, out_dtype, lse, partial=1,
                  kv_offset=kv_offset, flags=_capi.FLAG_INDEPENDENT if independent else 0)
        check(_capi.load().mslk_attn(ctypes.byref(a), _stream_handle(stream, q.device)))
        _remember_partial(key, a)
        return out, lse
    sq, sk, sv = _bmhk_strides(q, "q"), _bmhk_strides(k, "k"), _bmhk_strides(v, "v")
    so = _bmhk_strides(out, "out")
    lib = _capi.load()
    sc = 0.0 if scale is None else float(scale)
    if band is None:
        check(lib.mslk_attn_partial(q.data_ptr(), k.data_ptr(), v.data_ptr(), ctypes.byref(sq),
                                    ctypes.byref(sk), ctypes.byref(sv), ctypes.byref(so), B, M,
                                    Mkv, H, K, Kv, sc, mk, sl, int(kv_offset), out.data_ptr(),
                                    _DTYPES[out_dtype], lse.data_ptr(),
                                    _stream_handle(stream, q.device)))
        if key is not None:
            _remember_partial(key, _args(q, k, v, H, mk, scale, None, None, out, out_dtype, lse,
                                         partial=1, kv_offset=kv_offset))
    else:
        check(lib.mslk_attn_partial_band(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                         ctypes.byref(sq), ctypes.byref(sk), ctypes.byref(sv),
                                         ctypes.byref(so), B, M, Mkv, H, K, Kv, sc, mk, sl,
                                         ctypes.byref(band), int(kv_offset), out.data_ptr(),
                                         _DTYPES[out_dtype], lse.data_ptr(),
                                         _stream_handle(stream, q.device)))
    return out, lse


def _stacked(parts):
    """Chunks as (base tensor, chunk stride, n), or None when they are not equally spaced
    views of one allocation (then the varargs merge reads them where they lie)."""
    if isinstance(parts, torch.Tensor):
        return parts[0], (parts.stride(0) if parts.shape[0] > 1 else 0), parts.shape[0]
    base = parts[0]
    if len(parts) == 1:
        return base, 0, 1
    es = base.element_size()
    d = parts[1].data_ptr() - base.data_ptr()
    ok = d > 0 and d % es == 0 and all(
        p.shape == base.shape and p.stride() == base.stride() and p.dtype == base.dtype and
        p.data_ptr() - base.data_ptr() == i * d for i, p in enumerate(parts))
    return (base, d // es, len(parts)) if ok else None


def _flat_chunk(o, what):
    """A 5-D BMGHK chunk output [B,M,G,H,Kv] (or lse [B,G,H,M]) as its 4-D / 3-D view."""
    if what == "out" and o.dim() == 5:
        return _merge_heads(o, "out_split chunk")
    if what == "lse" and o.dim() == 4:
        return o.view(o.shape[0], o.shape[1] * o.shape[2], o.shape[3])
    return o


def merge_attentions(out_split, lse_split, *, write_lse=True, output_dtype=torch.bfloat16,
                     out=None, lse=None, stream=None):
    """Exact LSE merge of chunk results; returns (out, lse) with lse None when ``write_lse``
    is False.

    ``out_split`` is a stacked fp32 tensor [n,B,M,H,Kv] or a list of n chunk tensors
    [B,M,H,Kv] (5-D BMGHK chunks [B,M,G,H,Kv] with lse [B,G,H,M] give a 5-D result);
    ``lse_split`` likewise [n,B,H,M] or a list.  Equally spaced views of one allocation go
    to the stacked merge; separately allocated chunks go to the varargs merge, which reads
    each chunk where it lies (nothing is copied or stacked).
    """
    outs = list(out_split.unbind(0)) if isinstance(out_split, torch.Tensor) else list(out_split)
    lses = list(lse_split.unbind(0)) if isinstance(lse_split, torch.Tensor) else list(lse_split)
    if not outs:
        raise MslkError(_capi.MSLK_ERR_INVALID_ARG, "merge_attentions: no chunks")
    if len(outs) != len(lses):
        raise ValueError("different numbers of output and lse chunks")
    five = outs[0].dim() == 5
    if five:
        B, M, G, Hg, Kv = outs[0].shape
        if out is None:
            out = torch.empty((B, M, G, Hg, Kv), dtype=output_dtype, device=outs[0].device)
        if write_lse and lse is None:
            lse = torch.empty((B, G, Hg, M), dtype=torch.float32, device=outs[0].device)
        merge_attentions([_flat_chunk(o, "out") for o in outs], [_flat_chunk(x, "lse") for x in lses],
                         write_lse=write_lse, output_dtype=output_dtype, out=_merge_heads(out, "out"),
                         lse=None if not write_lse else lse.view(B, G * Hg, M), stream=stream)
        return out, (lse if write_lse else None)
    o0, l0 = outs[0], lses[0]
    if any(o.dtype != torch.float32 for o in outs) or any(x.dtype != torch.float32 for x in lses):
        raise ValueError("chunk outputs and lse must be float32")
    if any(not x.is_contiguous() for x in lses):
        raise ValueError("each lse chunk must be a contiguous [B,H,M] tensor")
    B, M, H, Kv = o0.shape
    if any(o.shape != o0.shape or o.stride() != o0.stride() for o in outs):
        raise ValueError("every chunk output must have the same shape and strides")
    if any(x.shape != (B, H, M) for x in lses):
        raise ValueError(f"each lse chunk must be [B,H,M] = {(B, H, M)}")
    if output_dtype not in _DTYPES:
        raise ValueError("output_dtype must be torch.bfloat16 or torch.float32")
    if out is None:
        out = torch.empty((B, M, H, Kv), dtype=output_dtype, device=o0.device)
    if write_lse and lse is None:
        lse = torch.empty((B, H, M), dtype=torch.float32, device=o0.device)
    if not write_lse:
        lse = None
    ss = _bmhk_strides(o0, "out_split")
    so = _bmhk_strides(out, "out")
    lib = _capi.load()
    st_o = out_split if isinstance(out_split, torch.Tensor) else outs
    st_l = lse_split if isinstance(lse_split, torch.Tensor) else lses
    so_, sl_ = _stacked(st_o), _stacked(st_l)
    if so_ is not None and sl_ is not None:
        (ob, cs_o, n), (lb, cs_l, _) = so_, sl_
        check(lib.mslk_merge_attentions(ob.data_ptr(), lb.data_ptr(), n, cs_o, cs_l, B, M, H, Kv,
                                        ctypes.byref(ss), ctypes.byref(so), out.data_ptr(),
                                        _DTYPES[out.dtype], _ptr(lse),
                                        _stream_handle(stream, o0.device)))
        return out, lse
    n = len(outs)
    if n > _capi.MERGE_MAX_VARARGS:
        raise ValueError(f"at most {_capi.MERGE_MAX_VARARGS} separately allocated chunks")
    optrs = (ctypes.c_void_p * n)(*[o.data_ptr() for o in outs])
    lptrs = (ctypes.c_void_p * n)(*[x.data_ptr() for x in lses])
    check(lib.mslk_merge_attentions_varargs(optrs, lptrs, n, B, M, H, Kv, ctypes.byref(ss),
                                            ctypes.byref(so), out.data_ptr(), _DTYPES[out.dtype],
                                            _ptr(lse), _stream_handle(stream, o0.device)))
    return out, lse


def splitk_size(batch: int, seqlen_kv: int, kv_heads: int = 1, tile_n: int = 256,
                sm_count: int | None = None) -> int:
    """Keys per split-KV chunk (0: one split covers the keys); the library's rule for the
    pages' get_splitk_heuristic, host-only (see mslk_splitk_size)."""
    return int(_capi.load().mslk_splitk_size(int(batch), int(seqlen_kv), int(kv_heads), int(tile_n),
                                             0 if sm_count is None else int(sm_count)))


def attn_split_kv(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, *, n_chunks: int = 0,
                  mask="none", scale=None, out=None, lse=True, out_dtype=torch.bfloat16,
                  workspace=None, stream=None, bottom_right=False, window_left=None,
                  window_right=None):
    """Exact split-KV attention in one library call: partials over ``n_chunks`` equal key
    chunks (0: the split-size rule), then the merge.  Dense masks.  Returns (out, lse).

    ``workspace`` (optional) is a uint8 CUDA tensor of at least ``split_kv_workspace_bytes``
    bytes, 256-byte aligned; without it one is allocated here."""
    q, k, v = _as_bmhk(q), _as_bmhk(k), _as_bmhk(v)
    _check_inputs(q, k, v)
    Hkv = _kv_heads(q, k, v)
    B, M, H, K = q.shape
    Kv = v.shape[3]
    if out is None:
        out = torch.empty((B, M, H, Kv), dtype=out_dtype, device=q.device)
    if lse is True:
        lse = torch.empty((B, H, M), dtype=torch.float32, device=q.device)
    elif lse is False:
        lse = None
    a = _args(q, k, v, Hkv, _mask_kind(mask), scale, None, _band(bottom_right, window_left, window_right),
              out, out.dtype, lse)
    lib = _capi.load()
    need = ctypes.c_size_t(0)
    check(lib.mslk_attn_split_kv_workspace(ctypes.byref(a), int(n_chunks), ctypes.byref(need)))
    if workspace is None:
        workspace = torch.empty(max(need.value, 1), dtype=torch.uint8, device=q.device)
    check(lib.mslk_attn_split_kv(ctypes.byref(a), int(n_chunks), workspace.data_ptr(),
                                 workspace.numel() * workspace.element_size(),
                                 _stream_handle(stream, q.device)))
    return out, lse


def attn_split_kv_static(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, *, n_chunks: int = 0,
                         mask="none", scale=None, out=None, lse=True, out_dtype=torch.bfloat16,
                         stream=None, bottom_right=False, window_left=None, window_right=None):
    """``attn_split_kv`` for callers that cannot allocate device memory when they call: the
    library keeps the workspace in a fixed array of ``SPLIT_KV_STATIC_BYTES`` per device (see
    mslk_attn_split_kv_static).  With ``out`` and ``lse`` given, nothing is allocated; calls
    that overlap on the GPU share the array and race, so keep them on one stream."""
    q, k, v = _as_bmhk(q), _as_bmhk(k), _as_bmhk(v)
    _check_inputs(q, k, v)
    Hkv = _kv_heads(q, k, v)
    B, M, H, K = q.shape
    Kv = v.shape[3]
    if out is None:
        out = torch.empty((B, M, H, Kv), dtype=out_dtype, device=q.device)
    if lse is True:
        lse = torch.empty((B, H, M), dtype=torch.float32, device=q.device)
    elif lse is False:
        lse = None
    a = _args(q, k, v, Hkv, _mask_kind(mask), scale, None, _band(bottom_right, window_left, window_right),
              out, out.dtype, lse)
    check(_capi.load().mslk_attn_split_kv_static(ctypes.byref(a), int(n_chunks),
                                                 _stream_handle(stream, q.device)))
    return out, lse


SPLIT_KV_STATIC_BYTES = _capi.SPLIT_KV_STATIC_BYTES


def split_kv_workspace_bytes(q, k, v, *, n_chunks: int = 0, mask="none", out_dtype=torch.bfloat16,
                             bottom_right=False, window_left=None, window_right=None) -> int:
    """Bytes of workspace ``attn_split_kv`` needs for these tensors and chunk count."""
    q, k, v = _as_bmhk(q), _as_bmhk(k), _as_bmhk(v)
    Hkv = _kv_heads(q, k, v)
    B, M, H, K = q.shape
    out = torch.empty((B, M, H, v.shape[3]), dtype=out_dtype, device="meta")
    a = _args(q, k, v, Hkv, _mask_kind(mask), None, None, _band(bottom_right, window_left, window_right),
              out, out_dtype, None, ptrs=False)
    need = ctypes.c_size_t(0)
    check(_capi.load().mslk_attn_split_kv_workspace(ctypes.byref(a), int(n_chunks), ctypes.byref(need)))
    return int(need.value)


def device_status(stream=None) -> int:
    """Synchronise ``stream``; return the status of the device error word (and clear it)."""
    return int(_capi.load().mslk_device_status(_stream_handle(stream)))


def set_wait_timeout_ns(ns: int) -> None:
    _capi.load().mslk_set_wait_timeout_ns(int(ns))


def diag_bounded_wait(stream=None) -> None:
    check(_capi.load().mslk_diag_bounded_wait(_stream_handle(stream)))


def set_path_policy(policy: int) -> None:
    """0 automatic, 1 always the tensor-core kernel."""
    _capi.load().mslk_set_path_policy(int(policy))


def last_error() -> str:
    r = _capi.load().mslk_last_error()
    return r.decode() if r else ""


def version() -> int:
    return int(_capi.load().mslk_version())


__all__: Sequence[str] = [
    "attn_fwd", "attn_partial", "merge_attentions", "attn_split_kv", "attn_split_kv_static",
    "split_kv_workspace_bytes",
    "splitk_size", "device_status", "set_wait_timeout_ns",
    "diag_bounded_wait", "set_path_policy", "last_error", "version", "MslkError", "MASKS",
]
