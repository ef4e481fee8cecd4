"""fp64 CPU oracle for fused multi-head attention forward, split-KV partial, and LSE merge.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or links this
module: only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg use it.  It shares no code with the CUDA library and imports nothing from it.

What it computes is the plain definition of the method, written out in float64 with
the score matrix materialised (MSLK kernel reference, "Attention - Core fMHA" >
``memory_efficient_attention``: scaled Q.K^T, bias/mask, softmax, times V; the fused
kernels reach the same result without materialising the scores):

    x[i, j]   = scale * sum_k q[b, i, h, k] * k[b, j, h, k]          (j in A_i)
    m_i       = max_{j in A_i} x[i, j]
    l_i       = sum_{j in A_i} exp(x[i, j] - m_i)
    out[b,i,h]= sum_{j in A_i} exp(x[i, j] - m_i) * v[b, j, h, :] / l_i
    lse[b,h,i]= m_i + ln(l_i)                   (natural log; includes the scale)

Subtracting m_i is an exact rewrite of softmax (the factor exp(-m_i) cancels).  A row
whose allowed set A_i is empty returns out = 0 and lse = -inf (the pages are silent
here; this is the only reading under which the LSE merge stays exact).

Allowed sets (MSLK kernel reference, "Attention - Biases & masks"):
  * MASK_NONE               every key j < Mkv.
  * MASK_CAUSAL             ``LowerTriangularMask``: top-left aligned, keep key j iff
                            its global position kv_offset + j <= i (zeros on and below
                            the diagonal, -inf above).
  * MASK_BLOCKDIAG          ``BlockDiagonalMask``: packed sequences (B = 1); query i in
                            sequence s sees exactly the keys of sequence s.
  * MASK_BLOCKDIAG_CAUSAL   ``BlockDiagonalCausalMask``: as above plus top-left causal
                            inside each block, on positions relative to the block
                            starts (kv_offset added to the key position).

Alignment and local windows (same page: ``LowerTriangularFromBottomRightMask``,
``LowerTriangularFromBottomRightLocalAttentionMask``, ``LocalAttentionFromBottomRightMask``,
``BlockDiagonalCausalFromBottomRightMask``, ``BlockDiagonalCausalLocalAttentionMask``,
``BlockDiagonalCausalLocalAttentionFromBottomRightMask``).  The pages name these without
formulas; the reading used here is the plainest one, on positions p_i (query) and p_j
(key, kv_offset added) inside a block of Lq queries and Lk keys:
  * ``bottom_right``: the diagonal is moved so that the last query lines up with the last
    key: shift = Lk - Lq (0 for top-left alignment);
  * causal kinds keep p_j - p_i <= shift;
  * ``window_left`` = wl keeps p_j - p_i >= shift - wl (a causal local window of
    ``window_size`` w keeps the w keys ending at the diagonal: wl = w - 1);
  * ``window_right`` = wr (non-causal kinds only) keeps p_j - p_i <= shift + wr.
So every mask is a band  lo <= p_j - p_i <= hi  (either side possibly unbounded).

Padded and paged key lanes (same page: ``BlockDiagonalPaddedKeysMask``,
``BlockDiagonalCausalWithOffsetPaddedKeysMask``, ``PagedBlockDiagonalPaddedKeysMask`` and
their local variants; again named without formulas, plainest reading): queries are packed
as for the block-diagonal masks; sequence s owns a key lane holding its ``seqlen_k[s]``
valid keys, logical key p of the lane living at K/V row ``seqstart_k[s] + p`` (padded
lanes) or, paged, at row ``block_table[s][p // page_size] * page_size + p % page_size`` of
a pool of pages.  Rows beyond a lane's valid keys are never read.  The masks then act on
the logical positions as for the block-diagonal kinds (``...CausalWithOffset...`` is the
bottom-right alignment).

Partial attention (``memory_efficient_attention_partial``) is the same definition over
one disjoint key/value chunk; ``kv_offset`` is the chunk's first key position, used only
by the causal masks.

Merge (``merge_attentions``: the exact normalised output over the union of chunks, not
an average):

    LSE      = ln sum_c exp(lse_c)          = M* + ln sum_c exp(lse_c - M*),  M* = max_c lse_c
    out      = sum_c exp(lse_c - LSE) * out_c
    (M* = -inf, i.e. every chunk empty:  out = 0, LSE = -inf)

Inputs are arrays of any float dtype holding the exact bf16 values; they are widened to
float64 here.  ``scale`` is the float32 value the library receives, widened to float64.
Heads of K/V: Hk dividing H.  Query head h reads K/V head h // (H / Hk): grouped-query
attention in the pages' BMGHK layout flattened group-major (query head g * (H / Hk) + i
belongs to group g, whose keys and values are shared; ``bmghk2bmhk``).  Hk = H is plain
multi-head attention; Hk = 1 is one head shared by every query head (what a stride-0
head expansion denotes).

Parity pins for every function here live in ``tests/oracle_pins.py``.
"""

from __future__ import annotations

import math

import numpy as np

MASK_NONE = 0
MASK_CAUSAL = 1
MASK_BLOCKDIAG = 2
MASK_BLOCKDIAG_CAUSAL = 3

_BLOCKDIAG_KINDS = (MASK_BLOCKDIAG, MASK_BLOCKDIAG_CAUSAL)


def widen_bf16_bits(bits: np.ndarray) -> np.ndarray:
    """Exact float64 values of raw bf16 bit patterns (uint16): bf16 is the top half of fp32."""
    u32 = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):
        return u32.view(np.float32).astype(np.float64)


def default_scale(K: int) -> float:
    """Scale used when the caller passes none: 1/sqrt(K) (``scale=None`` in the pages)."""
    return 1.0 / math.sqrt(K)


def _scale64(scale: float) -> float:
    # The library receives the scale as float32; the oracle uses that exact value.
    return float(np.float32(scale))


def _band(mask_kind, bottom_right, window_left, window_right, Lq, Lk):
    """(lo, hi) bounds on p_j - p_i for a block of Lq queries and Lk keys (None = open)."""
    if window_left is not None and window_left < 0:
        raise ValueError("window_left must be >= 0")
    if window_right is not None and window_right < 0:
        raise ValueError("window_right must be >= 0")
    causal = mask_kind in (MASK_CAUSAL, MASK_BLOCKDIAG_CAUSAL)
    if causal and window_right not in (None, 0):
        raise ValueError("causal masks have no right window")
    shift = (Lk - Lq) if bottom_right else 0
    if causal:
        hi = shift
    else:
        hi = None if window_right is None else shift + window_right
    lo = None if window_left is None else shift - window_left
    return lo, hi


def _block(qb, kb, vb, scale64, lo, hi, q_pos0, k_pos0):
    """Attention of one query block against one key block (one batch, one head).

    qb [Lq, K], kb [Lk, K], vb [Lk, Kv] in float64.  Key j is allowed for query i iff
    lo <= (k_pos0 + j) - (q_pos0 + i) <= hi (a None bound is open).
    Returns out [Lq, Kv] and lse [Lq].
    """
    Lq, Lk = qb.shape[0], kb.shape[0]
    x = scale64 * (qb @ kb.T)                                   # [Lq, Lk]
    if lo is not None or hi is not None:
        d = (k_pos0 + np.arange(Lk)[None, :]) - (q_pos0 + np.arange(Lq)[:, None])
        allowed = np.ones((Lq, Lk), dtype=bool)
        if hi is not None:
            allowed &= d <= hi
        if lo is not None:
            allowed &= d >= lo
        x = np.where(allowed, x, -np.inf)
    if Lk == 0:
        m = np.full(Lq, -np.inf)
    else:
        m = x.max(axis=1)                                       # -inf for empty rows
    empty = np.isneginf(m)
    p = np.exp(x - np.where(empty, 0.0, m)[:, None])            # masked entries -> 0
    l = p.sum(axis=1)
    with np.errstate(invalid="ignore", divide="ignore"):
        out = (p @ vb) / l[:, None]
        lse = m + np.log(l)
    out[empty] = 0.0
    lse[empty] = -np.inf
    return out, lse


def _check_shapes(q, k, v):
    if q.ndim != 4 or k.ndim != 4 or v.ndim != 4:
        raise ValueError("q, k, v must be [B, M, H, K]")
    B, M, H, K = q.shape
    if k.shape[0] != B or v.shape[0] != B or k.shape[1] != v.shape[1]:
        raise ValueError("batch / key length mismatch")
    if k.shape[3] != K:
        raise ValueError("q and k head dims differ")
    if k.shape[2] < 1 or H % k.shape[2] or v.shape[2] != k.shape[2]:
        raise ValueError("k/v must have a number of heads dividing H (grouped-query attention)")
    return B, M, H, K, k.shape[1], v.shape[3]


def attention_head(q, k, v, b, h, scale, mask_kind=MASK_NONE, cu_seqlens_q=None,
                   cu_seqlens_k=None, kv_offset=0, rows=None, bottom_right=False,
                   window_left=None, window_right=None):
    """out [M, Kv] and lse [M] (float64) for one (batch b, head h).

    ``rows`` (optional, dense masks only) restricts the result to those query rows;
    each row is independent of the others in the definition, so this is the same
    arithmetic on fewer rows.  ``bottom_right`` / ``window_left`` / ``window_right``
    select the alignment and local window described in the module docstring.
    """
    B, M, H, K, Mkv, Kv = _check_shapes(q, k, v)
    hk = h // (H // k.shape[2])  # the query head's group
    s64 = _scale64(scale)
    kb_all = np.asarray(k[b, :, hk, :], dtype=np.float64)
    vb_all = np.asarray(v[b, :, hk, :], dtype=np.float64)
    if mask_kind in _BLOCKDIAG_KINDS:
        if B != 1:
            raise ValueError("block-diagonal masks describe packed sequences: B must be 1")
        if rows is not None:
            raise ValueError("row sampling is for dense masks")
        cq = [int(t) for t in cu_seqlens_q]
        ck = [int(t) for t in cu_seqlens_k]
        if len(cq) != len(ck) or cq[0] != 0 or ck[0] != 0 or cq[-1] != M or ck[-1] != Mkv:
            raise ValueError("cu_seqlens must start at 0 and end at M / Mkv")
        out = np.zeros((M, Kv))
        lse = np.full(M, -np.inf)
        qb_all = np.asarray(q[b, :, h, :], dtype=np.float64)
        for s in range(len(cq) - 1):
            qs, qe, ks, ke = cq[s], cq[s + 1], ck[s], ck[s + 1]
            if qe == qs:
                continue
            lo, hi = _band(mask_kind, bottom_right, window_left, window_right, qe - qs, ke - ks)
            o_s, l_s = _block(qb_all[qs:qe], kb_all[ks:ke], vb_all[ks:ke], s64, lo, hi, 0,
                              kv_offset)
            out[qs:qe] = o_s
            lse[qs:qe] = l_s
        return out, lse
    if mask_kind not in (MASK_NONE, MASK_CAUSAL):
        raise ValueError(f"unknown mask kind {mask_kind}")
    lo, hi = _band(mask_kind, bottom_right, window_left, window_right, M, Mkv)
    if rows is None:
        qb = np.asarray(q[b, :, h, :], dtype=np.float64)
        return _block(qb, kb_all, vb_all, s64, lo, hi, 0, kv_offset)
    rows = np.asarray(rows, dtype=np.int64)
    out = np.empty((len(rows), Kv))
    lse = np.empty(len(rows))
    for n, i in enumerate(rows):
        qb = np.asarray(q[b, i:i + 1, h, :], dtype=np.float64)
        o_i, l_i = _block(qb, kb_all, vb_all, s64, lo, hi, int(i), kv_offset)
        out[n] = o_i[0]
        lse[n] = l_i[0]
    return out, lse


def attention(q, k, v, scale, mask_kind=MASK_NONE, cu_seqlens_q=None, cu_seqlens_k=None,
              kv_offset=0, bottom_right=False, window_left=None, window_right=None):
    """Full forward: out [B, M, H, Kv] and lse [B, H, M], float64.

    ``memory_efficient_attention_forward_requires_grad`` returns exactly this pair.
    """
    B, M, H, K, Mkv, Kv = _check_shapes(q, k, v)
    out = np.empty((B, M, H, Kv))
    lse = np.empty((B, H, M))
    for b in range(B):
        for h in range(H):
            o, l = attention_head(q, k, v, b, h, scale, mask_kind, cu_seqlens_q,
                                  cu_seqlens_k, kv_offset, None, bottom_right, window_left,
                                  window_right)
            out[b, :, h, :] = o
            lse[b, h, :] = l
    return out, lse


def lane_rows(s, seqlen_k, seqstart_k=None, block_table=None, page_size=None):
    """K/V row index of every logical key of lane s (padded start or page table)."""
    n = int(seqlen_k[s])
    p = np.arange(n, dtype=np.int64)
    if block_table is not None:
        pages = np.asarray(block_table[s], dtype=np.int64)
        return pages[p // page_size] * page_size + p % page_size
    return int(seqstart_k[s]) + p


def attention_lanes(q, k, v, scale, mask_kind, cu_seqlens_q, seqlen_k, seqstart_k=None,
                    block_table=None, page_size=None, bottom_right=False, window_left=None,
                    window_right=None):
    """Packed queries (B = 1) against per-sequence key lanes, padded or paged.

    q [1, total_q, H, K]; k, v [1, rows, Hk, D] holding the lanes (or the page pool).
    ``mask_kind`` is MASK_BLOCKDIAG or MASK_BLOCKDIAG_CAUSAL.  Returns out
    [1, total_q, H, Kv] and lse [1, H, total_q].
    """
    if mask_kind not in _BLOCKDIAG_KINDS:
        raise ValueError("key lanes take a block-diagonal mask kind")
    if q.shape[0] != 1 or k.shape[0] != 1:
        raise ValueError("key lanes use packed tensors (B = 1)")
    _, M, H, K = q.shape
    Kv = v.shape[3]
    s64 = _scale64(scale)
    cq = [int(t) for t in cu_seqlens_q]
    out = np.zeros((1, M, H, Kv))
    lse = np.full((1, H, M), -np.inf)
    for s in range(len(cq) - 1):
        qs, qe = cq[s], cq[s + 1]
        if qe == qs:
            continue
        rows = lane_rows(s, seqlen_k, seqstart_k, block_table, page_size)
        lo, hi = _band(mask_kind, bottom_right, window_left, window_right, qe - qs, len(rows))
        for h in range(H):
            hk = h // (H // k.shape[2])
            qb = np.asarray(q[0, qs:qe, h, :], dtype=np.float64)
            kb = np.asarray(k[0, rows, hk, :], dtype=np.float64)
            vb = np.asarray(v[0, rows, hk, :], dtype=np.float64)
            o_s, l_s = _block(qb, kb, vb, s64, lo, hi, 0, 0)
            out[0, qs:qe, h] = o_s
            lse[0, h, qs:qe] = l_s
    return out, lse


def attention_partial(q, k_chunk, v_chunk, scale, mask_kind=MASK_NONE, cu_seqlens_q=None,
                      cu_seqlens_k=None, kv_offset=0, window_left=None, window_right=None):
    """Partial attention over one disjoint K/V chunk (same definition, chunk keys only).

    ``kv_offset`` is the position of the chunk's first key in the full key sequence
    (inside each packed sequence, for the block-diagonal masks); masks compare it with the
    query position (top-left alignment: a bottom-right alignment over the full key
    sequence is expressed by folding Lk_full - Lq into kv_offset).
    """
    return attention(q, k_chunk, v_chunk, scale, mask_kind, cu_seqlens_q, cu_seqlens_k,
                     kv_offset, False, window_left, window_right)


def merge_attentions(out_split, lse_split):
    """Exact LSE merge of chunk results.

    out_split: [n, B, M, H, Kv] (or a list of n arrays [B, M, H, Kv]);
    lse_split: [n, B, H, M] (or a list).  Returns out [B, M, H, Kv], lse [B, H, M].
    Zero chunks is an error (``merge_attentions_autograd`` raises on zero partials).
    """
    outs = [np.asarray(o, dtype=np.float64) for o in out_split]
    lses = [np.asarray(s, dtype=np.float64) for s in lse_split]
    if len(outs) == 0 or len(outs) != len(lses):
        raise ValueError("merge needs at least one chunk and one lse per chunk")
    lse_stack = np.stack(lses)                                   # [n, B, H, M]
    m_star = lse_stack.max(axis=0)                               # [B, H, M]
    empty = np.isneginf(m_star)
    shift = np.where(empty, 0.0, m_star)
    w = np.exp(lse_stack - shift[None])                          # [n, B, H, M]
    sum_w = w.sum(axis=0)
    with np.errstate(divide="ignore", invalid="ignore"):
        lse = m_star + np.log(sum_w)
        coef = w / sum_w[None]                                   # exp(lse_c - LSE)
    lse[empty] = -np.inf
    coef[:, empty] = 0.0
    out = np.zeros(outs[0].shape)
    for c, o in enumerate(outs):
        out += np.transpose(coef[c], (0, 2, 1))[..., None] * o   # [B,H,M] -> [B,M,H,1]
    return out, lse



# --------------------------------------------------------------------------------------
# FP8 E4M3 inputs
# --------------------------------------------------------------------------------------
#
# The pages' Blackwell and FlashAttention-3 forward paths take FP8 E4M3 query, key and
# value tensors with tensorwise or per-head scales ("Attention - Core fMHA" backends'
# FP8 E4M3 topics; ``pack_fp8_tensorwise_per_head`` and the ``descale_q/k/v`` arguments of
# the raw flash3 op).  Plainest reading: element x of head h stands for the real number
# decode(x) * descale[h] (one shared value when tensorwise), and the attention is the
# definition above applied to those real numbers.
#
# E4M3 (PyTorch's float8_e4m3fn): bit 7 sign; bits 6..3 exponent, bias 7; bits 2..0
# mantissa.  Exponent field 0: subnormal, mantissa/8 * 2^-6.  Otherwise
# (1 + mantissa/8) * 2^(exponent - 7).  Exponent 15 with mantissa 7 (0x7F, 0xFF) is NaN;
# there are no infinities, so the largest finite magnitude is 1.75 * 2^8 = 448.

def decode_e4m3(codes) -> np.ndarray:
    """float64 values of E4M3 byte codes (any integer array of 0..255)."""
    c = np.asarray(codes).astype(np.int64) & 0xFF
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * 2.0 ** (e - 7))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sign * mag


def dequantize_e4m3(codes, descale) -> np.ndarray:
    """[B, M, Hx, D] E4M3 codes times a per-head descale (scalar or [Hx], float32)."""
    x = decode_e4m3(codes)
    d = np.asarray(descale, dtype=np.float32).astype(np.float64).reshape(-1)
    if d.size == 1:
        return x * d[0]
    if d.size != x.shape[2]:
        raise ValueError(f"descale has {d.size} entries for {x.shape[2]} heads")
    return x * d[None, None, :, None]


def attention_fp8(q8, k8, v8, descale_q, descale_k, descale_v, scale, mask_kind=MASK_NONE,
                  cu_seqlens_q=None, cu_seqlens_k=None, bottom_right=False, window_left=None,
                  window_right=None):
    """Attention forward on E4M3 inputs: the definition on the dequantized values."""
    return attention(dequantize_e4m3(q8, descale_q), dequantize_e4m3(k8, descale_k),
                     dequantize_e4m3(v8, descale_v), scale, mask_kind, cu_seqlens_q,
                     cu_seqlens_k, 0, bottom_right, window_left, window_right)


def attention_lanes_fp8(q8, k8, v8, descale_q, descale_k, descale_v, scale, mask_kind,
                        cu_seqlens_q, seqlen_k, seqstart_k=None, block_table=None,
                        page_size=None, bottom_right=False, window_left=None, window_right=None):
    """Key-lane attention on E4M3 inputs (padded or paged), on the dequantized values."""
    return attention_lanes(dequantize_e4m3(q8, descale_q), dequantize_e4m3(k8, descale_k),
                           dequantize_e4m3(v8, descale_v), scale, mask_kind, cu_seqlens_q,
                           seqlen_k, seqstart_k, block_table, page_size, bottom_right,
                           window_left, window_right)
