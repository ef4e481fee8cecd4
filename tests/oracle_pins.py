"""Pins for the fp64 oracle: checks against things other than the oracle itself.

Every ``pin_*`` function takes the oracle module as its argument and raises
``AssertionError`` on a mismatch, so the same pins run against the real oracle
(tests/test_oracle_pins.py) and against deliberately broken copies of it
(tests/test_oracle_mutants.py, which shows each plausible mistake trips a pin).

Sources of truth, none of them the oracle:
  * a pure-Python brute force (loops, ``math.exp``), with the mask materialised element
    by element from the pages' definitions (MSLK kernel reference, "Attention - Biases &
    masks": ``LowerTriangularMask`` gives zeros on/below the diagonal and -inf above;
    ``BlockDiagonalMask`` lets Q block i see only K/V block i; ``BlockDiagonalCausalMask``
    is top-left causal inside every block);
  * PyTorch's fp64 ``scaled_dot_product_attention`` and ``logsumexp`` (a special case
    that reduces to a library routine);
  * closed forms and invariants that hold for any input;
  * hand-derived cases stored in tests/golden/closed_form_cases.json.
"""

from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "closed_form_cases.json")
NEG_INF = float("-inf")


# --------------------------------------------------------------------------------------
# Pure-Python brute force
# --------------------------------------------------------------------------------------

def _seq_of(pos, cu):
    for s in range(len(cu) - 1):
        if cu[s] <= pos < cu[s + 1]:
            return s
    raise IndexError(pos)


def materialize_bias(kind, M, Mkv, kv_offset=0, cu_q=None, cu_k=None, bottom_right=False,
                     window_left=None, window_right=None):
    """Dense additive bias [M][Mkv] of 0.0 / -inf, one element at a time.

    Alignment and windows follow the mask classes' one-line descriptions: a bottom-right
    mask lines the last query up with the last key of its block (query row i of a block
    of Lq rows is paired with key row i + Lk - Lq); a causal local window of w keys keeps
    the w keys ending at the paired key; a non-causal local window keeps the keys from
    window_left before to window_right after the paired key.
    """
    bias = [[0.0] * Mkv for _ in range(M)]
    for i in range(M):
        for j in range(Mkv):
            if kind in (0, 1):
                qi, kj, Lq, Lk = i, kv_offset + j, M, Mkv
                keep = True
            else:                                           # block-diagonal (+ causal)
                si, sj = _seq_of(i, cu_q), _seq_of(j, cu_k)
                keep = si == sj
                qi, kj = i - cu_q[si], kv_offset + j - cu_k[sj]
                Lq, Lk = cu_q[si + 1] - cu_q[si], cu_k[sj + 1] - cu_k[sj]
            paired = qi + (Lk - Lq if bottom_right else 0)   # the key row query qi lines up with
            if keep and kind in (1, 3):
                keep = kj <= paired
            if keep and window_right is not None:
                keep = kj <= paired + window_right
            if keep and window_left is not None:
                keep = kj >= paired - window_left
            bias[i][j] = 0.0 if keep else NEG_INF
    return bias


def brute_attention(q, k, v, scale, kind=0, cu_q=None, cu_k=None, kv_offset=0,
                    bottom_right=False, window_left=None, window_right=None):
    """Loops over (b, h, i, j, d) with Python floats. Returns out [B][M][H][Kv], lse [B][H][M]."""
    q, k, v = (np.asarray(t, dtype=np.float64).tolist() for t in (q, k, v))
    B, M, H, K = len(q), len(q[0]), len(q[0][0]), len(q[0][0][0])
    Mkv, Hk, Kv = len(k[0]), len(k[0][0]), len(v[0][0][0])
    s = float(np.float32(scale))
    bias = materialize_bias(kind, M, Mkv, kv_offset, cu_q, cu_k, bottom_right, window_left,
                            window_right)
    out = [[[[0.0] * Kv for _ in range(H)] for _ in range(M)] for _ in range(B)]
    lse = [[[NEG_INF] * M for _ in range(H)] for _ in range(B)]
    for b in range(B):
        for h in range(H):
            hk = (h * Hk) // H  # query heads in Hk equal consecutive groups
            for i in range(M):
                x = []
                for j in range(Mkv):
                    dot = math.fsum(q[b][i][h][d] * k[b][j][hk][d] for d in range(K))
                    x.append(s * dot + bias[i][j])
                finite = [xj for xj in x if xj != NEG_INF]
                if not finite:
                    continue
                mx = max(finite)
                e = [math.exp(xj - mx) if xj != NEG_INF else 0.0 for xj in x]
                z = math.fsum(e)
                for d in range(Kv):
                    out[b][i][h][d] = math.fsum(e[j] * v[b][j][hk][d] for j in range(Mkv)) / z
                lse[b][h][i] = mx + math.log(z)
    return np.array(out), np.array(lse)


def brute_merge(outs, lses):
    """Per-element LSE merge with Python floats."""
    n = len(outs)
    outs = [np.asarray(o, dtype=np.float64) for o in outs]
    lses = [np.asarray(l_, dtype=np.float64) for l_ in lses]
    B, M, H, Kv = outs[0].shape
    out = np.zeros((B, M, H, Kv))
    lse = np.full((B, H, M), NEG_INF)
    for b in range(B):
        for h in range(H):
            for i in range(M):
                ls = [float(lses[c][b, h, i]) for c in range(n)]
                fin = [x for x in ls if x != NEG_INF]
                if not fin:
                    continue
                tot = math.log(math.fsum(math.exp(x) for x in fin)) if max(fin) < 700 else None
                if tot is None:
                    mx = max(fin)
                    tot = mx + math.log(math.fsum(math.exp(x - mx) for x in fin))
                lse[b, h, i] = tot
                for d in range(Kv):
                    out[b, i, h, d] = math.fsum(
                        math.exp(ls[c] - tot) * float(outs[c][b, i, h, d])
                        for c in range(n) if ls[c] != NEG_INF)
    return out, lse


# --------------------------------------------------------------------------------------
# helpers
# --------------------------------------------------------------------------------------

def _rand(rng, shape, scale=1.0):
    return rng.standard_normal(shape) * scale


def _bf16_round(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).double().numpy()


def _close(a, b, tol, what):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} vs {b.shape}"
    inf_a, inf_b = np.isneginf(a), np.isneginf(b)
    assert np.array_equal(inf_a, inf_b), f"{what}: -inf pattern differs"
    assert not np.isnan(a).any() and not np.isnan(b).any(), f"{what}: NaN"
    fin = ~inf_a
    if fin.any():
        err = np.max(np.abs(a[fin] - b[fin]))
        assert err <= tol, f"{what}: max |diff| {err:.3e} > {tol:.1e}"


def _tiny_cases():
    """Deterministic tiny shapes covering every mask, kv_offset, shared K/V heads."""
    rng = np.random.default_rng(1234)
    cases = []
    for kind in (0, 1, 2, 3):
        for trial in range(3):
            K = int(rng.integers(1, 9))
            Kv = int(rng.integers(1, 9))
            H = int(rng.integers(1, 3))
            Hk = H if trial != 2 else 1
            if kind >= 2:
                B = 1
                nq = [int(x) for x in rng.integers(0, 6, size=3)]
                nk = [int(x) for x in rng.integers(1, 6, size=3)]
                cu_q = [0]
                cu_k = [0]
                for a, b in zip(nq, nk):
                    cu_q.append(cu_q[-1] + a)
                    cu_k.append(cu_k[-1] + b)
                M, Mkv = cu_q[-1], cu_k[-1]
                if M == 0:
                    nq[0] = 2
                    cu_q = [0, 2, 2 + nq[1], 2 + nq[1] + nq[2]]
                    M = cu_q[-1]
            else:
                B = int(rng.integers(1, 3))
                M = int(rng.integers(1, 18))
                Mkv = int(rng.integers(1, 18))
                cu_q = cu_k = None
            kv_off = int(rng.integers(0, 4)) if kind in (1, 3) and trial == 1 else 0
            q = _bf16_round(_rand(rng, (B, M, H, K)))
            k = _bf16_round(_rand(rng, (B, Mkv, Hk, K)))
            v = _bf16_round(_rand(rng, (B, Mkv, Hk, Kv)))
            scale = float(rng.uniform(0.1, 1.5))
            cases.append((kind, q, k, v, scale, cu_q, cu_k, kv_off))
    return cases


# --------------------------------------------------------------------------------------
# Pins
# --------------------------------------------------------------------------------------

def pin_bruteforce(orc):
    """Oracle == element-by-element brute force on tiny inputs, every mask, to 1e-12."""
    for kind, q, k, v, scale, cu_q, cu_k, kv_off in _tiny_cases():
        o_ref, l_ref = brute_attention(q, k, v, scale, kind, cu_q, cu_k, kv_off)
        o, l_ = orc.attention(q, k, v, scale, kind, cu_q, cu_k, kv_off)
        _close(o, o_ref, 1e-12, f"out kind={kind}")
        _close(l_, l_ref, 1e-12, f"lse kind={kind}")


def pin_torch_sdpa(orc):
    """Oracle == torch fp64 scaled_dot_product_attention (+ logsumexp) with a boolean mask."""
    rng = np.random.default_rng(7)
    for kind, (M, Mkv) in ((0, (40, 57)), (1, (64, 64)), (1, (33, 70))):
        B, H, K, Kv = 2, 3, 32, 24
        q = _bf16_round(_rand(rng, (B, M, H, K)))
        k = _bf16_round(_rand(rng, (B, Mkv, H, K)))
        v = _bf16_round(_rand(rng, (B, Mkv, H, Kv)))
        scale = 0.3
        s64 = float(np.float32(scale))
        tq, tk, tv = (torch.from_numpy(t).permute(0, 2, 1, 3) for t in (q, k, v))
        if kind == 1:
            allow = torch.ones(M, Mkv, dtype=torch.bool).tril()
        else:
            allow = torch.ones(M, Mkv, dtype=torch.bool)
        ref = torch.nn.functional.scaled_dot_product_attention(
            tq, tk, tv, attn_mask=allow, scale=s64)
        scores = (tq @ tk.transpose(-1, -2)) * s64
        scores = scores.masked_fill(~allow, float("-inf"))
        ref_lse = torch.logsumexp(scores, dim=-1)
        o, l_ = orc.attention(q, k, v, scale, kind)
        _close(o, ref.permute(0, 2, 1, 3).numpy(), 1e-12, "sdpa out")
        _close(l_, ref_lse.numpy(), 1e-12, "sdpa lse")


def pin_single_key(orc):
    """Mkv = 1: out = v0 and lse = scale * q.k0 for every row."""
    rng = np.random.default_rng(3)
    q = _bf16_round(_rand(rng, (2, 5, 2, 8)))
    k = _bf16_round(_rand(rng, (2, 1, 2, 8)))
    v = _bf16_round(_rand(rng, (2, 1, 2, 6)))
    o, l_ = orc.attention(q, k, v, 0.7)
    s = float(np.float32(0.7))
    for b in range(2):
        for h in range(2):
            for i in range(5):
                _close(o[b, i, h], v[b, 0, h], 1e-14, "single key out")
                expect = s * math.fsum(q[b, i, h, d] * k[b, 0, h, d] for d in range(8))
                _close(l_[b, h, i], expect, 1e-12, "single key lse")


def pin_constant_v(orc):
    """Every value row equal to c: out = c whatever the scores (any mask, non-empty rows)."""
    rng = np.random.default_rng(4)
    q = _bf16_round(_rand(rng, (1, 9, 2, 16)))
    k = _bf16_round(_rand(rng, (1, 12, 2, 16)))
    c = np.array([0.5, -2.0, 3.25, 1.0])
    v = np.broadcast_to(c, (1, 12, 2, 4)).copy()
    for kind in (0, 1):
        o, _ = orc.attention(q, k, v, 0.9, kind)
        _close(o, np.broadcast_to(c, o.shape), 1e-13, "constant v")


def pin_causal_row0(orc):
    """Top-left causal, row 0 sees only key 0: out = v0, lse = scale * q0.k0."""
    rng = np.random.default_rng(5)
    q = _bf16_round(_rand(rng, (1, 6, 1, 8)))
    k = _bf16_round(_rand(rng, (1, 9, 1, 8)))
    v = _bf16_round(_rand(rng, (1, 9, 1, 5)))
    o, l_ = orc.attention(q, k, v, 0.4, 1)
    _close(o[0, 0, 0], v[0, 0, 0], 1e-14, "causal row0 out")
    s = float(np.float32(0.4))
    _close(l_[0, 0, 0], s * math.fsum(q[0, 0, 0] * k[0, 0, 0]), 1e-13, "causal row0 lse")
    # row 1 sees exactly keys 0 and 1 (two-term softmax written out)
    x0 = s * math.fsum(q[0, 1, 0] * k[0, 0, 0])
    x1 = s * math.fsum(q[0, 1, 0] * k[0, 1, 0])
    w1 = 1.0 / (1.0 + math.exp(x0 - x1))
    _close(o[0, 1, 0], (1 - w1) * v[0, 0, 0] + w1 * v[0, 1, 0], 1e-13, "causal row1 out")


def pin_zero_query(orc):
    """q = 0: uniform weights over the allowed set; out = mean of v there, lse = ln|A_i|."""
    rng = np.random.default_rng(6)
    M, Mkv = 7, 10
    q = np.zeros((1, M, 1, 8))
    k = _bf16_round(_rand(rng, (1, Mkv, 1, 8)))
    v = _bf16_round(_rand(rng, (1, Mkv, 1, 3)))
    for kind, kv_off in ((0, 0), (1, 0), (1, 2)):
        o, l_ = orc.attention(q, k, v, 1.0, kind, kv_offset=kv_off)
        for i in range(M):
            n = Mkv if kind == 0 else max(0, min(Mkv, i - kv_off + 1))
            if n == 0:
                assert l_[0, 0, i] == NEG_INF and np.all(o[0, i, 0] == 0.0), "empty row"
                continue
            _close(o[0, i, 0], v[0, :n, 0].mean(axis=0), 1e-14, "zero q out")
            _close(l_[0, 0, i], math.log(n), 1e-14, "zero q lse")


def pin_duplicate_keys(orc):
    """Concatenating K and V with themselves (no mask): out unchanged, lse + ln 2."""
    rng = np.random.default_rng(8)
    q = _bf16_round(_rand(rng, (2, 6, 2, 8)))
    k = _bf16_round(_rand(rng, (2, 11, 2, 8)))
    v = _bf16_round(_rand(rng, (2, 11, 2, 7)))
    o1, l1 = orc.attention(q, k, v, 0.6)
    o2, l2 = orc.attention(q, np.concatenate([k, k], 1), np.concatenate([v, v], 1), 0.6)
    _close(o2, o1, 1e-13, "dup out")
    _close(l2, l1 + math.log(2.0), 1e-13, "dup lse")


def pin_permute_keys(orc):
    """Permuting the keys (and values alike) changes nothing when there is no mask."""
    rng = np.random.default_rng(9)
    q = _bf16_round(_rand(rng, (1, 8, 2, 8)))
    k = _bf16_round(_rand(rng, (1, 13, 2, 8)))
    v = _bf16_round(_rand(rng, (1, 13, 2, 4)))
    perm = rng.permutation(13)
    o1, l1 = orc.attention(q, k, v, 0.5)
    o2, l2 = orc.attention(q, k[:, perm], v[:, perm], 0.5)
    _close(o2, o1, 1e-13, "perm out")
    _close(l2, l1, 1e-13, "perm lse")


def pin_scale_folds_into_q(orc):
    """attention(q, 2s) == attention(2q, s): the scale multiplies the scores."""
    rng = np.random.default_rng(10)
    q = _bf16_round(_rand(rng, (1, 5, 1, 8)))
    k = _bf16_round(_rand(rng, (1, 7, 1, 8)))
    v = _bf16_round(_rand(rng, (1, 7, 1, 3)))
    o1, l1 = orc.attention(q, k, v, 0.5)
    o2, l2 = orc.attention(2 * q, k, v, 0.25)
    _close(o2, o1, 1e-13, "scale out")
    _close(l2, l1, 1e-13, "scale lse")


def pin_grouped_query_heads(orc):
    """Grouped-query attention: query heads g*r .. g*r + r - 1 share K/V head g.  Checked
    against the brute force and against explicitly repeating each K/V head r times."""
    rng = np.random.default_rng(71)
    for (B, M, Mkv, H, Hk, kind) in ((1, 4, 5, 4, 2, 0), (2, 3, 6, 6, 3, 1), (1, 5, 5, 6, 2, 1)):
        q = _rand(rng, (B, M, H, 8))
        k = _rand(rng, (B, Mkv, Hk, 8))
        v = _rand(rng, (B, Mkv, Hk, 8))
        ro, rl = brute_attention(q, k, v, 0.4, kind)
        o, l_ = orc.attention(q, k, v, 0.4, kind)
        _close(o, ro, 1e-12, f"gqa out {H}/{Hk}")
        _close(l_, rl, 1e-12, f"gqa lse {H}/{Hk}")
        r = H // Hk
        ke, ve = np.repeat(k, r, axis=2), np.repeat(v, r, axis=2)  # head g*r + i <- group g
        oe, le = orc.attention(q, ke, ve, 0.4, kind)
        _close(o, oe, 1e-12, "gqa = repeated heads (out)")
        _close(l_, le, 1e-12, "gqa = repeated heads (lse)")


def pin_shared_kv_head(orc):
    """One K/V head shared by all query heads == that head copied to every query head."""
    rng = np.random.default_rng(11)
    q = _bf16_round(_rand(rng, (1, 6, 3, 8)))
    k1 = _bf16_round(_rand(rng, (1, 9, 1, 8)))
    v1 = _bf16_round(_rand(rng, (1, 9, 1, 5)))
    o1, l1 = orc.attention(q, k1, v1, 0.5, 1)
    o2, l2 = orc.attention(q, np.repeat(k1, 3, 2), np.repeat(v1, 3, 2), 0.5, 1)
    _close(o1, o2, 0.0, "shared head out")
    _close(l1, l2, 0.0, "shared head lse")
    # and each head matches brute force with its own query
    ob, lb = brute_attention(q, k1, v1, 0.5, 1)
    _close(o1, ob, 1e-12, "shared head brute out")
    _close(l1, lb, 1e-12, "shared head brute lse")


def _split_and_merge(orc, q, k, v, scale, kind, bounds, cu_q=None, cu_k_chunks=None):
    outs, lses = [], []
    for c, (s0, s1) in enumerate(bounds):
        cu_k = None if cu_k_chunks is None else cu_k_chunks[c]
        o, l_ = orc.attention_partial(q, k[:, s0:s1], v[:, s0:s1], scale, kind, cu_q, cu_k,
                                      kv_offset=s0 if kind == 1 else 0)
        outs.append(o)
        lses.append(l_)
    return orc.merge_attentions(outs, lses)


def pin_merge_any_chunking(orc):
    """Merge of partials over any disjoint chunking == full attention (no mask and causal)."""
    rng = np.random.default_rng(12)
    q = _bf16_round(_rand(rng, (2, 9, 2, 8)))
    k = _bf16_round(_rand(rng, (2, 16, 2, 8)))
    v = _bf16_round(_rand(rng, (2, 16, 2, 6)))
    for kind in (0, 1):
        o_full, l_full = orc.attention(q, k, v, 0.5, kind)
        for bounds in ([(0, 8), (8, 16)], [(0, 3), (3, 4), (4, 11), (11, 16)],
                       [(j, j + 1) for j in range(16)], [(0, 16)]):
            o, l_ = _split_and_merge(orc, q, k, v, 0.5, kind, bounds)
            _close(o, o_full, 1e-13, f"merge out kind={kind} n={len(bounds)}")
            _close(l_, l_full, 1e-13, f"merge lse kind={kind} n={len(bounds)}")


def pin_merge_against_brute(orc):
    """Oracle merge == per-element brute-force merge on random chunk results, incl. -inf."""
    rng = np.random.default_rng(13)
    n, B, M, H, Kv = 3, 2, 5, 2, 4
    outs = [_rand(rng, (B, M, H, Kv)) for _ in range(n)]
    lses = [_rand(rng, (B, H, M), 3.0) for _ in range(n)]
    lses[1][0, 1, 2] = NEG_INF
    lses[0][1, 0, 4] = lses[1][1, 0, 4] = lses[2][1, 0, 4] = NEG_INF
    o, l_ = orc.merge_attentions(np.stack(outs), np.stack(lses))
    ob, lb = brute_merge(outs, lses)
    _close(o, ob, 1e-13, "merge brute out")
    _close(l_, lb, 1e-13, "merge brute lse")


def pin_merge_identities(orc):
    """Single chunk is the identity; chunk order is irrelevant; a -inf chunk has no effect."""
    rng = np.random.default_rng(14)
    B, M, H, Kv = 1, 6, 2, 5
    outs = [_rand(rng, (B, M, H, Kv)) for _ in range(4)]
    lses = [_rand(rng, (B, H, M)) for _ in range(4)]
    o, l_ = orc.merge_attentions(outs[:1], lses[:1])
    _close(o, outs[0], 1e-15, "identity out")
    _close(l_, lses[0], 1e-15, "identity lse")
    o1, l1 = orc.merge_attentions(outs, lses)
    perm = [2, 0, 3, 1]
    o2, l2 = orc.merge_attentions([outs[i] for i in perm], [lses[i] for i in perm])
    _close(o1, o2, 1e-14, "perm out")
    _close(l1, l2, 1e-14, "perm lse")
    junk = _rand(rng, (B, M, H, Kv)) * 1e3
    o3, l3 = orc.merge_attentions(outs + [junk], lses + [np.full((B, H, M), NEG_INF)])
    _close(o3, o1, 1e-14, "-inf chunk out")
    _close(l3, l1, 1e-14, "-inf chunk lse")
    try:
        orc.merge_attentions([], [])
    except ValueError:
        pass
    else:
        raise AssertionError("zero chunks must be rejected")


def pin_varlen_equals_per_sequence(orc):
    """Packed block-diagonal (causal) attention == each sequence attended on its own."""
    rng = np.random.default_rng(15)
    lq, lk = [3, 5, 1, 4], [4, 5, 2, 6]
    cu_q = [0, 3, 8, 9, 13]
    cu_k = [0, 4, 9, 11, 17]
    q = _bf16_round(_rand(rng, (1, 13, 2, 8)))
    k = _bf16_round(_rand(rng, (1, 17, 2, 8)))
    v = _bf16_round(_rand(rng, (1, 17, 2, 6)))
    for kind, dense in ((2, 0), (3, 1)):
        o, l_ = orc.attention(q, k, v, 0.5, kind, cu_q, cu_k)
        for s in range(4):
            qs, ks = cu_q[s], cu_k[s]
            o_s, l_s = orc.attention(q[:, qs:qs + lq[s]], k[:, ks:ks + lk[s]],
                                     v[:, ks:ks + lk[s]], 0.5, dense)
            _close(o[:, qs:qs + lq[s]], o_s, 1e-14, f"varlen out kind={kind}")
            _close(l_[:, :, qs:qs + lq[s]], l_s, 1e-14, f"varlen lse kind={kind}")


def pin_varlen_partial_offset(orc):
    """Block-diagonal causal partials over per-sequence key chunks, merged == full."""
    rng = np.random.default_rng(16)
    lens = [6, 3, 7]
    cu = [0, 6, 9, 16]
    q = _bf16_round(_rand(rng, (1, 16, 1, 8)))
    k = _bf16_round(_rand(rng, (1, 16, 1, 8)))
    v = _bf16_round(_rand(rng, (1, 16, 1, 4)))
    o_full, l_full = orc.attention(q, k, v, 0.5, 3, cu, cu)
    # chunk c takes keys [c*2, c*2+2) of every sequence (shorter sequences run out)
    outs, lses = [], []
    for c in range(4):
        idx, cu_kc = [], [0]
        for s, L in enumerate(lens):
            sel = [cu[s] + j for j in range(2 * c, min(L, 2 * c + 2))]
            idx += sel
            cu_kc.append(cu_kc[-1] + len(sel))
        o, l_ = orc.attention_partial(q, k[:, idx], v[:, idx], 0.5, 3, cu, cu_kc,
                                      kv_offset=2 * c)
        outs.append(o)
        lses.append(l_)
    o, l_ = orc.merge_attentions(outs, lses)
    _close(o, o_full, 1e-13, "varlen partial out")
    _close(l_, l_full, 1e-13, "varlen partial lse")


def pin_empty_rows(orc):
    """Rows with no allowed key give out = 0 and lse = -inf (causal chunk past the row)."""
    rng = np.random.default_rng(17)
    q = _bf16_round(_rand(rng, (1, 4, 1, 8)))
    k = _bf16_round(_rand(rng, (1, 3, 1, 8)))
    v = _bf16_round(_rand(rng, (1, 3, 1, 4)))
    o, l_ = orc.attention_partial(q, k, v, 0.5, 1, kv_offset=2)
    assert np.all(o[0, :2] == 0.0) and np.all(np.isneginf(l_[0, 0, :2])), "empty rows"
    assert np.all(np.isfinite(l_[0, 0, 2:])), "rows 2, 3 have keys"


def _ev(x, env):
    """Evaluate a nested list whose leaves are numbers or closed-form expressions."""
    if isinstance(x, list):
        return [_ev(e, env) for e in x]
    if isinstance(x, str):
        return float(eval(x, {"__builtins__": {}}, env))
    return float(x)


def pin_golden_cases(orc):
    """Hand-derived closed-form cases (tests/golden/closed_form_cases.json)."""
    with open(GOLDEN) as f:
        spec = json.load(f)
    env = {"log": math.log, "inf": float("inf")}
    for case in spec["attention"]:
        q, k, v = (np.array(_ev(case[n], env)) for n in ("q", "k", "v"))
        o, l_ = orc.attention(q, k, v, case["scale"], case["mask_kind"])
        _close(o, np.array(_ev(case["out"], env)), 1e-12, case["name"] + " out")
        _close(l_, np.array(_ev(case["lse"], env)), 1e-12, case["name"] + " lse")
    for case in spec["merge"]:
        outs = np.array(_ev(case["out_split"], env))
        lses = np.array(_ev(case["lse_split"], env))
        o, l_ = orc.merge_attentions(outs, lses)
        _close(o, np.array(_ev(case["out"], env)), 1e-12, case["name"] + " out")
        _close(l_, np.array(_ev(case["lse"], env)), 1e-12, case["name"] + " lse")


def pin_widen_bf16(orc):
    """Bit widening of bf16 == PyTorch's bf16 -> fp64 conversion for every non-NaN pattern."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    got = orc.widen_bf16_bits(bits)
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok]), "bf16 widening"
    assert np.array_equal(np.isnan(got), np.isnan(ref)), "bf16 NaN patterns"


# --------------------------------------------------------------------------------------
# alignment and local windows
# --------------------------------------------------------------------------------------

def pin_window_single_key(orc):
    """A window of one key (causal window_left = 0, or non-causal 0/0) leaves query i the
    single paired key i + shift: out_i = v[paired], lse_i = scale * q_i . k[paired]; a
    query whose paired key falls outside the keys has an empty row."""
    rng = np.random.default_rng(41)
    for M, Mkv in ((5, 9), (7, 4), (6, 6)):
        q = _bf16_round(_rand(rng, (1, M, 2, 8)))
        k = _bf16_round(_rand(rng, (1, Mkv, 2, 8)))
        v = _bf16_round(_rand(rng, (1, Mkv, 2, 8)))
        s = 0.3
        for br in (False, True):
            shift = (Mkv - M) if br else 0
            want_o = np.zeros((1, M, 2, 8))
            want_l = np.full((1, 2, M), NEG_INF)
            for i in range(M):
                j = i + shift
                if 0 <= j < Mkv:
                    want_o[0, i] = v[0, j]
                    for h in range(2):
                        want_l[0, h, i] = float(np.float32(s)) * float(np.dot(q[0, i, h], k[0, j, h]))
            for kind, wr in ((orc.MASK_CAUSAL, None), (orc.MASK_NONE, 0)):
                o, l_ = orc.attention(q, k, v, s, kind, bottom_right=br, window_left=0,
                                      window_right=wr)
                _close(o, want_o, 1e-12, f"single-key window out M{M} Mkv{Mkv} br{br} kind{kind}")
                _close(l_, want_l, 1e-12, f"single-key window lse M{M} Mkv{Mkv} br{br} kind{kind}")


def pin_bottom_right_reductions(orc):
    """Bottom-right causal equals top-left causal when M = Mkv, and with one query it keeps
    every key (PyTorch's unmasked SDPA); a causal window wider than the keys changes
    nothing; a non-causal window wider on both sides is no mask."""
    rng = np.random.default_rng(42)
    q = _bf16_round(_rand(rng, (2, 6, 2, 16)))
    k = _bf16_round(_rand(rng, (2, 6, 2, 16)))
    v = _bf16_round(_rand(rng, (2, 6, 2, 16)))
    a = orc.attention(q, k, v, 0.25, orc.MASK_CAUSAL, bottom_right=True)
    b = orc.attention(q, k, v, 0.25, orc.MASK_CAUSAL)
    _close(a[0], b[0], 0.0, "br == tl causal at M = Mkv (out)")
    _close(a[1], b[1], 0.0, "br == tl causal at M = Mkv (lse)")
    q1 = q[:, :1]
    k9 = _bf16_round(_rand(rng, (2, 9, 2, 16)))
    v9 = _bf16_round(_rand(rng, (2, 9, 2, 16)))
    o, l_ = orc.attention(q1, k9, v9, 0.25, orc.MASK_CAUSAL, bottom_right=True)
    tq, tk, tv = (torch.from_numpy(np.ascontiguousarray(t.transpose(0, 2, 1, 3))) for t in (q1, k9, v9))
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, scale=float(np.float32(0.25)))
    _close(o, ref.transpose(1, 2).numpy(), 1e-12, "br causal, one query = no mask")
    x = torch.einsum("bhik,bhjk->bhij", tq, tk) * float(np.float32(0.25))
    _close(l_, torch.logsumexp(x, dim=-1).numpy(), 1e-12, "br causal, one query lse")
    wide = orc.attention(q, k9, v9, 0.25, orc.MASK_CAUSAL, window_left=20)
    base = orc.attention(q, k9, v9, 0.25, orc.MASK_CAUSAL)
    _close(wide[0], base[0], 0.0, "wide causal window (out)")
    both = orc.attention(q, k9, v9, 0.25, orc.MASK_NONE, bottom_right=True, window_left=20,
                         window_right=20)
    none = orc.attention(q, k9, v9, 0.25, orc.MASK_NONE)
    _close(both[0], none[0], 0.0, "wide local window = no mask (out)")
    _close(both[1], none[1], 0.0, "wide local window = no mask (lse)")


def pin_band_bruteforce(orc):
    """Windows and bottom-right alignment against the element-by-element brute force,
    dense and block-diagonal (blocks of unequal query and key lengths)."""
    rng = np.random.default_rng(43)
    q = _bf16_round(_rand(rng, (1, 7, 2, 8)))
    k = _bf16_round(_rand(rng, (1, 10, 2, 8)))
    v = _bf16_round(_rand(rng, (1, 10, 2, 8)))
    dense = [(1, True, None, None), (1, False, 2, None), (1, True, 3, None),
             (0, True, 2, 1), (0, False, 0, 3), (0, True, 4, 0)]
    for kind, br, wl, wr in dense:
        o, l_ = orc.attention(q, k, v, 0.5, kind, bottom_right=br, window_left=wl,
                              window_right=wr)
        bo, bl = brute_attention(q, k, v, 0.5, kind, bottom_right=br, window_left=wl,
                                 window_right=wr)
        _close(o, bo, 1e-12, f"band out kind{kind} br{br} wl{wl} wr{wr}")
        _close(l_, bl, 1e-12, f"band lse kind{kind} br{br} wl{wl} wr{wr}")
    cu_q, cu_k = [0, 3, 7], [0, 6, 10]
    for kind, br, wl in ((3, True, None), (3, False, 1), (3, True, 2), (2, True, None)):
        kw = {} if kind == 3 else {"window_left": 1, "window_right": 1}
        if kind == 3:
            kw = {"window_left": wl}
        o, l_ = orc.attention(q, k, v, 0.5, kind, cu_q, cu_k, bottom_right=br, **kw)
        bo, bl = brute_attention(q, k, v, 0.5, kind, cu_q, cu_k, bottom_right=br, **kw)
        _close(o, bo, 1e-12, f"blockdiag band out kind{kind} br{br} {kw}")
        _close(l_, bl, 1e-12, f"blockdiag band lse kind{kind} br{br} {kw}")


def pin_window_split_merge(orc):
    """A windowed causal forward equals the merge of windowed partials over any chunking
    (each chunk's kv_offset carries its key positions)."""
    rng = np.random.default_rng(44)
    q = _bf16_round(_rand(rng, (1, 9, 2, 8)))
    k = _bf16_round(_rand(rng, (1, 9, 2, 8)))
    v = _bf16_round(_rand(rng, (1, 9, 2, 8)))
    full = orc.attention(q, k, v, 0.4, orc.MASK_CAUSAL, window_left=3)
    for bounds in (((0, 4), (4, 9)), ((0, 2), (2, 5), (5, 9))):
        parts = [orc.attention_partial(q, k[:, a:b], v[:, a:b], 0.4, orc.MASK_CAUSAL,
                                       kv_offset=a, window_left=3) for a, b in bounds]
        o, l_ = orc.merge_attentions([p[0] for p in parts], [p[1] for p in parts])
        _close(o, full[0], 1e-12, f"windowed split {bounds} (out)")
        _close(l_, full[1], 1e-12, f"windowed split {bounds} (lse)")


def pin_rows_sampling(orc):
    """attention_head(rows=R) returns, for each sampled row, what the element-by-element
    brute force gives for that row: causal with a key offset, bottom-right alignment and
    left windows, rows unsorted and repeated, first and last rows included.  Each row's
    position must follow its own index (a row treated as row 0 sees only key 0 under a
    causal mask)."""
    rng = np.random.default_rng(45)
    B, M, Mkv, H, Hk, K, Kv = 2, 13, 16, 2, 1, 8, 6
    q = _bf16_round(_rand(rng, (B, M, H, K)))
    k = _bf16_round(_rand(rng, (B, Mkv, Hk, K)))
    v = _bf16_round(_rand(rng, (B, Mkv, Hk, Kv)))
    rows = [12, 0, 7, 3, 12, 1, 8]
    cases = [(orc.MASK_CAUSAL, 0, False, None, None), (orc.MASK_CAUSAL, 3, False, None, None),
             (orc.MASK_CAUSAL, 0, True, None, None), (orc.MASK_CAUSAL, 2, False, 4, None),
             (orc.MASK_CAUSAL, 0, True, 2, None), (orc.MASK_NONE, 0, True, 3, 1),
             (orc.MASK_NONE, 0, False, None, None)]
    for kind, off, br, wl, wr in cases:
        bo, bl = brute_attention(q, k, v, 0.7, kind, kv_offset=off, bottom_right=br,
                                 window_left=wl, window_right=wr)
        for b in range(B):
            for h in range(H):
                o, l_ = orc.attention_head(q, k, v, b, h, 0.7, kind, kv_offset=off, rows=rows,
                                           bottom_right=br, window_left=wl, window_right=wr)
                what = f"rows kind{kind} off{off} br{br} wl{wl} wr{wr} b{b} h{h}"
                _close(o, bo[b][rows, h, :], 1e-12, what + " (out)")
                _close(l_, bl[b, h, rows], 1e-12, what + " (lse)")


# --------------------------------------------------------------------------------------
# padded and paged key lanes
# --------------------------------------------------------------------------------------

def _lane_case(rng):
    lq, lk = [3, 1, 5, 2], [7, 9, 4, 11]
    pad = 12
    H, D = 2, 8
    q = _bf16_round(_rand(rng, (1, sum(lq), H, D)))
    k = np.zeros((1, pad * len(lk), H, D))
    v = np.zeros((1, pad * len(lk), H, D))
    for s, n in enumerate(lk):
        k[0, s * pad:s * pad + n] = _bf16_round(_rand(rng, (n, H, D)))
        v[0, s * pad:s * pad + n] = _bf16_round(_rand(rng, (n, H, D)))
    return lq, lk, pad, q, k, v


def pin_lanes_contiguous_equal_blockdiag(orc):
    """Lanes packed back to back (seqstart = previous ends) are the block-diagonal masks
    with cu_seqlens_k; bottom-right and windows included."""
    rng = np.random.default_rng(51)
    lq, lk, pad, q, k, v = _lane_case(rng)
    cu_q = [0] + list(np.cumsum(lq))
    cu_k = [0] + list(np.cumsum(lk))
    kc = np.concatenate([k[:, s * pad:s * pad + n] for s, n in enumerate(lk)], axis=1)
    vc = np.concatenate([v[:, s * pad:s * pad + n] for s, n in enumerate(lk)], axis=1)
    for kind, br, wl in ((orc.MASK_BLOCKDIAG, False, None), (orc.MASK_BLOCKDIAG_CAUSAL, True, None),
                         (orc.MASK_BLOCKDIAG_CAUSAL, False, 2), (orc.MASK_BLOCKDIAG_CAUSAL, True, 1)):
        a = orc.attention_lanes(q, kc, vc, 0.5, kind, cu_q, lk, seqstart_k=cu_k[:-1],
                                bottom_right=br, window_left=wl)
        b = orc.attention(q, kc, vc, 0.5, kind, cu_q, cu_k, bottom_right=br, window_left=wl)
        _close(a[0], b[0], 0.0, f"contiguous lanes = blockdiag out kind{kind} br{br} wl{wl}")
        _close(a[1], b[1], 0.0, f"contiguous lanes = blockdiag lse kind{kind} br{br} wl{wl}")


def pin_lanes_padding_unread(orc):
    """Rows past a lane's valid keys never reach the result (NaN there changes nothing)."""
    rng = np.random.default_rng(52)
    lq, lk, pad, q, k, v = _lane_case(rng)
    cu_q = [0] + list(np.cumsum(lq))
    starts = [s * pad for s in range(len(lk))]
    kn, vn = k.copy(), v.copy()
    for s, n in enumerate(lk):
        kn[0, s * pad + n:(s + 1) * pad] = np.nan
        vn[0, s * pad + n:(s + 1) * pad] = np.nan
    a = orc.attention_lanes(q, k, v, 0.5, orc.MASK_BLOCKDIAG_CAUSAL, cu_q, lk, seqstart_k=starts,
                            bottom_right=True)
    b = orc.attention_lanes(q, kn, vn, 0.5, orc.MASK_BLOCKDIAG_CAUSAL, cu_q, lk, seqstart_k=starts,
                            bottom_right=True)
    _close(a[0], b[0], 0.0, "padding unread (out)")
    _close(a[1], b[1], 0.0, "padding unread (lse)")


def pin_paged_equals_padded(orc):
    """Scattering every lane's logical pages to a random permutation of physical pages
    (and recording it in a block table) leaves the result unchanged."""
    rng = np.random.default_rng(53)
    lq, lk, pad, q, k, v = _lane_case(rng)
    cu_q = [0] + list(np.cumsum(lq))
    starts = [s * pad for s in range(len(lk))]
    ps = 4
    pages_per_lane = (pad + ps - 1) // ps
    n_pages = pages_per_lane * len(lk) + 3
    perm = rng.permutation(n_pages)
    table = perm[:pages_per_lane * len(lk)].reshape(len(lk), pages_per_lane)
    kp = np.full((1, n_pages * ps, 2, 8), np.nan)
    vp = np.full((1, n_pages * ps, 2, 8), np.nan)
    for s, n in enumerate(lk):
        for p in range(n):
            row = table[s][p // ps] * ps + p % ps
            kp[0, row] = k[0, starts[s] + p]
            vp[0, row] = v[0, starts[s] + p]
    for kind, br, wl in ((orc.MASK_BLOCKDIAG, False, None), (orc.MASK_BLOCKDIAG_CAUSAL, True, 2)):
        a = orc.attention_lanes(q, k, v, 0.5, kind, cu_q, lk, seqstart_k=starts, bottom_right=br,
                                window_left=wl)
        b = orc.attention_lanes(q, kp, vp, 0.5, kind, cu_q, lk, block_table=table, page_size=ps,
                                bottom_right=br, window_left=wl)
        _close(a[0], b[0], 0.0, f"paged = padded out kind{kind}")
        _close(a[1], b[1], 0.0, f"paged = padded lse kind{kind}")


# --------------------------------------------------------------------------------------
# FP8 E4M3 inputs
# --------------------------------------------------------------------------------------

def _torch_e4m3_table():
    """PyTorch's own float8_e4m3fn widening of every byte code (a library routine)."""
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()


def pin_e4m3_table(orc):
    """Every one of the 256 codes decodes as PyTorch's float8_e4m3fn does (NaN where it has NaN)."""
    ref = _torch_e4m3_table()
    got = np.asarray(orc.decode_e4m3(np.arange(256)), dtype=np.float64)
    assert np.array_equal(np.isnan(ref), np.isnan(got)), "NaN codes differ"
    fin = ~np.isnan(ref)
    assert np.array_equal(ref[fin], got[fin]), "decoded values differ"
    assert np.array_equal(np.signbit(ref[fin]), np.signbit(got[fin])), "signs of zero differ"


def pin_e4m3_known_values(orc):
    """Values fixed by the format's definition (sign, exponent bias 7, 3-bit mantissa,
    subnormals m/8 * 2^-6, 0x7F/0xFF NaN, largest finite 448), and ordering."""
    cases = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x0F: 1.875 * 2.0 ** -6,
             0x38: 1.0, 0x39: 1.125, 0x3C: 1.5, 0x40: 2.0, 0x77: 240.0, 0x7E: 448.0,
             0x81: -(2.0 ** -9), 0xB8: -1.0, 0xFE: -448.0}
    got = orc.decode_e4m3(np.array(list(cases)))
    for (code, want), g in zip(cases.items(), got):
        assert g == want, f"code {code:#04x}: {g} != {want}"
    assert np.isnan(orc.decode_e4m3(np.array([0x7F, 0xFF]))).all(), "0x7F/0xFF must be NaN"
    pos = orc.decode_e4m3(np.arange(0x7F))
    assert np.all(np.diff(pos) > 0), "positive codes must increase"


def _fp8_case(rng, B, M, Mkv, H, Hk, D):
    # finite codes only (NaN codes excluded), the whole range otherwise
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)])
    q8 = rng.choice(codes, size=(B, M, H, D))
    k8 = rng.choice(codes, size=(B, Mkv, Hk, D))
    v8 = rng.choice(codes, size=(B, Mkv, Hk, D))
    dq = np.float32(rng.uniform(0.001, 0.01, H))
    dk = np.float32(rng.uniform(0.001, 0.01, Hk))
    dv = np.float32(rng.uniform(0.001, 0.01, Hk))
    return q8, k8, v8, dq, dk, dv


def pin_fp8_bruteforce(orc):
    """Per-head descales, element by element through PyTorch's E4M3 table, then the brute force."""
    table = _torch_e4m3_table()
    rng = np.random.default_rng(61)
    for (B, M, Mkv, H, Hk, D, kind) in ((1, 3, 4, 2, 2, 4, 0), (2, 4, 5, 3, 1, 4, 1), (1, 3, 3, 2, 2, 8, 1)):
        q8, k8, v8, dq, dk, dv = _fp8_case(rng, B, M, Mkv, H, Hk, D)

        def deq(codes, d):
            out = np.zeros(codes.shape)
            for idx in np.ndindex(codes.shape):
                out[idx] = table[codes[idx]] * float(d[idx[2]])
            return out

        ro, rl = brute_attention(deq(q8, dq), deq(k8, dk), deq(v8, dv), 0.3, kind)
        o, l_ = orc.attention_fp8(q8, k8, v8, dq, dk, dv, 0.3, kind)
        _close(o, ro, 1e-12, f"fp8 brute out {B, M, Mkv, H, Hk, D, kind}")
        _close(l_, rl, 1e-12, f"fp8 brute lse {B, M, Mkv, H, Hk, D, kind}")


def pin_fp8_descale_folding(orc):
    """The value descale scales the output; the query and key descales multiply the scale."""
    rng = np.random.default_rng(62)
    q8, k8, v8, _, _, _ = _fp8_case(rng, 1, 5, 7, 2, 2, 8)
    one = np.ones(2, dtype=np.float32)
    a, b, c = np.float32(0.003), np.float32(0.004), np.float32(0.37)
    base_o, base_l = orc.attention_fp8(q8, k8, v8, one, one, one, 0.5 * float(a) * float(b))
    o, l_ = orc.attention_fp8(q8, k8, v8, np.full(2, a), np.full(2, b), np.full(2, c), 0.5)
    # (the folded scale is rounded to float32 once more: relative differences ~1e-7)
    _close(o, float(c) * base_o, 1e-5 * np.abs(base_o).max(), "descale_v scales out")
    _close(l_, base_l, 1e-5 * max(1.0, np.abs(base_l).max()), "descale_q * descale_k fold into the scale")
    # tensorwise (one value) equals the same value per head
    o2, l2 = orc.attention_fp8(q8, k8, v8, a, b, c, 0.5)
    _close(o2, o, 0.0, "tensorwise out")
    _close(l2, l_, 0.0, "tensorwise lse")


def pin_fp8_lanes(orc):
    """FP8 key lanes laid out contiguously equal the FP8 block-diagonal forward."""
    rng = np.random.default_rng(63)
    lq, lk = [2, 3], [3, 4]
    q8, k8, v8, dq, dk, dv = _fp8_case(rng, 1, 5, 7, 2, 2, 8)
    cu_q, cu_k = [0, 2, 5], [0, 3, 7]
    a = orc.attention_fp8(q8, k8, v8, dq, dk, dv, 0.4, orc.MASK_BLOCKDIAG_CAUSAL, cu_q, cu_k,
                          bottom_right=True)
    b = orc.attention_lanes_fp8(q8, k8, v8, dq, dk, dv, 0.4, orc.MASK_BLOCKDIAG_CAUSAL, cu_q, lk,
                                seqstart_k=cu_k[:-1], bottom_right=True)
    _close(a[0], b[0], 0.0, "fp8 lanes out")
    _close(a[1], b[1], 0.0, "fp8 lanes lse")
    assert lq == [2, 3]


PINS = [
    pin_e4m3_table,
    pin_e4m3_known_values,
    pin_fp8_bruteforce,
    pin_fp8_descale_folding,
    pin_fp8_lanes,
    pin_lanes_contiguous_equal_blockdiag,
    pin_lanes_padding_unread,
    pin_paged_equals_padded,
    pin_window_single_key,
    pin_bottom_right_reductions,
    pin_band_bruteforce,
    pin_window_split_merge,
    pin_rows_sampling,
    pin_bruteforce,
    pin_torch_sdpa,
    pin_single_key,
    pin_constant_v,
    pin_causal_row0,
    pin_zero_query,
    pin_duplicate_keys,
    pin_permute_keys,
    pin_scale_folds_into_q,
    pin_shared_kv_head,
    pin_grouped_query_heads,
    pin_merge_any_chunking,
    pin_merge_against_brute,
    pin_merge_identities,
    pin_varlen_equals_per_sequence,
    pin_varlen_partial_offset,
    pin_empty_rows,
    pin_golden_cases,
    pin_widen_bf16,
]
