"""FP8 E4M3 q/k/v: CUDA path vs the fp64 oracle on the dequantized values, through the C ABI.

Few query rows (the CUDA-core kernel) keep fp32 probabilities: the usual tolerances hold.
The tensor-core kernel rounds each probability p (relative to its running reference, at
most 2^8 above the row max) to E4M3 before P.V.  Round to nearest with 3 mantissa bits
errs by at most 2^-4 p on normal values and by at most 2^-10 (half the subnormal spacing,
2^-9) below, so an output element differs from exact attention by at most
    sum_j (2^-4 p_j + 2^-10) |v_j| / sum_j p_j            (p_j = exp(s_j - max s))
plus the bf16 rounding of the output (2^-8 relative) and fp32 slack.  The tests compute
that bound from the exact probabilities and check every element against it, and check
the RMS error against the uniform rounding-error model (variance (2^-4 p v)^2 / 3 per
term), which a systematic error (a wrong scale, a dropped key) would exceed.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import attention_fmha_fwd_gb300 as fa
import oracle
from attention_fmha_fwd_gb300 import inputs
from tests.gpu_util import compare
from tests.oracle_pins import materialize_bias

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


KIND = {"none": oracle.MASK_NONE, "causal": oracle.MASK_CAUSAL,
        "blockdiag": oracle.MASK_BLOCKDIAG, "blockdiag_causal": oracle.MASK_BLOCKDIAG_CAUSAL}


def _i32(x):
    return torch.tensor(x, dtype=torch.int32, device="cuda")


def _np(t):
    return t.numpy() if isinstance(t, torch.Tensor) else np.asarray(t)


def _run(q8, k8, v8, dq, dk, dv, mask, scale, policy=0, **kw):
    dev = lambda t: t.cuda() if isinstance(t, torch.Tensor) else t  # noqa: E731
    fa.set_path_policy(policy)
    try:
        out, lse = fa.attn_fwd_fp8(q8.cuda(), dev(k8), dev(v8), dev(dq), dev(dk), dev(dv),
                                   mask=mask, scale=scale, **kw)
        torch.cuda.synchronize()
    finally:
        fa.set_path_policy(0)
    return out.double().cpu().numpy(), lse.double().cpu().numpy()


def _p_rounding_check(out, ref, q, k, v, scale, kind, what, cu_q=None, cu_k=None, br=False,
                      wl=None, wr=None):
    """Element bound and RMS model for E4M3-rounded probabilities (see the module doc)."""
    B, M, H, D = q.shape
    Mkv = k.shape[1]
    s64 = float(np.float32(scale))
    bias = np.array(materialize_bias(KIND[kind], M, Mkv, 0, cu_q, cu_k, br, wl, wr))
    allowed = np.isfinite(bias)
    bound = np.zeros_like(ref)
    model_var = np.zeros_like(ref)
    for b in range(B):
        for h in range(H):
            hk = h // (H // k.shape[2])  # grouped K/V heads
            x = s64 * (q[b, :, h] @ k[b, :, hk].T) + bias
            rows = allowed.any(axis=1)
            mx = np.where(rows, np.max(np.where(allowed, x, -np.inf), axis=1), 0.0)
            p = np.where(allowed, np.exp(x - mx[:, None]), 0.0)
            l_ = np.where(rows, p.sum(axis=1), 1.0)
            av = np.abs(v[b, :, hk])
            bound[b, :, h] = ((2.0 ** -4) * p + (2.0 ** -10) * allowed) @ av / l_[:, None]
            model_var[b, :, h] = ((2.0 ** -8) / 3.0) * ((p * p) @ (av * av)) / (l_ * l_)[:, None]
    err = np.abs(out - ref)
    limit = bound + 2.0 ** -8 * np.abs(ref) + 1e-4
    worst = np.unravel_index(np.argmax(err - limit), err.shape)
    assert np.all(err <= limit), f"{what}: |d out| {err[worst]:.3e} > bound {limit[worst]:.3e} at {worst}"
    rms = np.sqrt(np.mean(err ** 2))
    rms_model = np.sqrt(np.mean(model_var)) + 2.0 ** -9 / np.sqrt(3) * np.sqrt(np.mean(ref ** 2))
    assert rms <= 2.0 * rms_model, f"{what}: RMS error {rms:.3e} > 2 x model {rms_model:.3e}"
    return float(err.max()), rms, rms_model


def _check_lse(lse, ref, what):
    """The row sums use the unrounded probabilities: the usual lse tolerance holds."""
    inf_ref = np.isneginf(ref)
    assert np.array_equal(np.isneginf(lse), inf_ref), f"{what}: -inf rows differ"
    if (~inf_ref).any():
        assert np.abs(lse[~inf_ref] - ref[~inf_ref]).max() <= 1e-3, f"{what}: lse"


# ------------------------------------------------------------------ CUDA-core kernel (M <= 8)

@pytest.mark.parametrize("B,M,Mkv,H,Hkv,D,mask,br,wl,per_head", [
    (2, 1, 3000, 4, None, 128, "none", False, None, True),
    (1, 5, 2500, 2, None, 64, "causal", True, 300, False),
    (2, 3, 1000, 8, 1, 128, "causal", True, None, True),      # shared K/V head
    (1, 8, 9000, 2, None, 128, "none", False, None, True),
])
def test_fp8_decode(B, M, Mkv, H, Hkv, D, mask, br, wl, per_head):
    q8, dq, k8, dk, v8, dv = inputs.qkv_fp8(B, M, Mkv, H, D, Hkv=Hkv, seed=M + Mkv, per_head=per_head)
    scale = D ** -0.5
    kd = k8.cuda()
    vd = v8.cuda()
    if Hkv == 1:
        kd, vd = kd.expand(-1, -1, H, -1), vd.expand(-1, -1, H, -1)
    out, lse = _run(q8, kd, vd, dq, dk, dv, mask, scale, policy=2, bottom_right=br, window_left=wl)
    ro, rl = oracle.attention_fp8(_np(q8), _np(k8), _np(v8), _np(dq), _np(dk), _np(dv), scale,
                                  KIND[mask], bottom_right=br, window_left=wl)
    compare(out, lse, ro, rl, f"fp8 decode B{B} M{M} Mkv{Mkv} H{H} D{D} {mask}")


def test_fp8_paged_decode():
    lq, lk, ps, H, D = [1, 2, 1, 4], [700, 64, 3001, 129], 64, 4, 128
    table, n_pages, spare = inputs.page_table(lk, ps, spare_pages=2, seed=5)
    q8, dq, k8, dk, v8, dv = inputs.qkv_fp8(1, sum(lq), n_pages * ps, H, D, seed=5)
    k8, v8 = k8.clone(), v8.clone()
    own = np.zeros(n_pages * ps, dtype=bool)
    for s in range(len(lk)):
        own[oracle.lane_rows(s, lk, block_table=table.numpy(), page_size=ps)] = True
    k8[0, torch.from_numpy(~own)] = 0x7F  # E4M3 NaN in every row no lane owns
    v8[0, torch.from_numpy(~own)] = 0x7F
    scale = D ** -0.5
    out, lse = _run(q8, k8.view(n_pages, ps, H, D), v8.view(n_pages, ps, H, D), dq, dk, dv,
                    "blockdiag_causal", scale, policy=2, seqlen_k=_i32(lk), block_table=table.cuda(),
                    page_size=ps, cu_seqlens_q=_i32(inputs.cu_seqlens(lq)), max_seqlen_q=max(lq),
                    max_seqlen_k=max(lk), bottom_right=True)
    ro, rl = oracle.attention_lanes_fp8(_np(q8), _np(k8), _np(v8), _np(dq), _np(dk), _np(dv), scale,
                                        oracle.MASK_BLOCKDIAG_CAUSAL, inputs.cu_seqlens(lq), lk,
                                        block_table=table.numpy(), page_size=ps, bottom_right=True)
    compare(out, lse, ro, rl, "fp8 paged decode")


# ------------------------------------------------------------------ tensor-core kernel

def _deq(x8, d):
    return oracle.dequantize_e4m3(_np(x8), _np(d))


@pytest.mark.parametrize("B,M,Mkv,H,mask,br,wl,per_head", [
    (1, 300, 700, 2, "none", False, None, True),
    (2, 640, 640, 2, "causal", False, None, True),
    (1, 200, 900, 2, "causal", True, 150, False),
    (1, 129, 129, 3, "none", False, None, True),
])
def test_fp8_tensor_core(B, M, Mkv, H, mask, br, wl, per_head):
    q8, dq, k8, dk, v8, dv = inputs.qkv_fp8(B, M, Mkv, H, 128, seed=M + 7, per_head=per_head)
    scale = 128 ** -0.5
    out, lse = _run(q8, k8, v8, dq, dk, dv, mask, scale, bottom_right=br, window_left=wl)
    ro, rl = oracle.attention_fp8(_np(q8), _np(k8), _np(v8), _np(dq), _np(dk), _np(dv), scale,
                                  KIND[mask], bottom_right=br, window_left=wl)
    _check_lse(lse, rl, f"fp8 tc M{M}")
    _p_rounding_check(out, ro, _deq(q8, dq), _deq(k8, dk), _deq(v8, dv), scale, mask,
                      f"fp8 tc B{B} M{M} Mkv{Mkv} {mask} br{br} wl{wl}", br=br, wl=wl)


@pytest.mark.parametrize("M,Mkv,mask,br", [(300, 700, "causal", True), (200, 200, "none", False)])
def test_fp8_tensor_core_head_dim_64(M, Mkv, mask, br):
    """Head dim 64 on the 128-wide E4M3 kernel: the tensor maps zero-fill columns 64..127."""
    q8, dq, k8, dk, v8, dv = inputs.qkv_fp8(2, M, Mkv, 2, 64, seed=M + 64)
    scale = 64 ** -0.5
    out, lse = _run(q8, k8, v8, dq, dk, dv, mask, scale, bottom_right=br)
    ro, rl = oracle.attention_fp8(_np(q8), _np(k8), _np(v8), _np(dq), _np(dk), _np(dv), scale,
                                  KIND[mask], bottom_right=br)
    _check_lse(lse, rl, f"fp8 tc d64 M{M}")
    _p_rounding_check(out, ro, _deq(q8, dq), _deq(k8, dk), _deq(v8, dv), scale, mask,
                      f"fp8 tc d64 M{M} {mask}", br=br)


def test_fp8_tensor_core_varlen():
    lq, lk = [100, 300, 20, 260], [200, 300, 400, 129]
    cu_q, cu_k = inputs.cu_seqlens(lq), inputs.cu_seqlens(lk)
    q8, dq, k8, dk, v8, dv = inputs.qkv_fp8(1, sum(lq), sum(lk), 2, 128, seed=13)
    scale = 128 ** -0.5
    out, lse = _run(q8, k8, v8, dq, dk, dv, "blockdiag_causal", scale, cu_seqlens_q=_i32(cu_q),
                    cu_seqlens_k=_i32(cu_k), max_seqlen_q=max(lq), max_seqlen_k=max(lk),
                    bottom_right=True)
    ro, rl = oracle.attention_fp8(_np(q8), _np(k8), _np(v8), _np(dq), _np(dk), _np(dv), scale,
                                  oracle.MASK_BLOCKDIAG_CAUSAL, cu_q, cu_k, bottom_right=True)
    _check_lse(lse, rl, "fp8 tc varlen")
    _p_rounding_check(out, ro, _deq(q8, dq), _deq(k8, dk), _deq(v8, dv), scale, "blockdiag_causal",
                      "fp8 tc varlen", cu_q=cu_q, cu_k=cu_k, br=True)


def test_fp8_tensor_core_paged():
    lq, lk, ps = [130, 40], [500, 257], 128
    table, n_pages, _ = inputs.page_table(lk, ps, spare_pages=2, seed=8)
    q8, dq, k8, dk, v8, dv = inputs.qkv_fp8(1, sum(lq), n_pages * ps, 2, 128, seed=8)
    scale = 128 ** -0.5
    out, lse = _run(q8, k8.view(n_pages, ps, 2, 128), v8.view(n_pages, ps, 2, 128), dq, dk, dv,
                    "blockdiag_causal", scale, seqlen_k=_i32(lk), block_table=table.cuda(),
                    page_size=ps, cu_seqlens_q=_i32(inputs.cu_seqlens(lq)), max_seqlen_q=max(lq),
                    max_seqlen_k=max(lk), bottom_right=True)
    ro, rl = oracle.attention_lanes_fp8(_np(q8), _np(k8), _np(v8), _np(dq), _np(dk), _np(dv), scale,
                                        oracle.MASK_BLOCKDIAG_CAUSAL, inputs.cu_seqlens(lq), lk,
                                        block_table=table.numpy(), page_size=ps, bottom_right=True)
    _check_lse(lse, rl, "fp8 tc paged")
    # the same keys laid out contiguously give the bound's probabilities
    rows = np.concatenate([oracle.lane_rows(s, lk, block_table=table.numpy(), page_size=ps)
                           for s in range(len(lk))])
    kc, vc = _deq(k8, dk)[:, rows], _deq(v8, dv)[:, rows]
    _p_rounding_check(out, ro, _deq(q8, dq), kc, vc, scale, "blockdiag_causal", "fp8 tc paged",
                      cu_q=inputs.cu_seqlens(lq), cu_k=inputs.cu_seqlens(lk), br=True)


def test_fp8_both_paths_agree_within_bound():
    """Eight query rows on both kernels: fp32 probabilities (CUDA cores) and E4M3
    probabilities (tensor cores) both within the E4M3 bound of the oracle."""
    q8, dq, k8, dk, v8, dv = inputs.qkv_fp8(1, 8, 2000, 2, 128, seed=31)
    scale = 128 ** -0.5
    ro, rl = oracle.attention_fp8(_np(q8), _np(k8), _np(v8), _np(dq), _np(dk), _np(dv), scale)
    a = _run(q8, k8, v8, dq, dk, dv, "none", scale, policy=2)
    compare(a[0], a[1], ro, rl, "fp8 8 rows, CUDA cores")
    fa.set_path_policy(1)
    try:
        b = _run(q8, k8, v8, dq, dk, dv, "none", scale)
    finally:
        fa.set_path_policy(0)
    _p_rounding_check(b[0], ro, _deq(q8, dq), _deq(k8, dk), _deq(v8, dv), scale, "none",
                      "fp8 8 rows, tensor cores")


def test_fp8_single_row_decode_on_tensor_cores():
    """One query row over 16 x 8 (batch, head) units: the automatic choice sends E4M3 decode
    to the tensor cores (split units), within the E4M3 probability bound of the oracle."""
    q8, dq, k8, dk, v8, dv = inputs.qkv_fp8(16, 1, 3000, 8, 128, seed=41)
    scale = 128 ** -0.5
    out, lse = _run(q8, k8, v8, dq, dk, dv, "causal", scale, bottom_right=True)
    ro, rl = oracle.attention_fp8(_np(q8), _np(k8), _np(v8), _np(dq), _np(dk), _np(dv), scale,
                                  oracle.MASK_CAUSAL, bottom_right=True)
    assert np.abs(lse - rl).max() <= 1e-3
    _p_rounding_check(out, ro, _deq(q8, dq), _deq(k8, dk), _deq(v8, dv), scale, "causal",
                      "fp8 one row, tensor cores", br=True)
