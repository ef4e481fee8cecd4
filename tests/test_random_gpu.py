"""Seeded random sweep over the call surface: CUDA path vs the fp64 oracle through the C ABI.

Every case draws, from its own seed, the batch, query and key counts (tile edges and ragged
tails included), query and K/V head counts (grouped heads), head dim (64, 96, 128), mask
(none / causal, top-left or bottom-right, left and right windows), forward or partial (with
a key offset and an fp32 or bf16 output), the scale and the path policy (automatic, tensor
cores, CUDA cores).  Sizes stay small enough for the oracle to finish each case in well
under a second; the tolerances are the parity bar of tests/gpu_util.py.
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
N_CASES = 200


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


def _draw(seed: int) -> dict:
    rng = np.random.default_rng(1000 + seed)
    c = dict(
        B=int(rng.integers(1, 4)),
        M=int(rng.choice([1, 2, 5, 8, 64, 127, 128, 129, 255, 256, 300, 513])),
        Mkv=int(rng.choice([1, 7, 128, 129, 200, 384, 777, 1500])),
        Hkv=int(rng.choice([1, 2])),
        group=int(rng.choice([1, 1, 2, 4])),
        D=int(rng.choice([64, 96, 128])),
        mask=str(rng.choice(["none", "causal"])),
        partial=bool(rng.random() < 0.3),
        scale=float(rng.uniform(0.03, 0.25)),
        policy=int(rng.choice([0, 0, 1, 2])),
    )
    c["bottom_right"] = bool(rng.random() < 0.5) and not c["partial"]
    c["window_left"] = int(rng.integers(0, 600)) if rng.random() < 0.3 else None
    c["window_right"] = (int(rng.integers(0, 300)) if c["mask"] == "none" and rng.random() < 0.3
                         else None)
    c["kv_offset"] = int(rng.integers(-400, 400)) if c["partial"] else 0
    c["out_dtype"] = torch.bfloat16 if rng.random() < 0.3 else torch.float32
    return c


@pytest.mark.parametrize("seed", range(N_CASES))
def test_random_case(seed):
    c = _draw(seed)
    B, M, Mkv, Hkv, D = c["B"], c["M"], c["Mkv"], c["Hkv"], c["D"]
    H = Hkv * c["group"]
    q, k, v = inputs.qkv(B, M, Mkv, H, D, Hkv=Hkv, seed=seed)
    wl, wr, s = c["window_left"], c["window_right"], c["scale"]
    fa.set_path_policy(c["policy"])
    try:
        if c["partial"]:
            out, lse = fa.attn_partial(*to_dev(q, k, v), mask=c["mask"], scale=s,
                                       kv_offset=c["kv_offset"], out_dtype=c["out_dtype"],
                                       window_left=wl, window_right=wr)
        else:
            out, lse = fa.attn_fwd(*to_dev(q, k, v), mask=c["mask"], scale=s,
                                   bottom_right=c["bottom_right"], window_left=wl,
                                   window_right=wr)
        torch.cuda.synchronize()
    finally:
        fa.set_path_policy(0)
    if c["partial"]:
        ro, rl = oracle.attention_partial(f32(q), f32(k), f32(v), s, KIND[c["mask"]],
                                          kv_offset=c["kv_offset"], window_left=wl,
                                          window_right=wr)
    else:
        ro, rl = oracle.attention(f32(q), f32(k), f32(v), s, KIND[c["mask"]],
                                  bottom_right=c["bottom_right"], window_left=wl,
                                  window_right=wr)
    compare(out.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl, f"seed {seed}: {c}")


# ------------------------------------------------------------------ E4M3 inputs

def _draw_fp8(seed: int) -> dict:
    rng = np.random.default_rng(5000 + seed)
    c = dict(
        B=int(rng.integers(1, 4)),
        M=int(rng.choice([1, 3, 8, 64, 129, 300])),
        Mkv=int(rng.choice([7, 128, 200, 777, 1500])),
        Hkv=int(rng.choice([1, 2])),
        group=int(rng.choice([1, 2, 4])),
        D=int(rng.choice([64, 96, 128])),
        mask=str(rng.choice(["none", "causal"])),
        per_head=bool(rng.random() < 0.5),
        scale=float(rng.uniform(0.03, 0.2)),
        policy=int(rng.choice([0, 0, 1, 2])),
        bottom_right=bool(rng.random() < 0.5),
    )
    c["window_left"] = int(rng.integers(0, 600)) if rng.random() < 0.3 else None
    c["window_right"] = (int(rng.integers(0, 300)) if c["mask"] == "none" and rng.random() < 0.3
                         else None)
    return c


@pytest.mark.parametrize("seed", range(60))
def test_random_fp8_case(seed):
    """E4M3 q/k/v with tensorwise or per-head descales on either kernel: lse within 1e-3 and
    the output within the E4M3 probability bound (which the CUDA-core kernel's exact
    products also meet)."""
    from tests.test_fp8_gpu import _check_lse, _deq, _p_rounding_check
    c = _draw_fp8(seed)
    B, M, Mkv, Hkv, D = c["B"], c["M"], c["Mkv"], c["Hkv"], c["D"]
    H = Hkv * c["group"]
    q8, dq, k8, dk, v8, dv = inputs.qkv_fp8(B, M, Mkv, H, D, Hkv=Hkv, seed=seed,
                                            per_head=c["per_head"])
    s, wl, wr, br = c["scale"], c["window_left"], c["window_right"], c["bottom_right"]
    fa.set_path_policy(c["policy"])
    try:
        out, lse = fa.attn_fwd_fp8(q8.cuda(), k8.cuda(), v8.cuda(), dq.cuda(), dk.cuda(), dv.cuda(),
                                   mask=c["mask"], scale=s, bottom_right=br, window_left=wl,
                                   window_right=wr)
        torch.cuda.synchronize()
    finally:
        fa.set_path_policy(0)
    ro, rl = oracle.attention_fp8(q8.numpy(), k8.numpy(), v8.numpy(), dq.numpy(), dk.numpy(),
                                  dv.numpy(), s, KIND[c["mask"]], bottom_right=br, window_left=wl,
                                  window_right=wr)
    what = f"fp8 seed {seed}: {c}"
    _check_lse(lse.double().cpu().numpy(), rl, what)
    _p_rounding_check(out.double().cpu().numpy(), ro, _deq(q8, dq), _deq(k8, dk), _deq(v8, dv), s,
                      c["mask"], what, br=br, wl=wl, wr=wr)


# ------------------------------------------------------------------ key lanes

@pytest.mark.parametrize("seed", range(40))
def test_random_lanes_case(seed):
    """Paged key lanes with ragged lengths (spare pages and lane tails poisoned with NaN),
    a few to a few hundred queries per sequence, page sizes 64 (few queries only), 128 and
    256, grouped heads, causal / windowed / full block-diagonal masks."""
    from tests.test_lanes_gpu import _paged
    rng = np.random.default_rng(9000 + seed)
    n = int(rng.integers(1, 7))
    few = rng.random() < 0.5
    lq = [int(x) for x in rng.choice([0, 1, 2, 5, 8] if few else [0, 1, 8, 100, 300], size=n)]
    if max(lq) == 0:
        lq[0] = 1
    lk = [int(x) for x in rng.integers(1, 3000, size=n)]
    page_size = int(rng.choice([64, 128, 256] if max(lq) <= 8 else [128, 256]))
    hkv = int(rng.choice([1, 2, 4]))
    mask = str(rng.choice(["blockdiag_causal", "blockdiag"]))
    br = bool(rng.random() < 0.7)
    wl = int(rng.integers(0, 500)) if rng.random() < 0.3 else None
    D = int(rng.choice([64, 128]))
    _paged(lq, lk, page_size, H=4, D=D, mask=mask, br=br, wl=wl, hkv=hkv, seed=seed,
           policy=int(rng.choice([0, 0, 1, 2])) if max(lq) <= 8 and page_size >= 128 else 0)
