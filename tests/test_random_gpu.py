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
