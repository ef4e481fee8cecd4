"""Seeded synthetic inputs shared by the tests, the benchmark and the smoke check.

This module holds no attention arithmetic: it only draws numbers and names shapes.

Recipe: one ``torch.Generator`` seeded with ``seed`` draws fp32 standard normals in the
order q, k, v, each rounded to bf16 (round-to-nearest-even).  Variable-length sequence
lengths come from a separate generator seeded the same way, drawn before q/k/v.
"""

from __future__ import annotations

import dataclasses

import torch


def randn_bf16(gen: torch.Generator, shape) -> torch.Tensor:
    """fp32 N(0, 1) from ``gen``, rounded to bf16 (CPU tensor)."""
    return torch.randn(tuple(shape), dtype=torch.float32, generator=gen).to(torch.bfloat16)


def qkv(B: int, M: int, Mkv: int, H: int, K: int, Kv: int | None = None,
        Hkv: int | None = None, seed: int = 0):
    """q [B,M,H,K], k [B,Mkv,Hkv,K], v [B,Mkv,Hkv,Kv] bf16 CPU tensors, drawn in that order."""
    Kv = K if Kv is None else Kv
    Hkv = H if Hkv is None else Hkv
    g = torch.Generator().manual_seed(seed)
    q = randn_bf16(g, (B, M, H, K))
    k = randn_bf16(g, (B, Mkv, Hkv, K))
    v = randn_bf16(g, (B, Mkv, Hkv, Kv))
    return q, k, v


def quantize_e4m3(x: torch.Tensor, head_axis: int = 2, per_head: bool = True):
    """E4M3 codes (uint8) and fp32 descales for a float tensor: descale = amax / 448 per
    head (or over the whole tensor), codes = x / descale rounded by PyTorch's own
    float8_e4m3fn conversion (round to nearest even).  Input generation only."""
    xf = x.float()
    if per_head:
        dims = [d for d in range(xf.dim()) if d != head_axis]
        amax = xf.abs().amax(dim=dims)
    else:
        amax = xf.abs().amax().reshape(1)
    descale = (amax.clamp_min(1e-12) / 448.0).float()
    shape = [1] * xf.dim()
    if per_head:
        shape[head_axis] = -1
    codes = (xf / descale.reshape(shape)).to(torch.float8_e4m3fn).view(torch.uint8)
    return codes, descale


def qkv_fp8(B: int, M: int, Mkv: int, H: int, K: int, Hkv: int | None = None, seed: int = 0,
            per_head: bool = True):
    """E4M3 q, k, v (uint8 codes, CPU) and their descales: ``qkv``'s bf16 draws quantized."""
    q, k, v = qkv(B, M, Mkv, H, K, Hkv=Hkv, seed=seed)
    out = []
    for t in (q, k, v):
        out.extend(quantize_e4m3(t, per_head=per_head))
    return tuple(out)  # q8, dq, k8, dk, v8, dv


def varlen_seqlens(n_seqs: int = 12, total: int = 16384, lo: int = 128, hi: int = 4096,
                   seed: int = 0) -> list[int]:
    """Sequence lengths for a packed batch: ``n_seqs`` integers uniform in [lo, hi],
    rescaled proportionally to sum to ``total`` (each floored, at least 1; the
    remainder goes to the last sequence)."""
    g = torch.Generator().manual_seed(seed)
    raw = torch.randint(lo, hi + 1, (n_seqs,), generator=g).tolist()
    s = sum(raw)
    lens = [max(1, (r * total) // s) for r in raw]
    lens[-1] += total - sum(lens)
    if lens[-1] < 1:
        raise ValueError("cannot fit the lengths into the requested total")
    return lens


def cu_seqlens(lengths) -> list[int]:
    """Cumulative offsets [0, L0, L0+L1, ...] of a packed batch."""
    out = [0]
    for n in lengths:
        out.append(out[-1] + int(n))
    return out


def page_table(lengths, page_size: int, spare_pages: int = 1, seed: int = 0):
    """A seeded paged layout for key lanes of the given lengths.

    Lane s gets ceil(L_s / page_size) pages; all pages (those plus ``spare_pages`` unused
    ones) are shuffled by a seeded permutation.  Table entries past a lane's pages point at
    the last spare page.  Returns (table [n_seqs, max_pages] int32, n_pages, spare) with
    ``spare`` the list of unused page indices (CPU tensors / ints).
    """
    if spare_pages < 1:
        raise ValueError("page_table needs at least one spare page")
    need = [(int(n) + page_size - 1) // page_size for n in lengths]
    n_pages = sum(need) + spare_pages
    g = torch.Generator().manual_seed(seed)
    perm = torch.randperm(n_pages, generator=g).tolist()
    spare = perm[sum(need):]
    max_pages = max(1, max(need))
    table = torch.full((len(need), max_pages), spare[-1], dtype=torch.int32)
    at = 0
    for s, n in enumerate(need):
        table[s, :n] = torch.tensor(perm[at:at + n], dtype=torch.int32)
        at += n
    return table, n_pages, spare


def equal_chunks(Mkv: int, n: int) -> list[tuple[int, int]]:
    """``n`` contiguous key ranges [start, end) covering [0, Mkv), as equal as possible."""
    return [(c * Mkv // n, (c + 1) * Mkv // n) for c in range(n)]


@dataclasses.dataclass(frozen=True)
class Workload:
    """One named attention workload (shapes only)."""

    name: str
    B: int
    M: int
    Mkv: int
    H: int
    K: int
    Kv: int
    mask: str            # "none" | "causal" | "blockdiag_causal"
    scale: float
    chunks: tuple = ()   # split-KV chunk counts exercised (partial + merge)
    n_seqs: int = 0      # packed sequences (block-diagonal masks)


WORKLOADS = {
    "tiny_fwd": Workload("tiny_fwd", 1, 128, 128, 2, 64, 64, "none", 0.125),
    "causal_fwd": Workload("causal_fwd", 2, 2048, 2048, 32, 128, 128, "causal",
                           1.0 / 128 ** 0.5),
    "split_kv": Workload("split_kv", 1, 128, 1024, 16, 128, 128, "none", 1.0 / 128 ** 0.5,
                         chunks=(2, 8)),
    # K/V drawn as G=8 groups of 1 head each, flattened to 8 heads.
    "decode_split_kv": Workload("decode_split_kv", 16, 1, 32768, 8, 128, 128, "none",
                                1.0 / 128 ** 0.5, chunks=(16,)),
    "varlen_packed": Workload("varlen_packed", 1, 16384, 16384, 32, 128, 128,
                              "blockdiag_causal", 1.0 / 128 ** 0.5, n_seqs=12),
}
