"""The seeded input generators: deterministic, and the structures they describe are valid."""

import torch

from attention_fmha_fwd_gb300 import inputs


def test_qkv_is_seeded():
    a = inputs.qkv(1, 5, 7, 2, 64, seed=3)
    b = inputs.qkv(1, 5, 7, 2, 64, seed=3)
    assert all(torch.equal(x, y) for x, y in zip(a, b))
    assert a[0].dtype == torch.bfloat16 and a[1].shape == (1, 7, 2, 64)


def test_page_table_is_a_partition():
    lens, ps = [1, 0, 256, 257, 1000], 128
    table, n_pages, spare = inputs.page_table(lens, ps, spare_pages=3, seed=4)
    need = [(n + ps - 1) // ps for n in lens]
    assert n_pages == sum(need) + 3 and len(spare) == 3
    used = [int(table[s, p]) for s, n in enumerate(need) for p in range(n)]
    assert sorted(used + spare) == list(range(n_pages))  # each page owned once
    for s, n in enumerate(need):                           # the rest point at a spare page
        assert all(int(table[s, p]) == spare[-1] for p in range(n, table.shape[1]))
    again = inputs.page_table(lens, ps, spare_pages=3, seed=4)[0]
    assert torch.equal(table, again)


def test_varlen_seqlens_sum():
    lens = inputs.varlen_seqlens(12, 16384, seed=0)
    assert sum(lens) == 16384 and min(lens) >= 1


def test_quantize_e4m3_round_trip():
    """Codes times descale reproduce the input to E4M3 precision (relative 2^-4 for normal
    values, 2^-10 descales below); the largest magnitude per head lands on 448."""
    x = inputs.qkv(1, 64, 8, 4, 32, seed=9)[0]
    codes, d = inputs.quantize_e4m3(x)
    back = codes.view(torch.float8_e4m3fn).float() * d.reshape(1, 1, -1, 1)
    err = (back - x.float()).abs()
    assert torch.all(err <= x.float().abs() * 2.0 ** -4 + d.reshape(1, 1, -1, 1) * 2.0 ** -10)
    top = codes.view(torch.float8_e4m3fn).float().abs().amax(dim=(0, 1, 3))
    assert torch.all(top == 448.0)
