"""Each plausible mistake planted in a copy of the oracle trips at least one pin.

The mutants are text substitutions on oracle/attention.py, loaded as throwaway
modules on the CPU; the real oracle is never modified.
"""

import importlib.util
import os
import sys
import types

import pytest

from tests import oracle_pins

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "oracle", "attention.py")

MUTANTS = {
    "causal_strict_diagonal": ("allowed &= d <= hi", "allowed &= d < hi"),
    "causal_ignores_offset": ("d = (k_pos0 + np.arange(Lk)[None, :])", "d = (np.arange(Lk)[None, :])"),
    "window_left_off_by_one": ("allowed &= d >= lo", "allowed &= d > lo"),
    "window_left_ignored": ("allowed &= d >= lo", "allowed &= d >= d"),
    "bottom_right_shift_sign": ("shift = (Lk - Lq) if bottom_right else 0",
                                "shift = (Lq - Lk) if bottom_right else 0"),
    "window_right_ignored": ("hi = None if window_right is None else shift + window_right", "hi = None"),
    "window_left_ignores_shift": ("lo = None if window_left is None else shift - window_left",
                                  "lo = None if window_left is None else -window_left"),
    "blockdiag_bottom_right_global_lengths": (
        "_band(mask_kind, bottom_right, window_left, window_right, qe - qs, ke - ks)",
        "_band(mask_kind, bottom_right, window_left, window_right, M, Mkv)"),
    "rows_position_zero": ("s64, lo, hi, int(i), kv_offset)", "s64, lo, hi, 0, kv_offset)"),
    "rows_position_off_by_one": ("s64, lo, hi, int(i), kv_offset)", "s64, lo, hi, int(i) + 1, kv_offset)"),
    "scale_dropped": ("x = scale64 * (qb @ kb.T)", "x = (qb @ kb.T)"),
    "scores_use_values": ("x = scale64 * (qb @ kb.T)", "x = scale64 * (qb @ vb.T)"),
    "lse_wrong_sign": ("lse = m + np.log(l)", "lse = m - np.log(l)"),
    "lse_drops_max": ("lse = m + np.log(l)", "lse = np.log(l)"),
    "out_not_normalised": ("out = (p @ vb) / l[:, None]", "out = (p @ vb)"),
    "exp_not_shifted": ("p = np.exp(x - np.where(empty, 0.0, m)[:, None])", "p = np.exp(x)"),
    "empty_rows_not_zeroed": ("    out[empty] = 0.0\n", ""),
    "shared_head_always_zero": ("hk = h // (H // k.shape[2])  # the query head's group", "hk = 0"),
    "gqa_heads_interleaved": ("hk = h // (H // k.shape[2])  # the query head's group",
                              "hk = h % k.shape[2]"),
    "blockdiag_sees_all_keys": ("_block(qb_all[qs:qe], kb_all[ks:ke], vb_all[ks:ke], s64,",
                                "_block(qb_all[qs:qe], kb_all, vb_all, s64,"),
    "blockdiag_absolute_positions": ("s64, lo, hi, 0,\n                              kv_offset)",
                                     "s64, lo, hi, qs,\n                              ks + kv_offset)"),
    "paged_index_swapped": ("return pages[p // page_size] * page_size + p % page_size",
                            "return pages[p % page_size] * page_size + p // page_size"),
    "lane_shared_head_always_zero": ("            hk = h // (H // k.shape[2])\n", "            hk = 0\n"),
    "lane_start_ignored": ("return int(seqstart_k[s]) + p", "return p"),
    "lane_reads_padding": ("n = int(seqlen_k[s])", "n = int(seqlen_k[s]) + 1"),
    "lane_bottom_right_uses_padding": (
        "_band(mask_kind, bottom_right, window_left, window_right, qe - qs, len(rows))",
        "_band(mask_kind, bottom_right, window_left, window_right, qe - qs, len(rows) + 1)"),
    "e4m3_bias_8": ("2.0 ** (e - 7)", "2.0 ** (e - 8)"),
    "e4m3_subnormal_implicit_one": ("m / 8.0 * 2.0 ** -6", "(1.0 + m / 8.0) * 2.0 ** -6"),
    "e4m3_no_nan": ("mag = np.where((e == 15) & (m == 7), np.nan, mag)", "mag = mag"),
    "e4m3_sign_ignored": ("sign = np.where(c & 0x80, -1.0, 1.0)", "sign = 1.0"),
    "fp8_descale_wrong_axis": ("d[None, None, :, None]", "d[None, :, None, None]"),
    "fp8_descale_first_head_only": ("return x * d[0]\n", "return x * d[0]\n    d = d[:1]\n"),
    "fp8_v_descale_ignored": ("dequantize_e4m3(v8, descale_v), scale, mask_kind, cu_seqlens_q,\n                     cu_seqlens_k",
                              "dequantize_e4m3(v8, 1.0), scale, mask_kind, cu_seqlens_q,\n                     cu_seqlens_k"),
    "fp8_k_uses_q_descale": ("attention(dequantize_e4m3(q8, descale_q), dequantize_e4m3(k8, descale_k),",
                             "attention(dequantize_e4m3(q8, descale_q), dequantize_e4m3(k8, descale_q),"),
    "merge_averages": ("coef = w / sum_w[None]", "coef = np.ones_like(w) / w.shape[0]"),
    "merge_lse_drops_shift": ("lse = m_star + np.log(sum_w)", "lse = np.log(sum_w)"),
    "merge_unnormalised": ("coef = w / sum_w[None]", "coef = w"),
    "merge_first_chunk_only": ("for c, o in enumerate(outs):", "for c, o in enumerate(outs[:1]):"),
    "scale_not_float32": ("return float(np.float32(scale))", "return float(scale)"),
    "bf16_widen_wrong_shift": ("<< np.uint32(16)", "<< np.uint32(15)"),
}


def _load_mutant(name, find, replace):
    with open(SRC) as f:
        src = f.read()
    assert src.count(find) == 1, f"mutant {name}: pattern must occur exactly once"
    mod = types.ModuleType(f"oracle_mutant_{name}")
    mod.__file__ = SRC
    exec(compile(src.replace(find, replace), f"<mutant {name}>", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    mod = _load_mutant(name, *MUTANTS[name])
    failures = []
    for pin in oracle_pins.PINS:
        try:
            pin(mod)
        except Exception as e:  # noqa: BLE001 - any failure (assert, shape error) counts
            failures.append((pin.__name__, type(e).__name__))
    assert failures, f"no pin caught mutant {name}"
