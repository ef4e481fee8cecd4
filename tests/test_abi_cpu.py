"""The C-ABI library without a GPU: it builds, loads, exports every declared symbol, and
rejects bad arguments with the documented status before touching the device."""

import ctypes
import os
import re

import pytest

from attention_fmha_fwd_gb300 import _capi, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mslk_attn.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _capi.load()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:mslk_status|void|int32_t|const char\*)\s+(mslk_\w+)\s*\(",
                       text, flags=re.M)
    return names


def test_header_declares_the_boundary():
    names = _declared_functions()
    for n in ("mslk_attn_fwd", "mslk_attn_partial", "mslk_merge_attentions", "mslk_last_error"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/mslk_attn.h but not exported"
    assert set(names) == set(_capi.SIGNATURES), "binding and header disagree"


def test_version(lib):
    assert lib.mslk_version() == 100


S = _capi.Strides
FAKE = 0x10000  # never dereferenced: every call below fails validation first


def _fwd(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, sq=S(8 * 128 * 64, 8 * 128, 128), sk=None, sv=None, so=None,
             B=2, M=64, Mkv=64, H=8, K=128, Kv=128, scale=0.0, mask=0, seqlens=None,
             out=FAKE, lse=FAKE)
    a.update(kw)
    for n in ("sk", "sv", "so"):
        if a[n] is None:
            a[n] = a["sq"]
    ref = lambda s: None if s is False else ctypes.byref(s)  # noqa: E731
    st = lib.mslk_attn_fwd(a["q"], a["k"], a["v"], ref(a["sq"]), ref(a["sk"]), ref(a["sv"]),
                           ref(a["so"]), a["B"], a["M"], a["Mkv"], a["H"], a["K"], a["Kv"],
                           a["scale"], a["mask"], a["seqlens"], a["out"], a["lse"], None)
    return st, lib.mslk_last_error().decode()


@pytest.mark.parametrize("kw,status,needle", [
    (dict(K=80, Kv=80), _capi.MSLK_ERR_UNSUPPORTED, "head dim 80 not supported (64, 96 or 128)"),
    (dict(K=128, Kv=64), _capi.MSLK_ERR_UNSUPPORTED, "Kv"),
    (dict(mask=7), _capi.MSLK_ERR_INVALID_ARG, "mask_kind"),
    (dict(B=-1), _capi.MSLK_ERR_INVALID_ARG, "negative"),
    (dict(sq=False), _capi.MSLK_ERR_INVALID_ARG, "null strides"),
    (dict(out=None), _capi.MSLK_ERR_INVALID_ARG, "out is null"),
    (dict(q=None), _capi.MSLK_ERR_INVALID_ARG, "null"),
    (dict(q=FAKE + 8), _capi.MSLK_ERR_MISALIGNED, "16-byte"),
    (dict(out=FAKE + 4), _capi.MSLK_ERR_MISALIGNED, "out base"),
    (dict(sq=S(8 * 128 * 64, 8 * 128 + 4, 128)), _capi.MSLK_ERR_MISALIGNED, "q sequence stride"),
    (dict(sk=S(8 * 128 * 64, 8 * 128, 0)), _capi.MSLK_ERR_INVALID_ARG, "shared"),
    (dict(sq=S(8 * 128 * 64, 8 * 128, 0)), _capi.MSLK_ERR_MISALIGNED, "q head stride"),
    (dict(sq=S(-1, 8 * 128, 128)), _capi.MSLK_ERR_MISALIGNED, "negative"),
    (dict(mask=2), _capi.MSLK_ERR_INVALID_ARG, "packed batch"),
    (dict(mask=3, B=1), _capi.MSLK_ERR_INVALID_ARG, "cu_seqlens"),
])
def test_fwd_rejects(lib, kw, status, needle):
    st, why = _fwd(lib, **kw)
    assert st == status, why
    assert needle in why


def test_fwd_bad_seqlens(lib):
    sl = _capi.Seqlens(FAKE, FAKE, 0, 10, 10)
    st, why = _fwd(lib, mask=2, B=1, seqlens=ctypes.byref(sl))
    assert st == _capi.MSLK_ERR_INVALID_ARG and "seqlens" in why
    sl = _capi.Seqlens(FAKE, FAKE, 2, 65, 10)  # max_seqlen_q > M
    st, why = _fwd(lib, mask=2, B=1, seqlens=ctypes.byref(sl))
    assert st == _capi.MSLK_ERR_INVALID_ARG


def test_fwd_empty_sizes_are_noops(lib):
    for kw in (dict(M=0), dict(B=0), dict(H=0)):
        st, why = _fwd(lib, out=None, q=None, **kw)
        assert st == _capi.MSLK_OK, why


def test_partial_requires_lse(lib):
    s = S(8 * 128 * 64, 8 * 128, 128)
    st = lib.mslk_attn_partial(FAKE, FAKE, FAKE, ctypes.byref(s), ctypes.byref(s), ctypes.byref(s),
                               ctypes.byref(s), 2, 64, 64, 8, 128, 128, 0.0, 0, None, 0, FAKE,
                               _capi.DTYPE_FP32, None, None)
    assert st == _capi.MSLK_ERR_INVALID_ARG
    assert "lse is required" in lib.mslk_last_error().decode()
    st = lib.mslk_attn_partial(FAKE, FAKE, FAKE, ctypes.byref(s), ctypes.byref(s), ctypes.byref(s),
                               ctypes.byref(s), 2, 64, 64, 8, 128, 128, 0.0, 0, None, 0, FAKE,
                               5, FAKE, None)
    assert st == _capi.MSLK_ERR_INVALID_ARG


def _band_call(lib, band, mask=0, partial=False):
    s = S(8 * 128 * 64, 8 * 128, 128)
    r = ctypes.byref
    if partial:
        st = lib.mslk_attn_partial_band(FAKE, FAKE, FAKE, r(s), r(s), r(s), r(s), 2, 64, 64, 8, 128,
                                        128, 0.0, mask, None, r(band), 0, FAKE, _capi.DTYPE_FP32,
                                        FAKE, None)
    else:
        st = lib.mslk_attn_fwd_band(FAKE, FAKE, FAKE, r(s), r(s), r(s), r(s), 2, 64, 64, 8, 128, 128,
                                    0.0, mask, None, r(band), FAKE, FAKE, None)
    return st, lib.mslk_last_error().decode()


@pytest.mark.parametrize("band,mask,partial,needle", [
    ((0, -1, 3), 1, False, "right window"),         # causal kinds have no right window
    ((0, -2, -1), 0, False, "window sizes"),
    ((0, 4, -7), 0, True, "window sizes"),
    ((2, -1, -1), 0, False, "bottom_right"),
    ((1, 3, -1), 1, True, "forward only"),           # partials fold alignment into kv_offset
    ((0, -1, -1), 4, True, "forward only"),          # bottom-right kinds are forward only
])
def test_band_rejects(lib, band, mask, partial, needle):
    st, why = _band_call(lib, _capi.Band(*band), mask, partial)
    assert st == _capi.MSLK_ERR_INVALID_ARG, why
    assert needle in why


def test_band_kinds_pass_validation(lib):
    """Bottom-right kinds and windows get past validation (then fail at the CUDA layer
    here, without a device)."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    for band, mask in (((1, 7, -1), 1), ((0, 3, 5), 0), ((1, -1, 0), 0), ((0, -1, -1), 4)):
        st, why = _band_call(lib, _capi.Band(*band), mask)
        assert st == _capi.MSLK_ERR_CUDA, why
    st, why = _fwd(lib, mask=4)
    assert st == _capi.MSLK_ERR_CUDA, why


def _merge(lib, n=2, Kv=128, cs_out=2 * 64 * 8 * 128, out_split=FAKE, out=FAKE, dtype=0,
           lse_split=FAKE, lse=FAKE):
    s = S(64 * 8 * 128, 8 * 128, 128)
    st = lib.mslk_merge_attentions(out_split, lse_split, n, cs_out, 2 * 8 * 64, 2, 64, 8, Kv,
                                   ctypes.byref(s), ctypes.byref(s), out, dtype, lse, None)
    return st, lib.mslk_last_error().decode()


def test_merge_rejects(lib):
    assert _merge(lib, n=0)[0] == _capi.MSLK_ERR_INVALID_ARG      # zero partials is an error
    assert _merge(lib, Kv=126)[0] == _capi.MSLK_ERR_UNSUPPORTED
    assert _merge(lib, out_split=FAKE + 4)[0] == _capi.MSLK_ERR_MISALIGNED
    assert _merge(lib, cs_out=6)[0] == _capi.MSLK_ERR_MISALIGNED
    assert _merge(lib, dtype=9)[0] == _capi.MSLK_ERR_INVALID_ARG
    assert _merge(lib, out=None)[0] == _capi.MSLK_ERR_INVALID_ARG
    # lse pointers are read and written as floats: a misaligned one is rejected before launch
    assert _merge(lib, lse_split=FAKE + 2) == (_capi.MSLK_ERR_MISALIGNED,
                                               "mslk_merge_attentions: lse_split/lse must be 4-byte aligned")
    assert _merge(lib, lse=FAKE + 1)[0] == _capi.MSLK_ERR_MISALIGNED


def test_valid_call_without_device_reports_cuda_error(lib):
    """A well-formed call gets past validation and fails cleanly at the CUDA layer when
    there is no device (this container); on a GPU machine it would launch."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    st, why = _fwd(lib)
    assert st == _capi.MSLK_ERR_CUDA, why


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(RuntimeError, match="no fallback"):
        _capi.load(str(tmp_path / "libmslk_attn.so"))


def _lanes_call(lib, lanes, mask=3, band=None, sl=None):
    s = S(8 * 128 * 64, 8 * 128, 128)
    r = ctypes.byref
    sl = _capi.Seqlens(FAKE, None, 4, 8, 64) if sl is None else sl
    st = lib.mslk_attn_fwd_lanes(FAKE, FAKE, FAKE, r(s), r(s), r(s), r(s), 64, 64, 8, 128, 128, 0.0,
                                 mask, r(sl), None if lanes is None else r(lanes),
                                 None if band is None else r(band), FAKE, FAKE, None)
    return st, lib.mslk_last_error().decode()


L = _capi.KvLanes


@pytest.mark.parametrize("lanes,mask,status,needle", [
    (L(FAKE, FAKE, None, 0, 0), 1, _capi.MSLK_ERR_INVALID_ARG, "block-diagonal"),
    (None, 3, _capi.MSLK_ERR_INVALID_ARG, "seqlen_k"),
    (L(None, FAKE, None, 0, 0), 3, _capi.MSLK_ERR_INVALID_ARG, "seqlen_k"),
    (L(FAKE, None, None, 0, 0), 3, _capi.MSLK_ERR_INVALID_ARG, "seqstart_k or block_table"),
    (L(FAKE, None, FAKE, 0, 4), 3, _capi.MSLK_ERR_INVALID_ARG, "page_size"),
    (L(FAKE, None, FAKE, 64, 0), 3, _capi.MSLK_ERR_INVALID_ARG, "max_pages"),
    (L(FAKE, None, FAKE, 96, 4), 3, _capi.MSLK_ERR_UNSUPPORTED, "multiple of 64"),
])
def test_lanes_rejects(lib, lanes, mask, status, needle):
    st, why = _lanes_call(lib, lanes, mask)
    assert st == status, why
    assert needle in why


def test_lanes_page_multiple_follows_query_rows(lib):
    """Sequences of more than 8 queries take the 128-key tensor-core tiles."""
    st, why = _lanes_call(lib, L(FAKE, None, FAKE, 64, 4), sl=_capi.Seqlens(FAKE, None, 4, 9, 64))
    assert st == _capi.MSLK_ERR_UNSUPPORTED and "multiple of 128" in why


def test_lanes_pass_validation(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    for lanes, mask, band in ((L(FAKE, FAKE, None, 0, 0), 2, None),
                              (L(FAKE, None, FAKE, 64, 4), 3, None),
                              (L(FAKE, None, FAKE, 256, 2), 5, _capi.Band(0, 100, -1))):
        st, why = _lanes_call(lib, lanes, mask, band)
        assert st == _capi.MSLK_ERR_CUDA, why


def _fp8_call(lib, scales="ok", B=2, M=64, K=128, sq=None, lanes=None, mask=0, sl=None):
    s = S(8 * 128 * 64, 8 * 128, 128) if sq is None else sq
    so = S(8 * 128 * 64, 8 * 128, 128)
    r = ctypes.byref
    if scales == "ok":
        scales = _capi.Fp8Scales(FAKE, FAKE, FAKE, 0)
    st = lib.mslk_attn_fwd_fp8(FAKE, FAKE, FAKE, r(s), r(s), r(s), r(so), B, M, 64, 8, K, K, 0.0,
                               mask, None if sl is None else r(sl), None,
                               None if lanes is None else r(lanes),
                               None if scales is None else r(scales), FAKE, FAKE, None)
    return st, lib.mslk_last_error().decode()


@pytest.mark.parametrize("kw,status,needle", [
    (dict(scales=None), _capi.MSLK_ERR_INVALID_ARG, "descale"),
    (dict(scales=_capi.Fp8Scales(FAKE, None, FAKE, 0)), _capi.MSLK_ERR_INVALID_ARG, "descale"),
    (dict(scales=_capi.Fp8Scales(FAKE, FAKE, FAKE, 2)), _capi.MSLK_ERR_INVALID_ARG, "per_tensor"),
    (dict(scales=_capi.Fp8Scales(FAKE, FAKE + 2, FAKE, 0)), _capi.MSLK_ERR_MISALIGNED, "4-byte"),
    (dict(sq=S(8 * 136 * 64, 8 * 136, 136)), _capi.MSLK_ERR_MISALIGNED, "16 elements"),  # 136 % 16
    (dict(K=80), _capi.MSLK_ERR_UNSUPPORTED, "head dim"),
    (dict(lanes=L(FAKE, FAKE, None, 0, 0), mask=2), _capi.MSLK_ERR_INVALID_ARG, "B = 1"),
])
def test_fp8_rejects(lib, kw, status, needle):
    st, why = _fp8_call(lib, **kw)
    assert st == status, why
    assert needle in why


def test_fp8_bf16_strides_pass(lib):
    """A stride that is a multiple of 8 bf16 elements but not of 16 bytes of E4M3 is refused
    only for the E4M3 call."""
    sq = S(8 * 136 * 64, 8 * 136, 136)
    st, why = _fwd(lib, sq=sq)
    assert st != _capi.MSLK_ERR_MISALIGNED, why


def test_fp8_pass_validation(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    for kw in (dict(), dict(K=64, M=4), dict(K=64), dict(scales=_capi.Fp8Scales(FAKE, FAKE, FAKE, 1)),
               dict(B=1, mask=3, lanes=L(FAKE, None, FAKE, 128, 4),
                    sl=_capi.Seqlens(FAKE, None, 4, 16, 64))):
        st, why = _fp8_call(lib, **kw)
        assert st == _capi.MSLK_ERR_CUDA, why


def test_attn_args_layout_matches_header(tmp_path):
    """The ctypes mirror of mslk_attn_args has the C struct's size and field offsets."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    fields = [f for f, _ in _capi.AttnArgs._fields_]
    src = tmp_path / "layout.c"
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "mslk_attn.h"\nint main(void) {\n'
                   '  printf("%zu\\n", sizeof(mslk_attn_args));\n'
                   + "".join(f'  printf("%zu\\n", offsetof(mslk_attn_args, {f}));\n' for f in fields)
                   + "  return 0;\n}\n")
    exe = tmp_path / "layout"
    subprocess.run([cc, "-I", os.path.join(ROOT, "include"), "-o", str(exe), str(src)], check=True)
    got = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    want = [ctypes.sizeof(_capi.AttnArgs)] + [getattr(_capi.AttnArgs, f).offset for f in fields]
    assert got == want


def _args(**kw):
    s = S(8 * 128 * 64, 8 * 128, 128)
    a = _capi.AttnArgs()
    a.q = a.k = a.v = a.out = a.lse = FAKE
    a.sq = a.sk = a.sv = a.so = s
    a.B, a.M, a.Mkv, a.H, a.Hkv, a.K, a.Kv = 2, 64, 64, 8, 0, 128, 128
    for k_, v_ in kw.items():
        setattr(a, k_, v_)
    return a


@pytest.mark.parametrize("kw,status,needle", [
    (dict(Hkv=3), _capi.MSLK_ERR_INVALID_ARG, "divide"),
    (dict(Hkv=-1), _capi.MSLK_ERR_INVALID_ARG, "negative Hkv"),
    (dict(partial=2), _capi.MSLK_ERR_INVALID_ARG, "partial"),
    (dict(partial=1, lse=None), _capi.MSLK_ERR_INVALID_ARG, "lse is required"),
    (dict(out_dtype=7), _capi.MSLK_ERR_INVALID_ARG, "out_dtype"),
    (dict(flags=6), _capi.MSLK_ERR_INVALID_ARG, "flags"),
])
def test_general_entry_rejects(lib, kw, status, needle):
    a = _args(**kw)
    st = lib.mslk_attn(ctypes.byref(a), None)
    why = lib.mslk_last_error().decode()
    assert st == status, why
    assert needle in why


def test_general_entry_rejects_lanes_partial_and_null(lib):
    lanes = L(FAKE, FAKE, None, 0, 0)
    sl = _capi.Seqlens(FAKE, None, 2, 32, 64)
    a = _args(partial=1, B=1, mask_kind=3, lanes=ctypes.addressof(lanes), seqlens=ctypes.addressof(sl))
    assert lib.mslk_attn(ctypes.byref(a), None) == _capi.MSLK_ERR_UNSUPPORTED
    assert lib.mslk_attn(None, None) == _capi.MSLK_ERR_INVALID_ARG


def test_general_entry_passes_validation(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    for kw in (dict(), dict(Hkv=2), dict(Hkv=8, partial=1, out_dtype=1), dict(Hkv=1, M=4),
               dict(M=1, partial=1, flags=_capi.FLAG_INDEPENDENT)):
        a = _args(**kw)
        st = lib.mslk_attn(ctypes.byref(a), None)
        assert st == _capi.MSLK_ERR_CUDA, lib.mslk_last_error().decode()


def test_binding_checks_kv_heads():
    import torch
    from attention_fmha_fwd_gb300 import api
    q = torch.empty(2, 5, 8, 64)
    assert api._kv_heads(q, torch.empty(2, 7, 2, 64), torch.empty(2, 7, 2, 64)) == 2
    for k, v in ((torch.empty(2, 7, 3, 64), torch.empty(2, 7, 3, 64)),   # 3 does not divide 8
                 (torch.empty(2, 7, 2, 64), torch.empty(2, 6, 2, 64)),   # key counts differ
                 (torch.empty(1, 7, 2, 64), torch.empty(1, 7, 2, 64)),   # batch differs
                 (torch.empty(2, 7, 2, 32), torch.empty(2, 7, 2, 32))):  # head dim differs
        with pytest.raises(ValueError):
            api._kv_heads(q, k, v)


# ------------------------------------------------------------------ kernel plan (no device)

TC, CC = _capi.PLAN_TENSOR_CORES, _capi.PLAN_CUDA_CORES
FOLD, SPLIT = _capi.PLAN_FOLDED_HEADS, _capi.PLAN_SPLIT_UNITS


def _plan(lib, a, policy=0):
    out = ctypes.c_int32(-1)
    lib.mslk_set_path_policy(policy)
    try:
        st = lib.mslk_attn_plan(ctypes.byref(a), ctypes.byref(out))
    finally:
        lib.mslk_set_path_policy(0)
    assert st == _capi.MSLK_OK, lib.mslk_last_error().decode()
    return out.value


@pytest.mark.parametrize("kw,policy,want", [
    (dict(B=2, M=2048, Mkv=2048, H=32, mask_kind=1), 0, TC),           # causal forward
    (dict(B=16, M=1, Mkv=32768, H=8), 0, CC),                          # bf16 decode: one row
    (dict(B=16, M=1, Mkv=32768, H=8), 1, TC | SPLIT),                  # ... forced
    (dict(B=16, M=4, Mkv=32768, H=8), 0, TC | SPLIT),                  # 4 rows, 128 units
    (dict(B=16, M=4, Mkv=32768, H=8), 2, CC),                          # ... forced
    (dict(B=1, M=4, Mkv=32768, H=8), 0, CC),                           # 4 rows, 8 units
    (dict(B=16, M=1, Mkv=32768, H=32, Hkv=8), 0, TC | FOLD | SPLIT),   # grouped decode
    (dict(B=2, M=1, Mkv=32768, H=32, Hkv=8), 0, CC),                   # ... too few units
    (dict(B=4, M=128, Mkv=4096, H=32), 0, TC | SPLIT),                 # one Q tile of rows
    (dict(B=4, M=129, Mkv=4096, H=32), 0, TC),                         # two Q tiles
    (dict(B=2, M=64, Mkv=0), 0, _capi.PLAN_FILL),                      # no keys
    (dict(B=2, M=0), 0, _capi.PLAN_NONE),                              # no queries
])
def test_plan_dense(lib, kw, policy, want):
    assert _plan(lib, _args(**kw), policy) == want


def test_plan_fp8_decode(lib):
    """One E4M3 row over 128 units goes to the tensor cores (split units); over 8 units it
    stays on the CUDA cores' cluster split."""
    scales = _capi.Fp8Scales(FAKE, FAKE, FAKE, 0)
    a = _args(B=16, M=1, Mkv=32768, H=8, fp8=ctypes.addressof(scales))
    assert _plan(lib, a) == TC | SPLIT
    a = _args(B=1, M=1, Mkv=32768, H=8, fp8=ctypes.addressof(scales))
    assert _plan(lib, a) == CC


@pytest.mark.parametrize("page_size,want", [(64, CC), (128, TC | SPLIT)])
def test_plan_paged_pages(lib, page_size, want):
    """Up to 4 queries per sequence over 64 sequences x 8 heads: the tensor cores would be
    faster, but 64-key pages (accepted for few queries) stay on the CUDA-core kernel."""
    lanes = L(FAKE, None, FAKE, page_size, 64)
    sl = _capi.Seqlens(FAKE, None, 64, 4, 4096)
    a = _args(B=1, M=256, Mkv=64 * page_size, H=8, mask_kind=3, lanes=ctypes.addressof(lanes),
              seqlens=ctypes.addressof(sl))
    assert _plan(lib, a) == want


def test_plan_validates_like_the_call(lib):
    out = ctypes.c_int32(-1)
    a = _args(Hkv=3)
    assert lib.mslk_attn_plan(ctypes.byref(a), ctypes.byref(out)) == _capi.MSLK_ERR_INVALID_ARG
    assert "divide" in lib.mslk_last_error().decode()
    assert lib.mslk_attn_plan(None, ctypes.byref(out)) == _capi.MSLK_ERR_INVALID_ARG
    assert lib.mslk_attn_plan(ctypes.byref(_args()), None) == _capi.MSLK_ERR_INVALID_ARG
