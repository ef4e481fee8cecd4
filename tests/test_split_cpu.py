"""Host-side logic of the split-KV call, the varargs merge and the BMGHK views (no GPU):
the split-size rule, argument rejection before any launch, workspace sizes, and the
flattening of 5-D tensors into views without copies."""

import ctypes

import pytest
import torch

from attention_fmha_fwd_gb300 import _capi, api, build

S = _capi.Strides
FAKE = 0x10000  # never dereferenced


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _capi.load()


@pytest.mark.parametrize("args,want", [
    ((16, 32768, 8, 256, 152), 16384),   # 128 units: two splits each fill 152 SMs
    ((1, 131072, 8, 256, 152), 6912),    # 8 units: 19 splits of ceil(131072 / 19) -> x256
    ((1, 1024, 16, 256, 152), 256),      # 16 units: 10 splits, at least one tile each
    ((1, 256, 1, 256, 152), 0),          # one tile of keys: no split
    ((200, 8192, 1, 256, 152), 0),       # more units than SMs: no split
    ((2, 5000, 4, 128, 64), 640),        # 8 units, 8 splits: 625 -> 640
    ((0, 100, 1, 256, 152), 0), ((1, 0, 1, 256, 152), 0), ((1, 100, 0, 256, 152), 0),
])
def test_splitk_size_rule(lib, args, want):
    assert lib.mslk_splitk_size(*args) == want


def test_splitk_size_defaults(lib):
    # tile_n <= 0 means 256; the result is always a multiple of it (or 0)
    assert lib.mslk_splitk_size(1, 100000, 2, 0, 152) == lib.mslk_splitk_size(1, 100000, 2, 256, 152)
    for b, n, h in ((1, 77777, 3), (3, 40000, 8), (1, 9000, 1)):
        got = lib.mslk_splitk_size(b, n, h, 128, 152)
        assert got % 128 == 0 and 0 <= got < n


def _args(**kw):
    s = S(8 * 128 * 64, 8 * 128, 128)
    a = _capi.AttnArgs()
    a.q = a.k = a.v = a.out = a.lse = FAKE
    a.sq = a.sk = a.sv = a.so = s
    a.B, a.M, a.Mkv, a.H, a.Hkv, a.K, a.Kv = 2, 64, 1024, 8, 0, 128, 128
    for k_, v_ in kw.items():
        setattr(a, k_, v_)
    return a


def _ws(lib, a, n):
    b = ctypes.c_size_t(0)
    st = lib.mslk_attn_split_kv_workspace(ctypes.byref(a), n, ctypes.byref(b))
    return st, b.value


def test_split_workspace_reads_no_pointers(lib):
    a = _args()
    a.q = a.k = a.v = a.out = a.lse = None
    st, b = _ws(lib, a, 4)
    assert st == _capi.MSLK_OK and b == _ws(lib, _args(), 4)[1]


def test_split_workspace_size(lib):
    a = _args()
    st, b = _ws(lib, a, 4)
    out_chunk, lse_chunk = 2 * 64 * 8 * 128 * 4, 2 * 8 * 64 * 4
    assert st == _capi.MSLK_OK
    assert b == 4 * out_chunk + 4 * lse_chunk
    # the chunk count is cut to one per key
    st, b1 = _ws(lib, _args(Mkv=3), 10)
    assert st == _capi.MSLK_OK and b1 == 3 * out_chunk + 3 * lse_chunk
    # n_chunks = 0 follows the split-size rule: 16 units -> ceil(152 or SMs / 16) splits
    st, b0 = _ws(lib, a, 0)
    assert st == _capi.MSLK_OK and b0 % (out_chunk + lse_chunk) == 0 and b0 >= out_chunk + lse_chunk


@pytest.mark.parametrize("kw,n,status,needle", [
    (dict(partial=1), 2, _capi.MSLK_ERR_INVALID_ARG, "forward"),
    (dict(mask_kind=3, B=1), 2, _capi.MSLK_ERR_UNSUPPORTED, "block-diagonal"),
    (dict(), -1, _capi.MSLK_ERR_INVALID_ARG, "n_chunks"),
    (dict(K=80, Kv=80), 2, _capi.MSLK_ERR_UNSUPPORTED, "head dim"),
    (dict(Hkv=3), 2, _capi.MSLK_ERR_INVALID_ARG, "divide"),
])
def test_split_rejects(lib, kw, n, status, needle):
    a = _args(**kw)
    st = lib.mslk_attn_split_kv(ctypes.byref(a), n, FAKE * 256, 1 << 30, None)
    why = lib.mslk_last_error().decode()
    assert st == status, why
    assert needle in why


def test_split_rejects_workspace(lib):
    a = _args()
    _, need = _ws(lib, a, 4)
    for ws, nb, status, needle in ((None, need, _capi.MSLK_ERR_INVALID_ARG, "workspace is null"),
                                   (FAKE * 256 + 64, need, _capi.MSLK_ERR_MISALIGNED, "256-byte"),
                                   (FAKE * 256, need - 4, _capi.MSLK_ERR_INVALID_ARG, "below")):
        st = lib.mslk_attn_split_kv(ctypes.byref(a), 4, ws, nb, None)
        assert st == status and needle in lib.mslk_last_error().decode()


def test_split_passes_validation(lib):
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    a = _args(mask_kind=4)
    _, need = _ws(lib, a, 4)
    st = lib.mslk_attn_split_kv(ctypes.byref(a), 4, FAKE * 256, need, None)
    assert st == _capi.MSLK_ERR_CUDA, lib.mslk_last_error().decode()


def _varargs(lib, n=3, outs=None, lses=None, out=FAKE, Kv=128):
    s = S(64 * 8 * 128, 8 * 128, 128)
    o = (ctypes.c_void_p * max(n, 1))(*(outs or [FAKE * (c + 1) for c in range(n)]))
    ls = (ctypes.c_void_p * max(n, 1))(*(lses or [FAKE * (c + 5) for c in range(n)]))
    st = lib.mslk_merge_attentions_varargs(o, ls, n, 2, 64, 8, Kv, ctypes.byref(s), ctypes.byref(s),
                                           out, 0, FAKE, None)
    return st, lib.mslk_last_error().decode()


def test_varargs_merge_rejects(lib):
    assert _varargs(lib, n=0)[0] == _capi.MSLK_ERR_INVALID_ARG
    st, why = _varargs(lib, n=_capi.MERGE_MAX_VARARGS + 1)
    assert st == _capi.MSLK_ERR_UNSUPPORTED and "at most 128" in why
    st, why = _varargs(lib, outs=[FAKE, FAKE + 8, FAKE])
    assert st == _capi.MSLK_ERR_MISALIGNED and "chunk 1 output" in why
    st, why = _varargs(lib, lses=[FAKE, FAKE, FAKE + 2])
    assert st == _capi.MSLK_ERR_MISALIGNED and "chunk 2 lse" in why
    st, why = _varargs(lib, outs=[FAKE, None, FAKE])
    assert st == _capi.MSLK_ERR_INVALID_ARG and "chunk 1 is null" in why
    assert _varargs(lib, Kv=126)[0] == _capi.MSLK_ERR_UNSUPPORTED
    assert _varargs(lib, out=None)[0] == _capi.MSLK_ERR_INVALID_ARG


def test_varargs_merge_passes_validation(lib):
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _varargs(lib)[0] == _capi.MSLK_ERR_CUDA


def test_bmghk_views_share_storage():
    """q [B,M,G,H,K] flattens group-major; K/V expanded over H become one head per group."""
    B, M, Mkv, G, H, K = 2, 5, 7, 3, 4, 16
    q = torch.randn(B, M, G, H, K)
    k1 = torch.randn(B, Mkv, G, 1, K)
    v1 = torch.randn(B, Mkv, G, 1, K)
    q4, k4, v4, g, h = api._bmghk(q, k1.expand(B, Mkv, G, H, K), v1.expand(B, Mkv, G, H, K))
    assert (g, h) == (G, H)
    assert q4.shape == (B, M, G * H, K) and q4.data_ptr() == q.data_ptr()
    assert k4.shape == (B, Mkv, G, K) and k4.data_ptr() == k1.data_ptr()
    for gi in range(G):
        for hi in range(H):
            assert torch.equal(q4[:, :, gi * H + hi], q[:, :, gi, hi])
            # query head gi * H + hi reads K/V head (gi * H + hi) // H = gi
            assert torch.equal(k4[:, :, (gi * H + hi) // H], k1[:, :, gi, 0])
    # distinct heads per group: G * H K/V heads, a view too
    kf = torch.randn(B, Mkv, G, H, K)
    _, k5, _, _, _ = api._bmghk(q, kf, kf)
    assert k5.shape == (B, Mkv, G * H, K) and k5.data_ptr() == kf.data_ptr()
    assert torch.equal(k5[:, :, 5], kf[:, :, 1, 1])


def test_bmghk_rejects_what_would_need_a_copy():
    q = torch.randn(2, 5, 3, 4, 16).transpose(2, 3).contiguous().transpose(2, 3)  # H outer
    k = torch.randn(2, 7, 3, 1, 16)
    with pytest.raises(ValueError, match="adjacent"):
        api._bmghk(q, k, k)
    with pytest.raises(ValueError, match="groups"):
        api._bmghk(torch.randn(2, 5, 3, 4, 16), torch.randn(2, 7, 2, 1, 16), torch.randn(2, 7, 2, 1, 16))
    with pytest.raises(ValueError, match="heads per group"):
        api._bmghk(torch.randn(2, 5, 3, 4, 16), torch.randn(2, 7, 3, 2, 16), torch.randn(2, 7, 3, 2, 16))
