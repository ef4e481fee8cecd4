"""ctypes declarations of the C ABI in include/mslk_attn.h (names and types only).

Loading fails loudly: there is no fallback when libmslk_attn.so is missing.
"""

from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmslk_attn.so")

MSLK_OK = 0
MSLK_ERR_INVALID_ARG = 1
MSLK_ERR_UNSUPPORTED = 2
MSLK_ERR_MISALIGNED = 3
MSLK_ERR_CUDA = 4
MSLK_ERR_DEVICE_TIMEOUT = 5
STATUS_NAMES = {
    0: "MSLK_OK", 1: "MSLK_ERR_INVALID_ARG", 2: "MSLK_ERR_UNSUPPORTED",
    3: "MSLK_ERR_MISALIGNED", 4: "MSLK_ERR_CUDA", 5: "MSLK_ERR_DEVICE_TIMEOUT",
}

MASK_NONE = 0
MASK_CAUSAL = 1
MASK_BLOCKDIAG = 2
MASK_BLOCKDIAG_CAUSAL = 3
MASK_CAUSAL_BOTTOM_RIGHT = 4
MASK_BLOCKDIAG_CAUSAL_BOTTOM_RIGHT = 5
DTYPE_BF16 = 0
DTYPE_FP32 = 1


class Strides(ctypes.Structure):
    _fields_ = [("b", ctypes.c_int64), ("m", ctypes.c_int64), ("h", ctypes.c_int64)]


class Seqlens(ctypes.Structure):
    _fields_ = [
        ("cu_seqlens_q", ctypes.c_void_p),
        ("cu_seqlens_k", ctypes.c_void_p),
        ("n_seqs", ctypes.c_int32),
        ("max_seqlen_q", ctypes.c_int32),
        ("max_seqlen_k", ctypes.c_int32),
    ]


class Band(ctypes.Structure):
    _fields_ = [("bottom_right", ctypes.c_int32), ("window_left", ctypes.c_int32),
                ("window_right", ctypes.c_int32)]


class KvLanes(ctypes.Structure):
    _fields_ = [("seqlen_k", ctypes.c_void_p), ("seqstart_k", ctypes.c_void_p),
                ("block_table", ctypes.c_void_p), ("page_size", ctypes.c_int32),
                ("max_pages", ctypes.c_int32)]


class Fp8Scales(ctypes.Structure):
    _fields_ = [("descale_q", ctypes.c_void_p), ("descale_k", ctypes.c_void_p),
                ("descale_v", ctypes.c_void_p), ("per_tensor", ctypes.c_int32)]


class AttnArgs(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("sq", Strides), ("sk", Strides), ("sv", Strides), ("so", Strides),
                ("B", ctypes.c_int32), ("M", ctypes.c_int32), ("Mkv", ctypes.c_int32),
                ("H", ctypes.c_int32), ("Hkv", ctypes.c_int32), ("K", ctypes.c_int32),
                ("Kv", ctypes.c_int32), ("scale", ctypes.c_float), ("mask_kind", ctypes.c_int32),
                ("seqlens", ctypes.c_void_p), ("band", ctypes.c_void_p), ("lanes", ctypes.c_void_p),
                ("fp8", ctypes.c_void_p), ("partial", ctypes.c_int32), ("kv_offset", ctypes.c_int64),
                ("out", ctypes.c_void_p), ("out_dtype", ctypes.c_int32), ("lse", ctypes.c_void_p),
                ("flags", ctypes.c_uint32)]


FLAG_INDEPENDENT = 1

# mslk_attn_plan results (bits)
PLAN_NONE = 0
PLAN_FILL = 1
PLAN_CUDA_CORES = 2
PLAN_TENSOR_CORES = 4
PLAN_FOLDED_HEADS = 8
PLAN_SPLIT_UNITS = 16

MERGE_MAX_VARARGS = 128
SPLIT_KV_STATIC_BYTES = 16 << 20


class MslkError(RuntimeError):
    """A non-OK mslk_status, with the library's reason string."""

    def __init__(self, status: int, reason: str):
        self.status = status
        self.reason = reason
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {reason}")


_P = ctypes.c_void_p
_S = ctypes.POINTER(Strides)
_i32 = ctypes.c_int32
_i64 = ctypes.c_int64

# name -> (restype, argtypes), in header order.
SIGNATURES = {
    "mslk_attn_fwd": (_i32, [_P, _P, _P, _S, _S, _S, _S, _i32, _i32, _i32, _i32, _i32, _i32,
                             ctypes.c_float, _i32, ctypes.POINTER(Seqlens), _P, _P, _P]),
    "mslk_attn_partial": (_i32, [_P, _P, _P, _S, _S, _S, _S, _i32, _i32, _i32, _i32, _i32, _i32,
                                 ctypes.c_float, _i32, ctypes.POINTER(Seqlens), _i64, _P, _i32,
                                 _P, _P]),
    "mslk_attn_fwd_band": (_i32, [_P, _P, _P, _S, _S, _S, _S, _i32, _i32, _i32, _i32, _i32, _i32,
                                  ctypes.c_float, _i32, ctypes.POINTER(Seqlens), ctypes.POINTER(Band),
                                  _P, _P, _P]),
    "mslk_attn_partial_band": (_i32, [_P, _P, _P, _S, _S, _S, _S, _i32, _i32, _i32, _i32, _i32,
                                      _i32, ctypes.c_float, _i32, ctypes.POINTER(Seqlens),
                                      ctypes.POINTER(Band), _i64, _P, _i32, _P, _P]),
    "mslk_attn_fwd_lanes": (_i32, [_P, _P, _P, _S, _S, _S, _S, _i32, _i32, _i32, _i32, _i32,
                                   ctypes.c_float, _i32, ctypes.POINTER(Seqlens),
                                   ctypes.POINTER(KvLanes), ctypes.POINTER(Band), _P, _P, _P]),
    "mslk_attn_fwd_fp8": (_i32, [_P, _P, _P, _S, _S, _S, _S, _i32, _i32, _i32, _i32, _i32, _i32,
                                 ctypes.c_float, _i32, ctypes.POINTER(Seqlens), ctypes.POINTER(Band),
                                 ctypes.POINTER(KvLanes), ctypes.POINTER(Fp8Scales), _P, _P, _P]),
    "mslk_attn": (_i32, [ctypes.POINTER(AttnArgs), _P]),
    "mslk_attn_plan": (_i32, [ctypes.POINTER(AttnArgs), ctypes.POINTER(ctypes.c_int32)]),
    "mslk_merge_attentions": (_i32, [_P, _P, _i32, _i64, _i64, _i32, _i32, _i32, _i32, _S, _S,
                                     _P, _i32, _P, _P]),
    "mslk_merge_attentions_varargs": (_i32, [ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(ctypes.c_void_p),
                                             _i32, _i32, _i32, _i32, _i32, _S, _S, _P, _i32, _P, _P]),
    "mslk_splitk_size": (_i32, [_i32, _i32, _i32, _i32, _i32]),
    "mslk_attn_split_kv": (_i32, [ctypes.POINTER(AttnArgs), _i32, _P, ctypes.c_size_t, _P]),
    "mslk_attn_split_kv_static": (_i32, [ctypes.POINTER(AttnArgs), _i32, _P]),
    "mslk_attn_split_kv_workspace": (_i32, [ctypes.POINTER(AttnArgs), _i32, ctypes.POINTER(ctypes.c_size_t)]),
    "mslk_last_error": (ctypes.c_char_p, []),
    "mslk_device_status": (_i32, [_P]),
    "mslk_set_wait_timeout_ns": (None, [_i64]),
    "mslk_diag_bounded_wait": (_i32, [_P]),
    "mslk_set_path_policy": (None, [_i32]),
    "mslk_version": (_i32, []),
}

_lib = None
_lock = threading.Lock()


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libmslk_attn.so (once) and declare its functions."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(
                f"{p} is missing: build it with attention_fmha_fwd_gb300.build.build() "
                "(nvcc, sm_103a); there is no fallback implementation")
        lib = ctypes.CDLL(p)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        if path is None:
            _lib = lib
        return lib


def check(status: int) -> None:
    if status != MSLK_OK:
        reason = load().mslk_last_error()
        raise MslkError(status, reason.decode() if reason else "")
