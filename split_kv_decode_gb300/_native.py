"""ctypes view of libsplitkv.so (the C ABI declared in include/split_kv_decode.h).

Loading never falls back to anything: if the library has not been built the
import of the product API raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libsplitkv.so")

DA_F32, DA_F16, DA_BF16 = 0, 1, 2
DA_OK, DA_EINVAL, DA_EUNSUPPORTED, DA_ENOSPACE, DA_ELAUNCH, DA_ETIMEOUT, DA_ECUDA = range(7)
STATUS_NAMES = {0: "DA_OK", 1: "DA_EINVAL", 2: "DA_EUNSUPPORTED", 3: "DA_ENOSPACE",
                4: "DA_ELAUNCH", 5: "DA_ETIMEOUT", 6: "DA_ECUDA"}
DA_MAX_BATCH = 256
DA_FLAG_NO_COMBINE = 0x1
DA_FLAG_GQA_SIMT = 0x2
DA_FLAG_NO_CAUSAL = 0x4
DA_FLAG_MLA_SIMT = 0x8
DA_FLAG_MLA_TC = 0x10
DA_FLAG_ONE_LAUNCH = 0x20
DA_FLAG_COMBINE_LOADS = 0x40
DA_MLA_EXACT_BELOW = 2048
DA_FLAG_TEST_NO_TMA = 0x100
DA_FLAG_TEST_BAD_LAUNCH = 0x200
DA_KERNEL_GQA_TMA, DA_KERNEL_MLA_TC, DA_KERNEL_GQA_TC = 1, 2, 3


class DaArgs(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32), ("n_heads", ctypes.c_int32),
        ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
        ("v_dim", ctypes.c_int32), ("capacity", ctypes.c_int32),
        ("k_batch_stride", ctypes.c_int64), ("k_pos_stride", ctypes.c_int64),
        ("k_head_stride", ctypes.c_int64),
        ("v_batch_stride", ctypes.c_int64), ("v_pos_stride", ctypes.c_int64),
        ("v_head_stride", ctypes.c_int64),
        ("kv_dtype", ctypes.c_int32), ("out_dtype", ctypes.c_int32),
        ("scale", ctypes.c_float), ("force_splits", ctypes.c_int32),
        ("flags", ctypes.c_int32), ("timeout_us", ctypes.c_int32),
        ("q_len", ctypes.c_int32),
    ]


class DaPlan(ctypes.Structure):
    _fields_ = [
        ("kernel", ctypes.c_int32), ("num_sms", ctypes.c_int32),
        ("ctas_per_sm", ctypes.c_int32), ("tile", ctypes.c_int32),
        ("grid", ctypes.c_int32), ("n_items", ctypes.c_int32),
        ("total_splits", ctypes.c_int32), ("max_splits", ctypes.c_int32),
        ("batch", ctypes.c_int32),
        ("seq_lens", ctypes.c_int32 * DA_MAX_BATCH),
        ("chunk", ctypes.c_int32 * DA_MAX_BATCH),
        ("n_splits", ctypes.c_int32 * DA_MAX_BATCH),
        ("split_base", ctypes.c_int32 * DA_MAX_BATCH),
        ("workspace_bytes", ctypes.c_int64),
        ("est_cost", ctypes.c_int64),
    ]


# name -> (restype, argtypes), in header order
_P = ctypes.c_void_p
class DaDev(ctypes.Structure):
    _fields_ = [
        ("seq_lens", ctypes.c_void_p), ("block_table", ctypes.c_void_p),
        ("max_blocks_per_seq", ctypes.c_int32), ("block_size", ctypes.c_int32),
        ("num_blocks", ctypes.c_int32), ("reserved", ctypes.c_int32),
        ("k_block_stride", ctypes.c_int64), ("v_block_stride", ctypes.c_int64),
    ]


class DaProj(ctypes.Structure):
    _fields_ = [
        ("w", ctypes.c_void_p), ("w_dtype", ctypes.c_int32), ("out_dim", ctypes.c_int32),
        ("head_stride", ctypes.c_int64), ("row_stride", ctypes.c_int64),
    ]


SIGNATURES = {
    "decode_attn_plan": (ctypes.c_int, [ctypes.POINTER(DaArgs), _P, ctypes.c_int,
                                        ctypes.POINTER(DaPlan)]),
    "decode_attn_workspace_bytes": (ctypes.c_int64, [ctypes.POINTER(DaPlan)]),
    "decode_attn_splitk_ex": (ctypes.c_int, [ctypes.POINTER(DaArgs), ctypes.POINTER(DaPlan), _P,
                                             _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "decode_attn_combine": (ctypes.c_int, [ctypes.POINTER(DaArgs), ctypes.POINTER(DaPlan), _P,
                                           _P, _P]),
    "decode_attn_combine_ranks": (ctypes.c_int, [ctypes.POINTER(DaArgs), ctypes.POINTER(DaPlan),
                                                 _P, ctypes.c_int, _P, _P]),
    "decode_attn_splitk": (ctypes.c_int, [_P, _P, _P, _P, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_int, ctypes.c_float, _P, _P]),
    "decode_attn_device_status": (ctypes.c_int, [_P, _P]),
    "decode_attn_splitk_noalloc": (ctypes.c_int, [ctypes.POINTER(DaArgs), ctypes.POINTER(DaPlan),
                                                  _P, _P, _P, _P, _P]),
    "decode_attn_splitk_dev": (ctypes.c_int, [ctypes.POINTER(DaArgs), ctypes.POINTER(DaPlan),
                                              ctypes.POINTER(DaDev), _P, _P, _P, _P, _P,
                                              ctypes.c_size_t, _P]),
    "decode_attn_combine_proj": (ctypes.c_int, [ctypes.POINTER(DaArgs), ctypes.POINTER(DaPlan),
                                                ctypes.POINTER(DaProj), _P, ctypes.c_int, _P,
                                                _P]),
    "decode_attn_splitk_proj": (ctypes.c_int, [ctypes.POINTER(DaArgs), ctypes.POINTER(DaPlan),
                                               ctypes.POINTER(DaProj), _P, _P, _P, _P, _P,
                                               ctypes.c_size_t, _P]),
    "decode_attn_last_error": (ctypes.c_char_p, []),
    "decode_attn_release": (None, []),
    "decode_attn_version": (ctypes.c_char_p, []),
}

_lock = threading.Lock()
_lib = None


def load() -> ctypes.CDLL:
    """Load the built library; raises if it is missing (there is no fallback)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"libsplitkv.so is not built ({LIB_PATH}); run "
                    "`python -m split_kv_decode_gb300.build` or __graft_entry__.build()")
            L = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib
