"""ctypes declarations of libsd's C ABI (include/sd.h).  Marshalling only."""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsd.so")

SD_OK = 0
SD_ERR_INVALID_ARG = -1
SD_ERR_UNSUPPORTED = -2
SD_ERR_CUDA = -3
SD_ERR_TIMEOUT = -4
SD_ERR_WORKSPACE = -5

SD_IDX_SIG, SD_IDX_PLANES, SD_IDX_MINMAX, SD_IDX_LANDMARK = 0, 1, 2, 3
SD_PLAN_WATERFILL, SD_PLAN_FIXED, SD_PLAN_FULL, SD_PLAN_TOPQ, SD_PLAN_SPLIT = 0, 1, 2, 3, 4
SD_SCORE_I32, SD_SCORE_F32 = 0, 1


class SdShape(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("hq", ctypes.c_int32), ("hkv", ctypes.c_int32),
                ("d", ctypes.c_int32), ("n", ctypes.c_int64), ("n_cap", ctypes.c_int64)]


class SdEncoder(ctypes.Structure):
    _fields_ = [("W1", ctypes.c_void_p), ("b1", ctypes.c_void_p), ("hidden", ctypes.c_int32),
                ("W2", ctypes.c_void_p), ("b2", ctypes.c_void_p)]


class SdResident(ctypes.Structure):
    _fields_ = [("n_slots", ctypes.c_int32), ("slot_unit", ctypes.c_void_p),
                ("slot_last", ctypes.c_void_p), ("unit_slot", ctypes.c_void_p)]


class SdSelect(ctypes.Structure):
    _fields_ = [("k", ctypes.c_int32), ("sink", ctypes.c_int32), ("local", ctypes.c_int32),
                ("block", ctypes.c_int32)]


# name -> (restype, argtypes); the same list as include/sd.h
_p, _i, _i64, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
_PS, _PE, _PL = ctypes.POINTER(SdShape), ctypes.POINTER(SdEncoder), ctypes.POINTER(SdSelect)
_PR = ctypes.POINTER(SdResident)
SIGNATURES = {
    "sd_build_index": (_i, [_i, _PS, _p, _PE, _p, _p, _p]),
    "sd_append_index": (_i, [_i, _PS, _i64, _p, _PE, _p, _p, _p]),
    "sd_encode_query": (_i, [_PS, _p, _PE, _p, _p]),
    "sd_plan": (_i, [_PS, _p, _p, _i, _i, _p, _p]),
    "sd_score": (_i, [_i, _PS, _p, _p, _p, _p, _p, _p]),
    "sd_topk_workspace_size": (_sz, [_i64, _i64, _PL]),
    "sd_topk": (_i, [_i, _p, _i64, _i64, _i64, _PL, _p, _i64, _p, _p, _sz, _p]),
    "sd_plan_score": (_i, [_PS, _p, _p, _p, _p, _i, _i, _p, _p, _p, _p]),
    "sd_topk_wmax": (_i, [_p, _p, _i64, _i64, _PL, _p, _i64, _p, _p, _sz, _p]),
    "sd_hamming_topk_workspace_size": (_sz, [_PS, _PL]),
    "sd_hamming_topk": (_i, [_PS, _p, _p, _PL, _p, _i64, _p, _p, _sz, _p]),
    "sd_select_attend_workspace_size": (_sz, [_PS, _PL, _i64]),
    "sd_select_attend": (_i, [_PS, _p, _p, _PL, _p, _p, _p, ctypes.c_float, _p, _i64, _p, _i64,
                              _p, _p, _p, _sz, _p]),
    "sd_score_topk_workspace_size": (_sz, [_PS, _PL]),
    "sd_score_topk": (_i, [_PS, _p, _p, _p, _p, _PL, _p, _p, _i64, _p, _p, _sz, _p]),
    "sd_gather_attend_workspace_size": (_sz, [_PS, _i64]),
    "sd_gather_attend": (_i, [_PS, _p, _p, _p, _p, _i64, _p, _i64, ctypes.c_float, _p, _p, _p,
                              _sz, _p]),
    "sd_gather_attend_noalloc": (_i, [_PS, _p, _p, _p, _p, _i64, _p, _i64, ctypes.c_float, _p,
                                      _p, _p]),
    "sd_offload_gather": (_i, [_PS, _p, _p, _p, _p, _p, _p]),
    "sd_delta_select": (_i, [_PS, _PL, _p, _p, _i64, _p, ctypes.c_int32, ctypes.c_int32, _PR,
                             _p, _p, _p, _p, _p, _i64, _p, _p]),
    "sd_resident_gather": (_i, [_PS, ctypes.c_int32, _p, _p, _p, _p, _p, ctypes.c_int32,
                                ctypes.c_int32, _p, _p, _p]),
    "sd_shard_candidates": (_i, [_p, _i64, _i64, _p, _i64, _p, ctypes.c_int32, ctypes.c_int32,
                                 _i64, ctypes.c_int32, _p, _p, _p, _p]),
    "sd_topk_merge": (_i, [_i64, ctypes.c_int32, ctypes.c_int32, _p, _p, _p, _p, _i64, _p, _p]),
    "sd_shard_select": (_i, [_i64, _p, _i64, _p, _i64, _i64, ctypes.c_int32, ctypes.c_int32,
                             ctypes.c_int32, _p, _i64, _p, _p]),
    "sd_attend_combine": (_i, [ctypes.c_int32, _i64, ctypes.c_int32, _p, _p, _p, _p, _p]),
    "sd_device_status": (_i, [_p]),
    "sd_set_fallback_paths": (_i, [_i]),
    "sd_debug_set_device_error": (_i, [_p]),
    "sd_event_wait": (_i, [_p, _i64]),
    "sd_copy": (_i, [_p, _p, _sz, _p]),
    "sd_last_error": (ctypes.c_char_p, []),
    "sd_version": (_i, []),
    "sd_launch_count": (_i64, []),
}

_lib = None


def load(path: str = LIB_PATH):
    """Loads libsd.so.  Raises if it has not been built: there is no fallback."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"libsd.so not found at {path}; build it with "
            "`python -m top_sparse_decode_gb300.build` (needs nvcc)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib
