"""ctypes declarations of the C ABI in include/kvc.h (argument marshalling only).

Every function here has the name and argument order of the C entry point.
Loading fails loudly when ``libsinkwin.so`` has not been built: there is no
fallback implementation.
"""

from __future__ import annotations

import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libsinkwin.so")

KVC_OK, KVC_EINVAL, KVC_ESTATE, KVC_ECUDA, KVC_ETIMEOUT, KVC_EUNSUPPORTED = 0, -1, -2, -3, -4, -5
KVC_BF16, KVC_FP4 = 0, 1
KVC_MAX_WINDOW = 16
KVC_WS_WORDS = 1024
KVC_QUANT_WS_WORDS = 256
KVC_INIT_MAGIC = 0x4B564331

_vp = ctypes.c_void_p
_i32 = ctypes.c_int32
_i64 = ctypes.c_int64


class KvcCache(ctypes.Structure):
    """Mirror of ``struct kvc_cache`` (field order and natural alignment)."""

    _fields_ = [
        ("heads", _i32), ("head_dim", _i32), ("tokens_per_frame", _i32),
        ("chunk_frames", _i32), ("window_chunks", _i32), ("dtype", _i32),
        ("k", _vp), ("v", _vp), ("k_scale", _vp), ("v_scale", _vp),
        ("k_gscale", _vp), ("v_gscale", _vp), ("dev_ws", _vp),
        ("attn_ws", _vp), ("attn_ws_bytes", ctypes.c_uint64),
        ("stage", _vp), ("stage_bytes", ctypes.c_uint64),
        ("scrub_on_evict", _i32), ("rope_offset_frames", _i32),
        ("init_magic", _i32), ("shot", _i32),
        ("chunk_of_region", _i64 * (1 + KVC_MAX_WINDOW)),
        ("frame0_of_region", _i64 * (1 + KVC_MAX_WINDOW)),
        ("last_chunk", _i64),
    ]


# name -> (restype, argtypes), exactly the declarations of include/kvc.h
SIGNATURES = {
    "kvc_sizeof_cache": (ctypes.c_size_t, []),
    "kvc_cache_bytes": (ctypes.c_size_t, [ctypes.POINTER(KvcCache), _i32]),
    "kvc_init": (_i32, [ctypes.POINTER(KvcCache)]),
    "kvc_append": (_i32, [ctypes.POINTER(KvcCache), _vp, _vp, _i64, _vp]),
    "kvc_append_shot": (_i32, [ctypes.POINTER(KvcCache), _vp, _vp, _i64, _vp]),
    "kvc_evict": (_i32, [ctypes.POINTER(KvcCache), _i64, _vp]),
    "sinkwin_attn": (_i32, [ctypes.POINTER(KvcCache), _vp, _vp, _i32, ctypes.c_float, _vp]),
    "kvc_recache": (_i32, [ctypes.POINTER(KvcCache), _vp, _vp, _vp, ctypes.c_float,
                           ctypes.POINTER(_i64), _i32, _i32, _i32, ctypes.c_float, _vp]),
    "kvc_project_append": (_i32, [ctypes.POINTER(KvcCache), _vp, _vp, _vp, _vp, ctypes.c_float,
                                  _i64, _i32, _i32, _i32, ctypes.c_float, _vp, _vp]),
    "kvc_quant_fp4": (_i32, [_vp, _i64, _vp, _vp, _vp, _vp, _vp]),
    "kvc_quant_fp4_noalloc": (_i32, [_vp, _i64, _vp, _vp, _vp, _vp]),
    "kvc_gemm_fp4": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp, _vp,
                            ctypes.c_size_t, _vp, _vp]),
    "kvc_last_device_error": (_i32, [ctypes.POINTER(KvcCache), _vp]),
    "kvc_watchdog_selftest": (_i32, [_vp, _i32, _vp]),
    "kvc_status_string": (ctypes.c_char_p, [_i32]),
}


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build the CUDA library first "
            "(python sink_short_window_sinkwin_b300/build.py)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if lib.kvc_sizeof_cache() != ctypes.sizeof(KvcCache):
        raise ImportError("kvc_cache layout mismatch between kvc.h and the binding")
    return lib


class KvcError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


_lib: ctypes.CDLL | None = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        _lib = load()
    return _lib


def status_string(status: int) -> str:
    return lib().kvc_status_string(int(status)).decode()


def check(status: int, what: str) -> None:
    if status != KVC_OK:
        raise KvcError(status, what)
