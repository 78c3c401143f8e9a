"""ctypes binding of the C ABI in include/gdn.h (argument marshalling only).

Every step of the recurrence runs in the CUDA library; this module passes
pointers, sizes and the stream handle through and turns status codes into
exceptions.  There is no CPU path: if the library is missing, loading fails.
"""
import ctypes
import os

from .build import lib_path

GDN_OK = 0
STATUS_NAMES = {
    0: "GDN_OK", 1: "GDN_ERR_NULL_POINTER", 2: "GDN_ERR_INVALID_ARG",
    3: "GDN_ERR_UNSUPPORTED_SHAPE", 4: "GDN_ERR_UNSUPPORTED_DTYPE", 5: "GDN_ERR_MISALIGNED",
    6: "GDN_ERR_BAD_CU_SEQLENS", 7: "GDN_ERR_WORKSPACE_TOO_SMALL", 8: "GDN_ERR_DEVICE_TIMEOUT",
    9: "GDN_ERR_CUDA", 10: "GDN_ERR_BAD_CACHE_LEN",
}
GDN_F32, GDN_BF16 = 0, 1
GDN_OPT_QK_L2NORM = 1
ALGOS = {"auto": 0, "scan": 1, "chunked": 2, "chunked_fused": 3, "chunked_split": 4,
         "chunked_coop": 5}
ATTN_LAYOUTS = {"auto": 0, "general": 1, "fixed_block": 2}

# Exported symbols, with ctypes signatures: (restype, argtypes)
_vp, _i32, _i64, _f32, _sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                              ctypes.c_size_t)
SIGNATURES = {
    "gdn_prefill": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i64, _i32,
                                   _i32, _i32, _i32, ctypes.c_int, _f32, ctypes.c_int, _vp, _sz,
                                   _vp]),
    "gdn_prefill_ex": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i64,
                                      _i32, _i32, _i32, _i32, ctypes.c_int, _f32, ctypes.c_int,
                                      _vp, _sz, ctypes.c_uint32, _vp]),
    "gdn_decode_step_ex": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32,
                                          _i32, _i32, ctypes.c_int, _f32, ctypes.c_uint32, _vp]),
    "gdn_prefill_workspace_size": (_sz, [_i32, _i64, _i32, _i32, _i32, _i32, ctypes.c_int,
                                         ctypes.c_int]),
    "gdn_prefill_streamed": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i32,
                                            _i32, _i32, _i32, ctypes.c_int, _f32, _i64, _vp, _sz,
                                            ctypes.c_uint32, _vp]),
    "gdn_prefill_streamed_workspace_size": (_sz, [_i64, _i32, _i32, _i32, _i32, ctypes.c_int]),
    "gdn_prefill_host": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i32, _i32,
                                        _i32, _i32, ctypes.c_int, _f32, _i64, _vp, _sz,
                                        ctypes.c_uint32, _vp]),
    "gdn_prefill_host_workspace_size": (_sz, [_i64, _i32, _i32, _i32, _i32, ctypes.c_int]),
    "gdn_prefill_noalloc": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32,
                                           _i64, _i32, _i32, _i32, _i32, ctypes.c_int, _f32,
                                           _vp]),
    "gdn_decode_step": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32,
                                       _i32, ctypes.c_int, _f32, _vp]),
    "gdn_decode_step_rmsnorm": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _f32,
                                               _i32, _i32, _i32, _i32, _i32, ctypes.c_int, _f32,
                                               ctypes.c_uint32, _vp]),
    "gdn_output_rmsnorm": (ctypes.c_int, [_vp, _vp, _i64, _i32, _i32, ctypes.c_int, _f32, _vp]),
    "gdn_decode_multi": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32,
                                        _i32, _i32, _i32, ctypes.c_int, _f32, ctypes.c_uint32,
                                        _vp]),
    "gdn_attn_decode": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32,
                                       ctypes.c_int, _f32, ctypes.c_int, _i32, _vp, _sz, _vp]),
    "gdn_attn_decode_workspace_size": (_sz, [_i32, _i32, _i32, _i32, _i32, ctypes.c_int, _i32]),
    "gdn_attn_decode_block_keys": (_i32, [_i32, _i32, _i32, _i32, _i32, ctypes.c_int, _i32]),
    "gdn_stream_status": (ctypes.c_int, [_vp]),
    "gdn_selftest_wait_timeout": (ctypes.c_int, [_i32, _vp]),
    "gdn_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "gdn_prefill_crossover_tokens": (_i32, [_i32, _i32, _i32, _i32, ctypes.c_int]),
    "gdn_prefill_form": (_i32, [_i32, _i64, _i32, _i32, _i32, _i32, ctypes.c_int, ctypes.c_int,
                                _sz, ctypes.c_uint32, _i32]),
}

_LIB = None


class GdnError(RuntimeError):
    def __init__(self, status, where=""):
        self.status = int(status)
        name = STATUS_NAMES.get(self.status, f"status {self.status}")
        super().__init__(f"{where}: {name}" if where else name)


def load(path=None):
    """Load the shared library (once) and attach the ctypes signatures."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    p = path or lib_path()
    if not os.path.exists(p):
        raise RuntimeError(
            f"CUDA library {p} is missing; build it first (python -c 'import __graft_entry__ as "
            f"g; g.build()'). There is no CPU fallback.")
    lib = ctypes.CDLL(p)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _LIB = lib
    return lib


def check(status, where):
    if status != GDN_OK:
        raise GdnError(status, where)
