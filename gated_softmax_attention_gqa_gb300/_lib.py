"""ctypes view of libgattn.so: one Python callable per C entry point of
include/gattn.h, same names, same argument order.  Marshalling only."""
import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libgattn.so")

EXPORTS = (
    "gattn_strerror",
    "gattn_prefill_workspace_size",
    "gattn_prefill",
    "gattn_prefill_varlen_workspace_size",
    "gattn_prefill_varlen",
    "gattn_decode_workspace_size",
    "gattn_decode",
    "gattn_decode_append",
    "gattn_decode_paged",
    "gattn_decode_noalloc",
    "gattn_get_device_status",
    "gattn_set_profile_events",
    "gattn_selftest_wait_timeout",
    "gattn_o_proj",
)

_lib = None

_vp, _i, _i64, _sz, _d, _f = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_double, ctypes.c_float


class GattnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {strerror(status)}")


def load():
    """Load libgattn.so; raises if it has not been built (there is no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"libgattn.so is not built ({LIB_PATH}); run `python -c \"import __graft_entry__ as g; g.build()\"`")
    lib = ctypes.CDLL(LIB_PATH)
    lib.gattn_strerror.restype = ctypes.c_char_p
    lib.gattn_strerror.argtypes = [_i]
    lib.gattn_prefill_workspace_size.restype = _sz
    lib.gattn_prefill_workspace_size.argtypes = [_i, _i, _i, _i, _i, _i]
    lib.gattn_prefill.restype = _i
    lib.gattn_prefill.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _d, _f, _i, _i64, _i64,
                                  _i64, _i64, _i, _vp, _sz, _vp, _vp]
    lib.gattn_decode_workspace_size.restype = _sz
    lib.gattn_prefill_varlen_workspace_size.restype = _sz
    lib.gattn_prefill_varlen_workspace_size.argtypes = [_i, _i, _i, _i, _i, _i]
    lib.gattn_prefill_varlen.restype = _i
    lib.gattn_prefill_varlen.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _d, _f, _i, _i64,
                                         _i64, _i64, _i64, _i, _vp, _sz, _vp, _vp]
    lib.gattn_decode_workspace_size.argtypes = [_i, _i, _i, _i, _i]
    lib.gattn_decode.restype = _i
    lib.gattn_decode.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _d, _f, _i, _vp, _sz, _vp, _vp]
    lib.gattn_decode_noalloc.restype = _i
    lib.gattn_decode_append.restype = _i
    lib.gattn_decode_append.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _d, _f, _i,
                                        _vp, _sz, _vp, _vp]
    lib.gattn_decode_paged.restype = _i
    lib.gattn_decode_paged.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _d,
                                       _f, _i, _vp, _sz, _vp, _vp]
    lib.gattn_decode_noalloc.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _d, _f, _i, _vp, _vp]
    lib.gattn_get_device_status.restype = _i
    lib.gattn_get_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint), _vp]
    lib.gattn_selftest_wait_timeout.restype = _i
    lib.gattn_selftest_wait_timeout.argtypes = [ctypes.c_ulonglong, _vp, _vp]
    lib.gattn_o_proj.restype = _i
    lib.gattn_o_proj.argtypes = [_vp, _vp, _i, _i, _i, _vp, _vp]
    lib.gattn_set_profile_events.restype = None
    lib.gattn_set_profile_events.argtypes = [_vp, _vp]
    _lib = lib
    return lib


def strerror(status: int) -> str:
    return load().gattn_strerror(int(status)).decode()


def check(status: int, where: str):
    if status != 0:
        raise GattnError(status, where)
