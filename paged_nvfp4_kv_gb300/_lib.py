"""ctypes view of libpnkv.so (the C ABI declared in include/pnkv.h).

Loading fails loudly when the library has not been built: there is no
fallback implementation of any call.
"""
import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libpnkv.so")

PNKV_OK = 0
PNKV_ERR_INVALID_ARG = -1
PNKV_ERR_UNSUPPORTED = -2
PNKV_ERR_CUDA = -3

PNKV_KV_BF16 = 0
PNKV_KV_NVFP4 = 1
PNKV_KV_FP8 = 2
PNKV_KV_INT8 = 3

DEV_ERR_BITS = {1: "page id", 2: "position", 4: "seq_len", 8: "qo_indptr", 16: "timeout",
                32: "seq index"}


class YarnParams(ctypes.Structure):
    _fields_ = [("theta", ctypes.c_double), ("factor", ctypes.c_double),
                ("original_max", ctypes.c_int64), ("beta_fast", ctypes.c_double),
                ("beta_slow", ctypes.c_double), ("rotary_dim", ctypes.c_int32),
                ("deployed_range", ctypes.c_int32)]


class CacheDesc(ctypes.Structure):
    _fields_ = [("pool", ctypes.c_void_p), ("num_pages", ctypes.c_int64),
                ("page_size", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("k_scale", ctypes.c_float), ("v_scale", ctypes.c_float)]


# (name, restype, argtypes) of every exported call, in header order.
_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_F = ctypes.c_float
SIGNATURES = [
    ("pnkv_page_bytes", ctypes.c_int, [ctypes.POINTER(CacheDesc), ctypes.POINTER(_I64)]),
    ("yarn_rope_tables", ctypes.c_int, [ctypes.POINTER(YarnParams), _I64, _P, _P, _P]),
    ("kv_append_nvfp4", ctypes.c_int,
     [ctypes.POINTER(CacheDesc), _P, _I64, _I32, _P, _P, _I64, _P, _P, _I32, _P, _P, _P, _P, _I64,
      _I32, _P, _P]),
    ("pnkv_decode_slots", _I64, [ctypes.POINTER(CacheDesc), _I32, _I32, _I32]),
    ("pnkv_work_meta_ints", _I64, [_I32, _I32]),
    ("paged_decode_attention", ctypes.c_int,
     [ctypes.POINTER(CacheDesc), _P, _P, _P, _I64, _P, _I32, _I64, _I32, _I32, _F, _I32, _P, _P,
      _I64, _P, _P, _P]),
    ("paged_prefill_attention_fp4q", ctypes.c_int,
     [ctypes.POINTER(CacheDesc), _P, _P, _P, _I64, _P, _I32, _I64, _I32, _I32, _F, _I32, _F, _P,
      _P, _I64, _P, _P, _P]),
    ("split_kv_combine", ctypes.c_int,
     [_P, _P, _P, _P, _I32, _I64, _I32, _I32, _I32, _I32, _P, _I32, _P, _P]),
    ("paged_decode_attention_noalloc", ctypes.c_int,
     [ctypes.POINTER(CacheDesc), _P, _P, _P, _I64, _P, _I32, _I32, _I32, _F, _I32, _I64, _P, _I32,
      _P, _P, _P]),
    ("pnkv_set_wait_limit_ns", _I64, [_I64]),
    ("pnkv_status_string", ctypes.c_char_p, [ctypes.c_int]),
    ("pnkv_version", ctypes.c_int, []),
]

_lib = None


def load():
    """The loaded library (built beforehand by ``_build.build()``)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                "libpnkv.so is not built (%s); run paged_nvfp4_kv_gb300._build.build() or "
                "__graft_entry__.build() first" % LIB_PATH)
        lib = ctypes.CDLL(LIB_PATH)
        for name, res, args in SIGNATURES:
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def check(status, what):
    if status != PNKV_OK:
        text = load().pnkv_status_string(status).decode()
        raise RuntimeError("%s failed: %s (%d)" % (what, text, status))
