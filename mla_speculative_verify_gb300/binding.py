"""ctypes binding of libmla_verify_sm103.so: the C entry points under the same names.

Argument marshalling only: every step of the decode runs in the library's
kernels. PyTorch is used for device memory and streams. If the library is
missing the import of this module's loader fails loudly; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

from . import build as _build

MLA_OK = 0
MLA_ERR_INVALID_ARG = -1
MLA_ERR_UNSUPPORTED = -2
MLA_ERR_BUFFER = -3
MLA_ERR_CUDA = -4
MLA_ERR_PLAN = -5
MLA_KV_BF16 = 0
MLA_KV_FP8_E4M3 = 1
MLA_DEVICE_WAIT_TIMEOUT = 0x1
MLA_DEVICE_PLAN_MISMATCH = 0x2
MLA_DEVICE_BAD_PAGE = 0x4
MLA_STATIC_WORKSPACE_BYTES = 16 << 20

_P = ctypes.c_void_p
_I32P = ctypes.POINTER(ctypes.c_int32)
_SZP = ctypes.POINTER(ctypes.c_size_t)
_IP = ctypes.POINTER(ctypes.c_int)


class PlanOptions(ctypes.Structure):
    _fields_ = [("force_splits", ctypes.c_int), ("max_rows_per_cta", ctypes.c_int),
                ("min_pages_per_split", ctypes.c_int), ("force_fold", ctypes.c_int),
                ("unit_pages", ctypes.c_int), ("cta_pair", ctypes.c_int), ("pair_slots", ctypes.c_int),
                ("debug_skip_copy", ctypes.c_int)]


class MlaError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{msg} (status {code})")
        self.code = code


# name -> (restype, argtypes); the same names and order as include/mla_decode.h
SIGNATURES = {
    "mla_decode_plan": (ctypes.c_int, [_I32P, _I32P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_int, _P, ctypes.c_size_t, _SZP, _SZP]),
    "mla_decode_plan_ex": (ctypes.c_int, [_I32P, _I32P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_int, ctypes.POINTER(PlanOptions), _P, ctypes.c_size_t, _SZP,
                                          _SZP]),
    "mla_decode_plan_info": (ctypes.c_int, [_P, ctypes.c_size_t, _IP, _IP, _IP, _IP, _IP]),
    "mla_decode_run": (ctypes.c_int, [_P, _P, ctypes.c_size_t, _P, _P, _P, ctypes.c_int, ctypes.c_int, _P, _P,
                                      ctypes.c_float, ctypes.c_float, _P, _P, _P, ctypes.c_size_t, _P, _P]),
    "mla_decode_run_static_ws": (ctypes.c_int, [_P, _P, ctypes.c_size_t, _P, _P, _P, ctypes.c_int, ctypes.c_int, _P,
                                                 _P, ctypes.c_float, ctypes.c_float, _P, _P, _P, _P]),
    "mla_device_pair_slots": (ctypes.c_int, [ctypes.c_int, _IP]),
    "mla_last_error": (ctypes.c_char_p, []),
    "mla_version": (ctypes.c_int, []),
}

_lib = None
_lock = threading.Lock()


def library_path() -> str:
    return _build.LIB_PATH


def load(path: str | None = None, build_if_missing: bool = True):
    """Load the library (building it first if needed) and declare the signatures."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or _build.LIB_PATH
        if build_if_missing and path is None:
            _build.build()
        if not os.path.exists(p):
            raise ImportError(f"the sm_103a library {p} is missing; run __graft_entry__.build()")
        lib = ctypes.CDLL(p)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        if path is None:
            _lib = lib
        return lib


def last_error(lib=None) -> str:
    lib = lib or load()
    return lib.mla_last_error().decode()


def check(code: int, lib=None) -> None:
    if code != MLA_OK:
        raise MlaError(code, last_error(lib))


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def plan(seq_lens, q_lens, num_heads: int, kv_dtype: int, num_sms: int, options: PlanOptions | None = None,
         page_size: int = 64):
    """mla_decode_plan(_ex): returns (plan bytes as a uint8 numpy array, workspace bytes)."""
    lib = load()
    s, q = _i32(seq_lens), _i32(q_lens)
    nbytes, ws = ctypes.c_size_t(0), ctypes.c_size_t(0)
    args = (s.ctypes.data_as(_I32P), q.ctypes.data_as(_I32P), int(s.shape[0]), int(num_heads), int(page_size),
            int(kv_dtype), int(num_sms))
    opt = ctypes.byref(options) if options is not None else None
    rc = lib.mla_decode_plan_ex(*args, opt, None, 0, ctypes.byref(nbytes), ctypes.byref(ws))
    if rc != MLA_ERR_BUFFER:
        check(rc, lib)
    buf = np.zeros(nbytes.value, dtype=np.uint8)
    rc = lib.mla_decode_plan_ex(*args, opt, buf.ctypes.data_as(_P), buf.nbytes, ctypes.byref(nbytes),
                                ctypes.byref(ws))
    check(rc, lib)
    return buf, int(ws.value)


_pair_slots = {}


def device_pair_slots(device: int) -> int:
    """mla_device_pair_slots: clusters of two CTAs the device runs at once (cached)."""
    if device not in _pair_slots:
        lib = load()
        n = ctypes.c_int(0)
        check(lib.mla_device_pair_slots(int(device), ctypes.byref(n)), lib)
        _pair_slots[device] = int(n.value)
    return _pair_slots[device]


def plan_info(plan_bytes: np.ndarray) -> dict:
    lib = load()
    vals = [ctypes.c_int(0) for _ in range(5)]
    check(lib.mla_decode_plan_info(plan_bytes.ctypes.data_as(_P), plan_bytes.nbytes, *[ctypes.byref(v) for v in vals]),
          lib)
    return dict(zip(["n_units", "n_merge", "total_q", "num_heads", "kv_dtype"], [v.value for v in vals]))


def run(plan_dev_ptr: int, plan_host: np.ndarray, q_ptr: int, kv_ptr: int, page_table_ptr: int, page_table_stride: int,
        num_pages: int, seq_lens_ptr: int, q_lens_ptr: int, sm_scale: float, kv_scale: float, out_ptr: int,
        lse_ptr: int | None, workspace_ptr: int | None, workspace_bytes: int, status_ptr: int | None,
        stream_handle: int) -> None:
    """mla_decode_run with raw device pointers (ints) and a cudaStream_t handle."""
    lib = load()
    rc = lib.mla_decode_run(plan_dev_ptr, plan_host.ctypes.data_as(_P), plan_host.nbytes, q_ptr, kv_ptr,
                            page_table_ptr, int(page_table_stride), int(num_pages), seq_lens_ptr, q_lens_ptr,
                            float(sm_scale), float(kv_scale), out_ptr, lse_ptr, workspace_ptr, int(workspace_bytes),
                            status_ptr, stream_handle)
    check(rc, lib)


def run_static_ws(plan_dev_ptr: int, plan_host: np.ndarray, q_ptr: int, kv_ptr: int, page_table_ptr: int,
                  page_table_stride: int, num_pages: int, seq_lens_ptr: int, q_lens_ptr: int, sm_scale: float,
                  kv_scale: float, out_ptr: int, lse_ptr: int | None, status_ptr: int | None,
                  stream_handle: int) -> None:
    """mla_decode_run_static_ws: the decode with the library's own split-KV scratch."""
    lib = load()
    rc = lib.mla_decode_run_static_ws(plan_dev_ptr, plan_host.ctypes.data_as(_P), plan_host.nbytes, q_ptr, kv_ptr,
                                      page_table_ptr, int(page_table_stride), int(num_pages), seq_lens_ptr,
                                      q_lens_ptr, float(sm_scale), float(kv_scale), out_ptr, lse_ptr, status_ptr,
                                      stream_handle)
    check(rc, lib)


def declared_functions(header: str | None = None) -> list[str]:
    """Names of the functions include/mla_decode.h declares (for the export test)."""
    import re

    header = header or os.path.join(_build.INCLUDE, "mla_decode.h")
    text = open(header).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(mla_\w+)\s*\(", text, flags=re.M)))
