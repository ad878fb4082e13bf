"""ctypes front end of ``mla_oracle.c`` (float64 MLA verify-decode oracle).

TEST INFRASTRUCTURE ONLY (see the package docstring). The arithmetic lives in
``mla_oracle.c``; this file only compiles it with gcc and marshals numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

MODE_DIRECT, MODE_FOLDED, MODE_SPLIT = 0, 1, 2
KV_BF16, KV_FP8_E4M3 = 0, 1
D_QK, D_V = 576, 512

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mla_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libmla_oracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/libmla_oracle.so`` (gcc, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(path: str):
    """Load a compiled oracle library and declare its signatures."""
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    lib.mla_oracle_decode.restype = ctypes.c_int
    lib.mla_oracle_decode.argtypes = [
        P, P, ctypes.c_int, ctypes.c_double, P, ctypes.c_int, ctypes.c_int, P, P,
        ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int, P, P, P, P, ctypes.c_int,
    ]
    lib.mla_oracle_e4m3_to_double.restype = ctypes.c_double
    lib.mla_oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
    lib.mla_oracle_fold_factor.restype = ctypes.c_int
    lib.mla_oracle_fold_factor.argtypes = [ctypes.c_int, ctypes.c_int]
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(build())
    return _lib


def load_variant(path: str):
    """Bind a separately compiled copy of the oracle (used by the tests that plant
    a mistake in a copy of the oracle source to show that the pins catch it)."""
    return _bind(path)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def e4m3_to_double(code: int) -> float:
    """Value of one OCP FP8 E4M3 byte, decoded from its bit fields."""
    return _load().mla_oracle_e4m3_to_double(int(code) & 0xFF)


def fold_factor(q: int, H: int) -> int:
    """Largest divisor F of q with H*F <= 128."""
    return _load().mla_oracle_fold_factor(int(q), int(H))


def decode(q_bits, kv_bits, kv_dtype, kv_scale, page_table, page_size, seq_lens, q_lens, H,
           sm_scale, mode=MODE_DIRECT, split_bounds=None, nthreads=None, lib=None):
    """Run the oracle.

    q_bits: uint16 array [total_q, H, 576] holding bf16 bit patterns.
    kv_bits: uint16 [rows, 576] (bf16 bits) or uint8 [rows, 576] (e4m3 codes).
    page_table: int32 [B, stride]; seq_lens, q_lens: int32 [B].
    split_bounds (MODE_SPLIT): list of B increasing int sequences, each from 0 to ctx_b.
    Returns (out float64 [total_q, H, 512], lse float64 [total_q, H]).
    """
    lib = lib if lib is not None else _load()
    q_bits = np.ascontiguousarray(q_bits, dtype=np.uint16)
    kv_bits = np.ascontiguousarray(kv_bits, dtype=np.uint16 if kv_dtype == KV_BF16 else np.uint8)
    page_table = np.ascontiguousarray(page_table, dtype=np.int32)
    seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    q_lens = np.ascontiguousarray(q_lens, dtype=np.int32)
    B = int(seq_lens.shape[0])
    total_q = int(q_lens.sum())
    assert q_bits.shape == (total_q, H, D_QK), q_bits.shape
    assert kv_bits.ndim == 2 and kv_bits.shape[1] == D_QK
    assert page_table.ndim == 2 and page_table.shape[0] == B
    out = np.zeros((total_q, H, D_V), dtype=np.float64)
    lse = np.zeros((total_q, H), dtype=np.float64)
    sb = so = None
    if mode == MODE_SPLIT:
        assert split_bounds is not None and len(split_bounds) == B
        flat, offs = [], [0]
        for seq in split_bounds:
            flat.extend(int(x) for x in seq)
            offs.append(len(flat))
        sb = np.asarray(flat, dtype=np.int32)
        so = np.asarray(offs, dtype=np.int32)
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    rc = lib.mla_oracle_decode(
        _ptr(q_bits), _ptr(kv_bits), int(kv_dtype), float(kv_scale), _ptr(page_table),
        int(page_table.shape[1]), int(page_size), _ptr(seq_lens), _ptr(q_lens), B, int(H),
        float(sm_scale), int(mode), _ptr(sb) if sb is not None else None,
        _ptr(so) if so is not None else None, _ptr(out), _ptr(lse), int(nthreads))
    if rc != 0:
        raise ValueError(f"oracle rejected its arguments (code {rc})")
    return out, lse
