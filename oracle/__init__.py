"""CPU oracle for tree-verify attention (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU baseline /
reference arm use this package.  The product path never imports it.

``verify_attn_oracle.c`` holds the arithmetic (plain definition in double
precision, see its header).  This module compiles it with gcc and marshals
numpy arrays to it through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "verify_attn_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

ERRORS = {-1: "bad argument", -2: "slot id outside the pool", -3: "mask_indptr inconsistent",
          -4: "row outside the batch", -5: "out of memory"}


def build(force: bool = False) -> str:
    """Compile liboracle.so next to its source (OpenMP when gcc supports it)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", _LIB + ".tmp", _SRC, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            path = os.environ.get("ORACLE_LIB")  # tests load planted-mistake builds this way
            if not path:
                path = build()
            lib = ctypes.CDLL(path)
            p = ctypes.c_void_p
            i64 = ctypes.c_int64
            lib.oracle_verify_attn.argtypes = [p, i64, i64, p, i64, p, p, p, p, p, p,
                                               ctypes.c_double, ctypes.c_int, ctypes.c_int,
                                               p, i64, ctypes.c_int, p, p]
            lib.oracle_verify_attn.restype = ctypes.c_int
            lib.oracle_num_threads.restype = ctypes.c_int
            if hasattr(lib, "oracle_set_num_threads"):
                lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
            _lib = lib
    return _lib


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    """Thread count for later calls (for timing; the results do not depend on it)."""
    _load().oracle_set_num_threads(int(n))


def _bits16(x) -> np.ndarray:
    """bf16 tensor / uint16 array -> contiguous numpy uint16 bit patterns."""
    if hasattr(x, "detach"):
        import torch
        x = x.detach().to("cpu").contiguous().view(torch.int16).numpy()
    return np.ascontiguousarray(x).view(np.uint16)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p) if a.size else ctypes.c_void_p(0)


def verify_attn(q, kv_pool, qo_indptr, kv_indptr, kv_indices, out_cache_loc, custom_mask,
                mask_indptr, sm_scale, num_heads, rows=None, num_splits=0):
    """Oracle output rows.

    q: [total_q, H, 576] bf16 (tensor or uint16 bits); kv_pool: [pool, 576].
    rows: None for every row (row = t*H + h) or an int64 list of row ids.
    Returns (out float64 [n, 512], lse float64 [n]).
    """
    lib = _load()
    qb = _bits16(q).reshape(-1, num_heads, 576)
    pool = _bits16(kv_pool).reshape(-1, 576)
    qo = np.ascontiguousarray(qo_indptr, dtype=np.int32)
    kvp = np.ascontiguousarray(kv_indptr, dtype=np.int32)
    kvi = np.ascontiguousarray(kv_indices, dtype=np.int32)
    ocl = np.ascontiguousarray(out_cache_loc, dtype=np.int64)
    msk = np.ascontiguousarray(custom_mask, dtype=np.uint8)
    mip = np.ascontiguousarray(mask_indptr, dtype=np.int64)
    batch = len(qo) - 1
    if rows is None:
        n = int(qo[-1]) * num_heads
        rows_arr = None
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        n = rows_arr.size
    out = np.zeros((n, 512), dtype=np.float64)
    lse = np.zeros(n, dtype=np.float64)
    if msk.size == 0:
        msk = np.zeros(1, dtype=np.uint8)
    rc = lib.oracle_verify_attn(_ptr(qb), qb.shape[1] * 576, 576, _ptr(pool), pool.shape[0],
                                _ptr(qo), _ptr(kvp), _ptr(kvi), _ptr(ocl), _ptr(msk), _ptr(mip),
                                float(sm_scale), batch, int(num_heads),
                                _ptr(rows_arr) if rows_arr is not None else ctypes.c_void_p(0),
                                n, int(num_splits), _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError(f"oracle: {ERRORS.get(rc, rc)}")
    return out, lse


def run(inp, rows=None, num_splits=0):
    """Oracle on a ``VerifyInputs``-like object (attributes as in workloads)."""
    return verify_attn(inp.q, inp.kv_pool, inp.qo_indptr, inp.kv_indptr, inp.kv_indices,
                       inp.out_cache_loc, inp.custom_mask, inp.mask_indptr, inp.sm_scale,
                       inp.num_heads, rows=rows, num_splits=num_splits)


def save_kv(kv_pool_bits: np.ndarray, out_cache_loc: np.ndarray, kv_new_bits: np.ndarray) -> np.ndarray:
    """The KV save step ("The Launch Wrapper", section The KV Cache Ordering
    Insight): a copy of the pool (bf16 bit patterns, [pool_size, 576] uint16)
    with row out_cache_loc[i] replaced by kv_new[i] for every i.  Slots must
    be distinct and inside the pool (the definition has no other case)."""
    pool = np.array(kv_pool_bits, dtype=np.uint16, copy=True)
    loc = np.asarray(out_cache_loc, dtype=np.int64)
    if loc.size and (loc.min() < 0 or loc.max() >= pool.shape[0]):
        raise ValueError("slot outside the pool")
    if len(np.unique(loc)) != loc.size:
        raise ValueError("slots must be distinct")
    pool[loc] = np.asarray(kv_new_bits, dtype=np.uint16).reshape(loc.size, -1)
    return pool
