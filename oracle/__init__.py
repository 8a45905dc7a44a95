"""fp64 CPU oracle for paged GQA decode attention (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
may import this package. The library path never does, and the oracle imports
nothing from the library: the two share no code.

The arithmetic lives in ``ref_decode.cpp`` (plain loops, fp64, optional OpenMP
over (request, query head)); this module only builds it, loads it and marshals
numpy arrays. Every function's definition and its source passage are given in
the C++ file's header.

Parity pins (tests/test_oracle_pins.py) tie it to things other than itself:
torch's fp64 scaled_dot_product_attention and logsumexp on dense gathers, closed
forms (L = 1, q = 0, identical V rows, a hand-derived example under
tests/golden/), and invariants (slot permutation, split + LSE merge, GQA with
Hq = Hkv, equal queries in a group).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ref_decode.cpp")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the oracle with g++ (-O2, OpenMP). Returns the shared-object path."""
    if (not force and src == _SRC and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["g++", "-O2", "-std=c++17", "-fopenmp", "-fPIC", "-shared", src, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


class OracleLib:
    """The oracle's entry points, bound to one compiled shared object."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        lib.oracle_decode.argtypes = [P, P, P, P, P, I64, I64, I64, I64, I64,
                                      ctypes.c_float, P, P, ctypes.c_int]
        lib.oracle_decode.restype = ctypes.c_int
        lib.oracle_prefill.argtypes = [P, P, P, P, P, P, I64, I64, I64, I64, I64,
                                       ctypes.c_float, P, P, ctypes.c_int]
        lib.oracle_prefill.restype = ctypes.c_int
        lib.oracle_append.argtypes = [P, P, P, I64, I64, I64]
        lib.oracle_append.restype = ctypes.c_int
        lib.oracle_lse_merge.argtypes = [P, P, I64, I64, I64, P, P]
        lib.oracle_lse_merge.restype = ctypes.c_int
        lib.oracle_max_threads.restype = ctypes.c_int
        self.lib = lib
        self.path = path

    def max_threads(self) -> int:
        return int(self.lib.oracle_max_threads())

    def decode(self, q_bits, k_pool_bits, v_pool_bits, kv_indptr, kv_indices, n_qo_heads,
               n_kv_heads, head_dim, sm_scale, n_threads: int = 0):
        """Decode attention in fp64.

        q_bits: [B, Hq, D] uint16 bf16 patterns; k/v_pool_bits: [S, Hkv, D] uint16;
        kv_indptr: [B+1] int32; kv_indices: int32. ``sm_scale`` is taken as a
        float32 and widened. Returns (out [B, Hq, D] float64, lse [B, Hq] float64).
        """
        q = _c(q_bits, np.uint16)
        k = _c(k_pool_bits, np.uint16)
        v = _c(v_pool_bits, np.uint16)
        indptr = _c(kv_indptr, np.int32)
        indices = _c(kv_indices, np.int32)
        B = indptr.size - 1
        S = k.size // (n_kv_heads * head_dim)
        assert q.size == B * n_qo_heads * head_dim and v.size == k.size
        if indices.size == 0:
            indices = np.zeros(1, np.int32)
        out = np.empty((B, n_qo_heads, head_dim), np.float64)
        lse = np.empty((B, n_qo_heads), np.float64)
        rc = self.lib.oracle_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(indptr), _ptr(indices),
                                    B, n_qo_heads, n_kv_heads, head_dim, S,
                                    float(np.float32(sm_scale)), _ptr(out), _ptr(lse),
                                    int(n_threads))
        if rc != 0:
            raise ValueError("oracle_decode: bad arguments")
        return out, lse

    def prefill(self, q_bits, k_pool_bits, v_pool_bits, qo_indptr, kv_indptr, kv_indices,
                n_qo_heads, n_kv_heads, head_dim, sm_scale, n_threads: int = 0):
        """Causal chunked-prefill attention in fp64.

        q_bits: [NQ, Hq, D] uint16 (NQ = qo_indptr[-1]); request b's chunk is rows
        qo_indptr[b] .. qo_indptr[b+1], its newest C_b tokens, at list positions
        L_b - C_b .. L_b - 1. Returns (out [NQ, Hq, D] float64, lse [NQ, Hq] float64).
        """
        q = _c(q_bits, np.uint16)
        k = _c(k_pool_bits, np.uint16)
        v = _c(v_pool_bits, np.uint16)
        qo = _c(qo_indptr, np.int32)
        indptr = _c(kv_indptr, np.int32)
        indices = _c(kv_indices, np.int32)
        B = indptr.size - 1
        assert qo.size == B + 1
        NQ = int(qo[-1]) if B >= 0 and qo.size else 0
        S = k.size // (n_kv_heads * head_dim)
        assert q.size == NQ * n_qo_heads * head_dim and v.size == k.size
        if indices.size == 0:
            indices = np.zeros(1, np.int32)
        out = np.empty((NQ, n_qo_heads, head_dim), np.float64)
        lse = np.empty((NQ, n_qo_heads), np.float64)
        rc = self.lib.oracle_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(qo), _ptr(indptr),
                                     _ptr(indices), B, n_qo_heads, n_kv_heads, head_dim, S,
                                     float(np.float32(sm_scale)), _ptr(out), _ptr(lse),
                                     int(n_threads))
        if rc != 0:
            raise ValueError("oracle_prefill: bad arguments")
        return out, lse

    def append(self, pool_bits, slot_ids, rows_bits):
        """Row append on a copy of the pool: pool[slot_ids[i]] = rows[i]. Returns the copy."""
        pool = np.array(pool_bits, dtype=np.uint16, copy=True, order="C")
        ids = _c(slot_ids, np.int32).reshape(-1)
        rows = _c(rows_bits, np.uint16)
        n = ids.size
        if n == 0:
            return pool
        row_elems = rows.size // n
        S = pool.size // row_elems
        rc = self.lib.oracle_append(_ptr(pool), _ptr(ids), _ptr(rows), n, row_elems, S)
        if rc != 0:
            raise ValueError("oracle_append: slot out of range")
        return pool

    def lse_merge(self, outs, lses):
        """Merge attention results over disjoint parts of the same contexts.

        outs: [n_parts, R, D] float64, lses: [n_parts, R] float64 -> (out [R, D], lse [R]).
        """
        outs = _c(outs, np.float64)
        lses = _c(lses, np.float64)
        n_parts, R, D = outs.shape
        out = np.empty((R, D), np.float64)
        lse = np.empty(R, np.float64)
        self.lib.oracle_lse_merge(_ptr(outs), _ptr(lses), n_parts, R, D, _ptr(out), _ptr(lse))
        return out, lse


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def default() -> OracleLib:
    """The oracle built from ref_decode.cpp (compiled on first use)."""
    global _lib
    with _lock:
        if _lib is None:
            _lib = OracleLib(build())
    return _lib


def max_threads() -> int:
    return default().max_threads()


def decode(*args, **kwargs):
    return default().decode(*args, **kwargs)


def prefill(*args, **kwargs):
    return default().prefill(*args, **kwargs)


def append(*args, **kwargs):
    return default().append(*args, **kwargs)


def lse_merge(*args, **kwargs):
    return default().lse_merge(*args, **kwargs)
