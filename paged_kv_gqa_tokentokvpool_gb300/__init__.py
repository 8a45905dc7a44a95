"""Paged GQA decode attention over a page-size-1 token KV pool, for GB300 (sm_103a).

A thin ctypes binding of the C ABI in ``include/pkv.h`` (``libpkv.so``, built
in-tree by ``build.py``). The functions keep the C names and argument order; they
only turn torch tensors into pointers and sizes and raise ``PkvError`` on a
negative return code. Every step of the computation runs in the library's CUDA
kernels: there is no Python or CPU fallback, and the first call raises
ImportError if the library has not been built.

Typical decode step (one plan per step, reused by every layer):

    plan = paged_decode_plan_create(max_batch, max_tokens, 32, 8, 128)
    paged_decode_plan(plan, kv_indptr_cpu)                 # once per step
    for layer in layers:
        kvpool_append(k_pool[l], v_pool[l], slot_ids, k_new[l], v_new[l])
        paged_decode_attn(q[l], k_pool[l], v_pool[l], kv_indptr, kv_indices,
                          batch, 32, 8, 128, sm_scale, out[l], lse[l], plan)
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpkv.so")

PKV_OK = 0
PKV_ERR_INVALID_ARG = -1
PKV_ERR_UNSUPPORTED = -2
PKV_ERR_PLAN = -3
PKV_ERR_CUDA = -4
PKV_ERR_INDEX = -5
PKV_PLAN_EARLY_GATHER = 1
PKV_PLAN_PERSISTENT = 2
PKV_PLAN_SINGLE_LAUNCH = 4

EXPORTED = ("kvpool_append", "paged_decode_plan_create", "paged_decode_plan",
            "paged_decode_attn", "paged_decode_plan_destroy", "paged_decode_plan_host",
            "paged_decode_plan_info", "paged_decode_plan_status", "paged_decode_attn_static",
            "paged_decode_append_attn", "paged_decode_plan_shared", "kvpool_offload",
            "kvpool_prefetch", "paged_decode_plan_set_flags", "paged_prefill_plan_create",
            "paged_prefill_plan", "paged_prefill_attn", "paged_prefill_plan_destroy",
            "paged_prefill_plan_host", "paged_prefill_plan_status",
            "paged_decode_plan_host_times", "paged_decode_attn_static_status",
            "paged_decode_attn_tiered", "paged_decode_plan_mode",
            "pkv_set_debug_checks", "pkv_inject_stall",
            "pkv_last_error")


class PkvError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"[{code}] {message}")
        self.code = code
        self.message = message


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it first (python -m "
            "paged_kv_gqa_tokentokvpool_gb300.build, or __graft_entry__.build()). "
            "This package has no CPU fallback.")
    lib = ctypes.CDLL(LIB_PATH)
    P, I32, I64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    lib.kvpool_append.argtypes = [P, P, P, P, P, I64, I32, I32, I64, P]
    lib.paged_decode_plan_create.argtypes = [ctypes.POINTER(P), I32, I64, I32, I32, I32]
    lib.paged_decode_plan.argtypes = [P, P, I32, P]
    lib.paged_decode_attn.argtypes = [P, P, P, P, P, I32, I32, I32, I32, ctypes.c_float, P, P,
                                      P, P]
    lib.paged_decode_plan_destroy.argtypes = [P]
    lib.paged_decode_plan_destroy.restype = None
    lib.paged_decode_plan_host.argtypes = [P, I32, I32, I32, I32, I32, P, I32, P, I32, P, I32, P,
                                           P, I32, P, I32, P]
    lib.paged_decode_plan_shared.argtypes = [P, P, I32, P, I32, P, P]
    lib.kvpool_offload.argtypes = [P, P, P, P, P, P, I64, I32, I32, I64, I64, P]
    lib.kvpool_prefetch.argtypes = [P, P, P, P, P, P, I64, I32, I32, I64, I64, P]
    lib.paged_decode_plan_info.argtypes = [P, P, P, P, P, P]
    lib.paged_decode_plan_status.argtypes = [P, P]
    lib.paged_decode_plan_set_flags.argtypes = [P, ctypes.c_uint]
    lib.paged_decode_plan_host_times.argtypes = [P, P, P, P, I32]
    lib.paged_decode_attn_static_status.argtypes = [P, P]
    lib.paged_decode_plan_mode.argtypes = [P, P]
    lib.paged_decode_attn_tiered.argtypes = [P, P, P, I64, P, P, I64, P, P, I32, I32, I32, I32,
                                             ctypes.c_float, P, P, P, P]
    lib.paged_prefill_plan_create.argtypes = [ctypes.POINTER(P), I32, I64, I32, I32, I32]
    lib.paged_prefill_plan.argtypes = [P, P, P, I32, P]
    lib.paged_prefill_attn.argtypes = [P, P, P, P, P, P, I32, I32, I32, I32, ctypes.c_float,
                                       P, P, P, P]
    lib.paged_prefill_plan_host.argtypes = [P, P, I32, I32, I32, I32, I32, P, I32, P, I32, P]
    lib.paged_prefill_plan_status.argtypes = [P, P]
    lib.paged_prefill_plan_destroy.argtypes = [P]
    lib.paged_prefill_plan_destroy.restype = None
    lib.paged_decode_attn_static.argtypes = [P, P, P, P, P, P, I32, I32, I32, I32,
                                             ctypes.c_float, P, P, P]
    lib.paged_decode_append_attn.argtypes = [P, P, P, P, P, P, P, P, I32, I32, I32, I32, I64,
                                             ctypes.c_float, P, P, P, P]
    lib.pkv_set_debug_checks.argtypes = [I32]
    lib.pkv_set_debug_checks.restype = None
    lib.pkv_inject_stall.argtypes = [I32]
    lib.pkv_inject_stall.restype = None
    lib.pkv_last_error.argtypes = []
    lib.pkv_last_error.restype = ctypes.c_char_p
    for name in ("kvpool_append", "paged_decode_plan_create", "paged_decode_plan",
                 "paged_decode_attn", "paged_decode_plan_host", "paged_decode_plan_info",
                 "paged_decode_plan_status", "paged_decode_attn_static",
                 "paged_decode_append_attn", "paged_decode_plan_shared", "kvpool_offload",
                 "kvpool_prefetch", "paged_decode_plan_set_flags", "paged_prefill_plan_create",
                 "paged_prefill_plan", "paged_prefill_attn", "paged_prefill_plan_host",
                 "paged_prefill_plan_status", "paged_decode_plan_host_times",
                 "paged_decode_attn_static_status", "paged_decode_attn_tiered",
                 "paged_decode_plan_mode"):
        getattr(lib, name).restype = ctypes.c_int
    return lib


_lib = None


def library() -> ctypes.CDLL:
    """The loaded libpkv.so (loaded on first use; ImportError if it was not built)."""
    global _lib
    if _lib is None:
        _lib = _load()
    return _lib


def pkv_last_error() -> str:
    return library().pkv_last_error().decode()


def pkv_set_debug_checks(on: bool) -> None:
    library().pkv_set_debug_checks(1 if on else 0)


def pkv_inject_stall(n_launches: int) -> None:
    """The next n attention launches withhold their copies: their bounded waits
    expire and the plan's status word is set (failure-detection tests)."""
    library().pkv_inject_stall(int(n_launches))


def _check(rc: int) -> None:
    if rc != PKV_OK:
        raise PkvError(rc, pkv_last_error())


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, torch.Tensor):
        return ctypes.c_void_p(t.data_ptr())
    if isinstance(t, np.ndarray):
        return t.ctypes.data_as(ctypes.c_void_p)
    return ctypes.c_void_p(int(t))


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _dev(t: torch.Tensor, dtype, name: str):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


class Plan:
    """Owns a ``pkv_plan*``; freed by ``paged_decode_plan_destroy`` or on collection."""

    def __init__(self, handle: ctypes.c_void_p, shape):
        self.handle = handle
        self.shape = shape

    def info(self) -> dict:
        vals = [ctypes.c_int() for _ in range(5)]
        _check(library().paged_decode_plan_info(self.handle, *[ctypes.byref(v) for v in vals]))
        return dict(zip(("batch", "n_units", "n_merges", "chunk_tokens", "n_ctas"),
                        (v.value for v in vals)))

    def status(self) -> int:
        """Read and clear the device status word (0 = every pipeline wait completed)."""
        v = ctypes.c_int()
        _check(library().paged_decode_plan_status(self.handle, ctypes.byref(v)))
        return v.value

    def single_launch(self) -> bool:
        """True when the plan's steps run as single launches of the cluster kernel
        (paged_decode_plan_mode)."""
        v = ctypes.c_int()
        _check(library().paged_decode_plan_mode(self.handle, ctypes.byref(v)))
        return bool(v.value)

    def set_flags(self, flags: int) -> None:
        """paged_decode_plan_set_flags (e.g. PKV_PLAN_EARLY_GATHER)."""
        paged_decode_plan_set_flags(self, flags)

    def timing(self, reset: bool = False) -> dict:
        """Host time of the plan calls since the last reset (paged_decode_plan_host_times):
        per call on average, in the partition (compute_us) and waiting for a free
        staging buffer (wait_us)."""
        c, w, n = ctypes.c_double(), ctypes.c_double(), ctypes.c_int64()
        _check(library().paged_decode_plan_host_times(self.handle, ctypes.byref(c),
                                                      ctypes.byref(w), ctypes.byref(n),
                                                      1 if reset else 0))
        calls = max(n.value, 1)
        return {"compute_us": c.value / calls, "wait_us": w.value / calls, "calls": n.value}

    def reset_timing(self) -> None:
        self.timing(reset=True)

    def __del__(self):
        if getattr(self, "handle", None) and _lib is not None:
            _lib.paged_decode_plan_destroy(self.handle)
            self.handle = None


def kvpool_append(k_pool, v_pool, slot_ids, k_new, v_new, n=None, n_kv_heads=None,
                  head_dim=None, pool_slots=None, stream=None) -> None:
    """k_pool[slot_ids[i]] = k_new[i]; v_pool[slot_ids[i]] = v_new[i] (bit-exact)."""
    _dev(k_pool, torch.bfloat16, "k_pool")
    _dev(v_pool, torch.bfloat16, "v_pool")
    _dev(slot_ids, torch.int32, "slot_ids")
    _dev(k_new, torch.bfloat16, "k_new")
    _dev(v_new, torch.bfloat16, "v_new")
    S, hkv, d = k_pool.shape
    if v_pool.shape != k_pool.shape or k_new.shape != v_new.shape:
        raise ValueError("pool / new-row shapes disagree")
    n = slot_ids.numel() if n is None else n
    _check(library().kvpool_append(_ptr(k_pool), _ptr(v_pool), _ptr(slot_ids), _ptr(k_new),
                              _ptr(v_new), n, hkv if n_kv_heads is None else n_kv_heads,
                              d if head_dim is None else head_dim,
                              S if pool_slots is None else pool_slots, _stream(stream)))


def _host_pool(t, name):
    if not isinstance(t, torch.Tensor) or t.is_cuda:
        raise TypeError(f"{name} must be a (pinned) CPU tensor")
    if t.dtype != torch.bfloat16 or not t.is_contiguous():
        raise TypeError(f"{name} must be a contiguous bf16 tensor")
    return t


def kvpool_offload(k_pool, v_pool, dev_slots, k_host, v_host, host_slots, stream=None) -> None:
    """k_host[host_slots[i]] = k_pool[dev_slots[i]] (and V); host pools pinned."""
    _dev(k_pool, torch.bfloat16, "k_pool")
    _dev(v_pool, torch.bfloat16, "v_pool")
    _dev(dev_slots, torch.int32, "dev_slots")
    _dev(host_slots, torch.int32, "host_slots")
    _host_pool(k_host, "k_host")
    _host_pool(v_host, "v_host")
    S, hkv, d = k_pool.shape
    _check(library().kvpool_offload(_ptr(k_pool), _ptr(v_pool), _ptr(dev_slots), _ptr(k_host),
                                    _ptr(v_host), _ptr(host_slots), dev_slots.numel(), hkv, d, S,
                                    k_host.shape[0], _stream(stream)))


def kvpool_prefetch(k_pool, v_pool, dev_slots, k_host, v_host, host_slots, stream=None) -> None:
    """k_pool[dev_slots[i]] = k_host[host_slots[i]] (and V); host pools pinned."""
    _dev(k_pool, torch.bfloat16, "k_pool")
    _dev(v_pool, torch.bfloat16, "v_pool")
    _dev(dev_slots, torch.int32, "dev_slots")
    _dev(host_slots, torch.int32, "host_slots")
    _host_pool(k_host, "k_host")
    _host_pool(v_host, "v_host")
    S, hkv, d = k_pool.shape
    _check(library().kvpool_prefetch(_ptr(k_pool), _ptr(v_pool), _ptr(dev_slots), _ptr(k_host),
                                     _ptr(v_host), _ptr(host_slots), dev_slots.numel(), hkv, d, S,
                                     k_host.shape[0], _stream(stream)))


def paged_decode_plan_create(max_batch: int, max_tokens: int, n_qo_heads: int,
                             n_kv_heads: int, head_dim: int) -> Plan:
    h = ctypes.c_void_p()
    _check(library().paged_decode_plan_create(ctypes.byref(h), max_batch, max_tokens, n_qo_heads,
                                         n_kv_heads, head_dim))
    return Plan(h, (n_qo_heads, n_kv_heads, head_dim))


def _host_indptr(kv_indptr) -> np.ndarray:
    if isinstance(kv_indptr, torch.Tensor):
        if kv_indptr.is_cuda:
            raise TypeError("plans take HOST copies of the offset arrays")
        kv_indptr = kv_indptr.numpy()
    return np.ascontiguousarray(kv_indptr, dtype=np.int32)


def paged_decode_plan(plan: Plan, kv_indptr_host, batch=None, stream=None) -> None:
    ip = _host_indptr(kv_indptr_host)
    batch = ip.size - 1 if batch is None else batch
    plan._indptr_keepalive = ip
    _check(library().paged_decode_plan(plan.handle, _ptr(ip), batch, _stream(stream)))


def paged_decode_plan_shared(plan: Plan, kv_indptr_host, shared_indptr_host, shared_len_host,
                             batch=None, stream=None) -> None:
    """paged_decode_plan with sharing groups: requests [shared_indptr[s],
    shared_indptr[s+1]) list the same first shared_len[s] slots."""
    ip = _host_indptr(kv_indptr_host)
    sp = np.ascontiguousarray(shared_indptr_host, dtype=np.int32)
    sl = np.ascontiguousarray(shared_len_host, dtype=np.int32)
    batch = ip.size - 1 if batch is None else batch
    plan._indptr_keepalive = (ip, sp, sl)
    _check(library().paged_decode_plan_shared(plan.handle, _ptr(ip), batch, _ptr(sp),
                                              max(sp.size - 1, 0), _ptr(sl), _stream(stream)))


def paged_decode_attn(q, k_pool, v_pool, kv_indptr, kv_indices, batch, n_qo_heads,
                      n_kv_heads, head_dim, sm_scale, out, lse, plan: Plan,
                      stream=None) -> None:
    _dev(q, torch.bfloat16, "q")
    _dev(k_pool, torch.bfloat16, "k_pool")
    _dev(v_pool, torch.bfloat16, "v_pool")
    _dev(kv_indptr, torch.int32, "kv_indptr")
    _dev(kv_indices, torch.int32, "kv_indices")
    _dev(out, torch.bfloat16, "out")
    if lse is not None:
        _dev(lse, torch.float32, "lse")
    _check(library().paged_decode_attn(_ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(kv_indptr),
                                  _ptr(kv_indices), batch, n_qo_heads, n_kv_heads, head_dim,
                                  float(sm_scale), _ptr(out), _ptr(lse), plan.handle,
                                  _stream(stream)))


def paged_decode_attn_tiered(q, k_pool, v_pool, k_host, v_host, kv_indptr, kv_indices, batch,
                             n_qo_heads, n_kv_heads, head_dim, sm_scale, out, lse, plan: Plan,
                             stream=None) -> None:
    """paged_decode_attn where a slot id s < 0 names row -1 - s of the pinned host pools
    k_host / v_host, read in place over the host link (see include/pkv.h)."""
    for t, name in ((q, "q"), (k_pool, "k_pool"), (v_pool, "v_pool"), (out, "out")):
        _dev(t, torch.bfloat16, name)
    for t, name in ((kv_indptr, "kv_indptr"), (kv_indices, "kv_indices")):
        _dev(t, torch.int32, name)
    _host_pool(k_host, "k_host")
    _host_pool(v_host, "v_host")
    if lse is not None:
        _dev(lse, torch.float32, "lse")
    _check(library().paged_decode_attn_tiered(
        _ptr(q), _ptr(k_pool), _ptr(v_pool), k_pool.shape[0], _ptr(k_host), _ptr(v_host),
        k_host.shape[0], _ptr(kv_indptr), _ptr(kv_indices), batch, n_qo_heads, n_kv_heads,
        head_dim, float(sm_scale), _ptr(out), _ptr(lse), plan.handle, _stream(stream)))


def paged_decode_append_attn(q, k_pool, v_pool, kv_indptr, kv_indices, slot_ids, k_new, v_new,
                             batch, n_qo_heads, n_kv_heads, head_dim, sm_scale, out, lse,
                             plan: Plan, stream=None) -> None:
    """kvpool_append + paged_decode_attn in one launch; slot_ids[b] must be request
    b's last listed slot (see include/pkv.h)."""
    for t, name in ((q, "q"), (k_pool, "k_pool"), (v_pool, "v_pool"), (k_new, "k_new"),
                    (v_new, "v_new"), (out, "out")):
        _dev(t, torch.bfloat16, name)
    for t, name in ((kv_indptr, "kv_indptr"), (kv_indices, "kv_indices"), (slot_ids, "slot_ids")):
        _dev(t, torch.int32, name)
    if lse is not None:
        _dev(lse, torch.float32, "lse")
    _check(library().paged_decode_append_attn(
        _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(kv_indptr), _ptr(kv_indices), _ptr(slot_ids),
        _ptr(k_new), _ptr(v_new), batch, n_qo_heads, n_kv_heads, head_dim, k_pool.shape[0],
        float(sm_scale), _ptr(out), _ptr(lse), plan.handle, _stream(stream)))


def paged_decode_attn_static(q, k_pool, v_pool, kv_indptr_host, kv_indptr, kv_indices,
                             batch=None, n_qo_heads=None, n_kv_heads=None, head_dim=None,
                             sm_scale=None, out=None, lse=None, stream=None) -> None:
    """paged_decode_attn without a plan and without any device allocation: the
    step is planned on every call and all scratch lives in the library's static
    32 MiB device array (see include/pkv.h for the sharing rules). batch defaults
    to the host offsets' length - 1 and may not exceed it."""
    _dev(q, torch.bfloat16, "q")
    _dev(k_pool, torch.bfloat16, "k_pool")
    _dev(v_pool, torch.bfloat16, "v_pool")
    _dev(kv_indptr, torch.int32, "kv_indptr")
    _dev(kv_indices, torch.int32, "kv_indices")
    _dev(out, torch.bfloat16, "out")
    if lse is not None:
        _dev(lse, torch.float32, "lse")
    ip = _host_indptr(kv_indptr_host)
    batch = ip.size - 1 if batch is None else int(batch)
    if batch < 0 or ip.size < batch + 1:
        raise ValueError(f"kv_indptr_host has {ip.size} entries; batch {batch} needs {batch + 1}")
    if kv_indptr.numel() < batch + 1:
        raise ValueError(f"kv_indptr has {kv_indptr.numel()} entries; batch {batch} needs {batch + 1}")
    S, hkv, d = k_pool.shape
    n_kv_heads = hkv if n_kv_heads is None else n_kv_heads
    head_dim = d if head_dim is None else head_dim
    n_qo_heads = q.shape[1] if n_qo_heads is None else n_qo_heads
    # ip (the host offsets) is referenced until the call returns
    _check(library().paged_decode_attn_static(
        _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(ip), _ptr(kv_indptr), _ptr(kv_indices), batch,
        n_qo_heads, n_kv_heads, head_dim, float(sm_scale), _ptr(out), _ptr(lse),
        _stream(stream)))


def paged_decode_attn_static_status(stream=None) -> int:
    """Wait for the stream, then read and clear the status word of the static entry
    point's array on the current device (0 = every pipeline wait completed)."""
    v = ctypes.c_int()
    _check(library().paged_decode_attn_static_status(_stream(stream), ctypes.byref(v)))
    return v.value


def paged_decode_plan_set_flags(plan: Plan, flags: int) -> None:
    """Options of the attention calls that use the plan (PKV_PLAN_* bits)."""
    _check(library().paged_decode_plan_set_flags(plan.handle if plan is not None else None,
                                                 int(flags)))


class PrefillPlan:
    """Owns a ``pkv_prefill_plan*``; freed by ``paged_prefill_plan_destroy`` or on collection."""

    def __init__(self, handle: ctypes.c_void_p, shape):
        self.handle = handle
        self.shape = shape

    def status(self) -> int:
        """Read and clear the device status word (0 = every pipeline wait completed)."""
        v = ctypes.c_int()
        _check(library().paged_prefill_plan_status(self.handle, ctypes.byref(v)))
        return v.value

    def __del__(self):
        if getattr(self, "handle", None) and _lib is not None:
            _lib.paged_prefill_plan_destroy(self.handle)
            self.handle = None


def paged_prefill_plan_create(max_batch: int, max_q_tokens: int, n_qo_heads: int,
                              n_kv_heads: int, head_dim: int) -> PrefillPlan:
    h = ctypes.c_void_p()
    _check(library().paged_prefill_plan_create(ctypes.byref(h), max_batch, max_q_tokens,
                                               n_qo_heads, n_kv_heads, head_dim))
    return PrefillPlan(h, (n_qo_heads, n_kv_heads, head_dim))


def paged_prefill_plan(plan: PrefillPlan, qo_indptr_host, kv_indptr_host, batch=None,
                       stream=None) -> None:
    """The step's prefill work list from HOST copies of the chunk and slot-list offsets."""
    qo = _host_indptr(qo_indptr_host)
    kv = _host_indptr(kv_indptr_host)
    batch = kv.size - 1 if batch is None else batch
    plan._indptr_keepalive = (qo, kv)
    _check(library().paged_prefill_plan(plan.handle, _ptr(qo), _ptr(kv), batch,
                                        _stream(stream)))


def paged_prefill_attn(q, k_pool, v_pool, qo_indptr, kv_indptr, kv_indices, batch, n_qo_heads,
                       n_kv_heads, head_dim, sm_scale, out, lse, plan: PrefillPlan,
                       stream=None) -> None:
    """Causal attention of the planned chunks: q/out [qo_indptr[batch], Hq, D] bf16."""
    for t, name in ((q, "q"), (k_pool, "k_pool"), (v_pool, "v_pool"), (out, "out")):
        _dev(t, torch.bfloat16, name)
    for t, name in ((qo_indptr, "qo_indptr"), (kv_indptr, "kv_indptr"),
                    (kv_indices, "kv_indices")):
        _dev(t, torch.int32, name)
    if lse is not None:
        _dev(lse, torch.float32, "lse")
    _check(library().paged_prefill_attn(
        _ptr(q), _ptr(k_pool), _ptr(v_pool), _ptr(qo_indptr), _ptr(kv_indptr), _ptr(kv_indices),
        batch, n_qo_heads, n_kv_heads, head_dim, float(sm_scale), _ptr(out), _ptr(lse),
        plan.handle, _stream(stream)))


def paged_prefill_plan_host(qo_indptr_host, kv_indptr_host, n_qo_heads: int, n_kv_heads: int,
                            head_dim: int, split_target: int, max_units: int = None,
                            max_merges: int = None) -> dict:
    """The prefill planner on the host (no CUDA call). Returns dict(units [n, 8],
    merges [m, 8], blocks) with the record layouts of include/pkv.h."""
    qo = _host_indptr(qo_indptr_host)
    kv = _host_indptr(kv_indptr_host)
    batch = kv.size - 1
    G = n_qo_heads // max(n_kv_heads, 1)
    tile = 64 // max(G, 1)
    if max_units is None:
        max_units = (int(qo[-1]) // max(tile, 1) + batch) * n_kv_heads + 2 * max(split_target, 0) + 1
    if max_merges is None:
        max_merges = max(split_target, 0) + 1
    units = np.zeros((max(max_units, 1), 8), np.int32)
    merges = np.zeros((max(max_merges, 1), 8), np.int32)
    counts = np.zeros(3, np.int32)
    _check(library().paged_prefill_plan_host(_ptr(qo), _ptr(kv), batch, n_qo_heads, n_kv_heads,
                                             head_dim, split_target, _ptr(units), max_units,
                                             _ptr(merges), max_merges, _ptr(counts)))
    nu, nm, nb = (int(x) for x in counts)
    return {"units": units[:nu].copy(), "merges": merges[:nm].copy(), "blocks": nb}


def paged_prefill_plan_destroy(plan: PrefillPlan) -> None:
    if plan.handle:
        library().paged_prefill_plan_destroy(plan.handle)
        plan.handle = None


def paged_decode_plan_destroy(plan: Plan) -> None:
    if plan.handle:
        library().paged_decode_plan_destroy(plan.handle)
        plan.handle = None


def paged_decode_plan_host(kv_indptr_host, n_kv_heads: int, head_dim: int, ctas: int,
                           heads_per_cta: int = 0, shared_indptr=None, shared_len=None,
                           requests_per_unit: int = 0, max_units: int = None,
                           max_merges: int = None, max_partials: int = None):
    """The planner alone (host, no CUDA).

    Returns dict(units [n, 8], cta_begin [ctas + 1], merges [m, 4], part_list,
    partials, chunk, ctas_used)."""
    ip = _host_indptr(kv_indptr_host)
    batch = ip.size - 1
    hpc = heads_per_cta or min(n_kv_heads, 512 // head_dim)
    groups = max(1, n_kv_heads // max(1, hpc))
    if max_units is None:
        max_units = 2 * ctas + 2 * max(batch, 1) * groups
    if max_merges is None:
        max_merges = max(batch, 1) * groups
    if max_partials is None:
        max_partials = max_units * max(1, requests_per_unit)
    sp = np.ascontiguousarray(shared_indptr if shared_indptr is not None else [0], np.int32)
    sl = np.ascontiguousarray(shared_len if shared_len is not None else [0], np.int32)
    n_shared = sp.size - 1
    units = np.zeros((max(max_units, 1), 8), np.int32)
    cta_begin = np.zeros(ctas + 1, np.int32)
    merges = np.zeros((max(max_merges, 1), 4), np.int32)
    part_list = np.zeros(max(max_partials, 1), np.int32)
    counts = np.zeros(5, np.int32)
    _check(library().paged_decode_plan_host(
        _ptr(ip), batch, n_kv_heads, head_dim, heads_per_cta, ctas, _ptr(sp), n_shared, _ptr(sl),
        requests_per_unit, _ptr(units), max_units, _ptr(cta_begin), _ptr(merges), max_merges,
        _ptr(part_list), max_partials, _ptr(counts)))
    nu, nc, nm, npart, chunk = (int(x) for x in counts)
    return {"units": units[:nu].copy(), "cta_begin": cta_begin.copy(), "ctas_used": nc,
            "merges": merges[:nm].copy(), "part_list": part_list[:npart].copy(),
            "partials": npart, "chunk": chunk}
