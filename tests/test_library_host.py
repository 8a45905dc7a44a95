"""Host-side checks of the C-ABI library (no GPU): exports, argument errors, planner."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_gqa_tokentokvpool_gb300 import build
    build.build()
    import paged_kv_gqa_tokentokvpool_gb300 as m
    return m


def declared_functions():
    names = []
    inc = os.path.join(ROOT, "include")
    for f in sorted(os.listdir(inc)):
        if f.endswith(".h"):
            text = open(os.path.join(inc, f)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\(", text, flags=re.M)
    return names


def test_header_declares_the_boundary():
    names = set(declared_functions())
    for n in ("kvpool_append", "paged_decode_plan_create", "paged_decode_plan",
              "paged_decode_attn", "paged_decode_plan_destroy", "pkv_last_error"):
        assert n in names


def test_library_exports_every_declared_symbol(pkv):
    lib = ctypes.CDLL(pkv.LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), f"libpkv.so does not export {name}"
    assert set(pkv.EXPORTED) <= set(declared_functions())


def test_errors_are_reported_before_any_launch(pkv):
    lib = pkv.library()
    buf = (ctypes.c_uint8 * 64)()
    p = ctypes.cast(buf, ctypes.c_void_p)
    # n < 0
    assert lib.kvpool_append(p, p, p, p, p, -1, 8, 128, 16, None) == pkv.PKV_ERR_INVALID_ARG
    assert "n = -1" in pkv.pkv_last_error()
    # NULL pointers
    assert lib.kvpool_append(None, p, p, p, p, 1, 8, 128, 16, None) == pkv.PKV_ERR_INVALID_ARG
    # row not a multiple of 16 bytes
    assert lib.kvpool_append(p, p, p, p, p, 1, 1, 4, 16, None) == pkv.PKV_ERR_UNSUPPORTED
    # more rows than slots
    assert lib.kvpool_append(p, p, p, p, p, 20, 8, 128, 16, None) == pkv.PKV_ERR_INVALID_ARG
    # n = 0 is a no-op that succeeds even with NULL pointers
    assert lib.kvpool_append(None, None, None, None, None, 0, 8, 128, 16, None) == pkv.PKV_OK
    # misaligned pool
    mis = ctypes.c_void_p(ctypes.addressof(buf) + 2)
    if ctypes.addressof(buf) % 16 == 0:
        assert lib.kvpool_append(mis, p, p, p, p, 1, 8, 128, 16, None) == pkv.PKV_ERR_INVALID_ARG
    # unsupported shapes are rejected by plan creation before touching the device
    h = ctypes.c_void_p()
    for hq, hkv, d in [(32, 8, 64), (30, 8, 128), (48, 4, 128), (32, 16, 128), (32, 0, 128)]:
        rc = lib.paged_decode_plan_create(ctypes.byref(h), 8, 1000, hq, hkv, d)
        assert rc == pkv.PKV_ERR_UNSUPPORTED, (hq, hkv, d, rc)
    assert lib.paged_decode_plan_create(ctypes.byref(h), 0, 1000, 32, 8, 128) == pkv.PKV_ERR_INVALID_ARG
    assert lib.paged_decode_plan_create(None, 8, 1000, 32, 8, 128) == pkv.PKV_ERR_INVALID_ARG
    # calls without a plan
    assert lib.paged_decode_plan(None, p, 1, None) == pkv.PKV_ERR_PLAN
    assert lib.paged_decode_attn(p, p, p, p, p, 1, 32, 8, 128, ctypes.c_float(0.1), p, p, None,
                                 None) == pkv.PKV_ERR_PLAN
    lib.paged_decode_plan_destroy(None)  # no-op


def check_plan(indptr, units, merges, chunk, cap):
    indptr = np.asarray(indptr, np.int64)
    B = indptr.size - 1
    lengths = np.diff(indptr)
    covered = [np.zeros(L, np.int32) for L in lengths]
    partial_owner = {}
    direct = set()
    for b, t0, t1, part in units:
        assert 0 <= b < B and 0 <= t0 <= t1 <= lengths[b]
        assert t1 - t0 <= max(chunk, lengths[b] if part < 0 else chunk)
        covered[b][t0:t1] += 1
        if part < 0:
            assert (t0, t1) == (0, lengths[b]), "a direct unit covers its whole context"
            assert b not in direct
            direct.add(b)
        else:
            assert part not in partial_owner
            partial_owner[part] = (b, t0, t1)
    for b in range(B):
        assert np.all(covered[b] == 1), f"request {b}: tokens not covered exactly once"
    merged = set()
    for b, first, count, _ in merges:
        assert count >= 2 and b not in merged and b not in direct
        merged.add(b)
        parts = [partial_owner[first + c] for c in range(count)]
        assert all(pb == b for pb, _, _ in parts)
        assert sum(t1 - t0 for _, t0, t1 in parts) == lengths[b]
        assert all(t1 > t0 for _, t0, t1 in parts), "split parts are non-empty"
    assert merged | direct == set(range(B))
    assert len(partial_owner) == sum(int(c) for _, _, c, _ in merges)
    if len(partial_owner):
        assert set(partial_owner) == set(range(len(partial_owner)))
    sizes = [t1 - t0 for _, t0, t1, _ in units]
    assert sizes == sorted(sizes, reverse=True), "units are listed longest first"
    assert len(units) <= max(cap, B)


@pytest.mark.parametrize("seed", range(12))
def test_planner_covers_every_token_once(pkv, seed):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 300))
    kind = seed % 4
    if kind == 0:
        lengths = rng.integers(0, 5000, B)
    elif kind == 1:
        lengths = np.rint(np.exp(rng.uniform(np.log(1), np.log(200000), B))).astype(np.int64)
    elif kind == 2:
        lengths = rng.integers(0, 40, B)
    else:
        lengths = np.full(B, int(rng.integers(1, 70000)))
    indptr = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    sms, per_sm = 152, int(rng.integers(1, 5))
    units, merges, chunk = pkv.paged_decode_plan_host(indptr, sms, per_sm)
    check_plan(indptr, units, merges, chunk, sms * per_sm * 4)
    assert chunk >= 1
    if lengths.max() > 256:
        assert chunk >= 256 and chunk % 64 == 0


def test_planner_edge_cases(pkv):
    # empty batch
    u, m, c = pkv.paged_decode_plan_host(np.zeros(1, np.int32), 152, 2)
    assert len(u) == 0 and len(m) == 0
    # all contexts empty: one (empty) direct unit per request
    u, m, c = pkv.paged_decode_plan_host(np.zeros(5, np.int32), 152, 2)
    assert len(u) == 4 and all(t0 == t1 == 0 and p == -1 for _, t0, t1, p in u)
    # a single huge context is split across the whole device
    u, m, c = pkv.paged_decode_plan_host(np.array([0, 131072], np.int32), 152, 2)
    assert len(m) == 1 and 152 <= len(u) <= 152 * 2 * 4
    check_plan([0, 131072], u, m, c, 152 * 8)
    # skewed batch like the 128-request long-context workload
    rng = np.random.default_rng(5)
    L = np.rint(np.exp(rng.uniform(np.log(128), np.log(32768), 127))).astype(np.int64)
    L = np.append(L, 131072)
    ip = np.concatenate([[0], np.cumsum(L)]).astype(np.int32)
    u, m, c = pkv.paged_decode_plan_host(ip, 152, 2)
    check_plan(ip, u, m, c, 152 * 8)
    assert max(t1 - t0 for _, t0, t1, _ in u) <= c


def test_planner_rejects_bad_input(pkv):
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_decode_plan_host(np.array([0, 5, 3], np.int32), 152, 2)
    assert e.value.code == pkv.PKV_ERR_INVALID_ARG
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_decode_plan_host(np.array([1, 5], np.int32), 152, 2)
    assert e.value.code == pkv.PKV_ERR_INVALID_ARG
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_decode_plan_host(np.array([0, 100000], np.int32), 152, 2, max_units=3)
    assert e.value.code == pkv.PKV_ERR_PLAN
