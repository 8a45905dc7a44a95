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
    for hq, hkv, d in [(32, 8, 64), (30, 8, 128), (48, 4, 128), (32, 16, 128), (32, 0, 128),
                       (24, 6, 128), (48, 3, 256)]:
        rc = lib.paged_decode_plan_create(ctypes.byref(h), 8, 1000, hq, hkv, d)
        assert rc == pkv.PKV_ERR_UNSUPPORTED, (hq, hkv, d, rc)
    assert lib.paged_decode_plan_create(ctypes.byref(h), 0, 1000, 32, 8, 128) == pkv.PKV_ERR_INVALID_ARG
    assert lib.paged_decode_plan_create(None, 8, 1000, 32, 8, 128) == pkv.PKV_ERR_INVALID_ARG
    # calls without a plan
    assert lib.paged_decode_plan(None, p, 1, None) == pkv.PKV_ERR_PLAN
    assert lib.paged_decode_attn(p, p, p, p, p, 1, 32, 8, 128, ctypes.c_float(0.1), p, p, None,
                                 None) == pkv.PKV_ERR_PLAN
    assert lib.paged_decode_plan_set_flags(None, pkv.PKV_PLAN_EARLY_GATHER) == pkv.PKV_ERR_PLAN
    # chunked prefill: shapes and sizes are checked before the device is touched
    for hq, hkv, d in [(32, 8, 64), (30, 8, 128), (48, 4, 128), (32, 0, 128)]:
        rc = lib.paged_prefill_plan_create(ctypes.byref(h), 8, 1000, hq, hkv, d)
        assert rc == pkv.PKV_ERR_UNSUPPORTED, (hq, hkv, d, rc)
    assert lib.paged_prefill_plan_create(ctypes.byref(h), 0, 1000, 32, 8, 128) == pkv.PKV_ERR_INVALID_ARG
    assert lib.paged_prefill_plan_create(None, 8, 1000, 32, 8, 128) == pkv.PKV_ERR_INVALID_ARG
    assert lib.paged_prefill_plan(None, p, p, 1, None) == pkv.PKV_ERR_PLAN
    assert lib.paged_prefill_attn(p, p, p, p, p, p, 1, 32, 8, 128, ctypes.c_float(0.1), p, p,
                                  None, None) == pkv.PKV_ERR_PLAN
    lib.paged_prefill_plan_destroy(None)  # no-op
    lib.paged_decode_plan_destroy(None)  # no-op
    # the plan's mode, host times and the static entry's status need their out arguments
    one = ctypes.c_int(7)
    assert lib.paged_decode_plan_mode(None, ctypes.byref(one)) == pkv.PKV_ERR_INVALID_ARG
    assert lib.paged_decode_plan_host_times(None, None, None, None, 0) == pkv.PKV_ERR_PLAN
    assert lib.paged_decode_attn_static_status(None, None) == pkv.PKV_ERR_INVALID_ARG
    assert lib.paged_decode_plan_set_flags(None, pkv.PKV_PLAN_PERSISTENT) == pkv.PKV_ERR_PLAN
    # host KV tier reads: both host pools and pool sizes are required before anything else
    f = ctypes.c_float(0.1)
    assert lib.paged_decode_attn_tiered(p, p, p, 16, None, p, 4, p, p, 1, 32, 8, 128, f, p, p,
                                        None, None) == pkv.PKV_ERR_INVALID_ARG
    assert "k_host and v_host" in pkv.pkv_last_error()
    assert lib.paged_decode_attn_tiered(p, p, p, 0, p, p, 4, p, p, 1, 32, 8, 128, f, p, p,
                                        None, None) == pkv.PKV_ERR_INVALID_ARG
    assert lib.paged_decode_attn_tiered(p, p, p, 16, p, p, 4, p, p, 1, 32, 8, 128, f, p, p,
                                        None, None) == pkv.PKV_ERR_PLAN


def test_header_constants_match_the_binding(pkv):
    text = open(os.path.join(ROOT, "include", "pkv.h")).read()
    flags = dict(re.findall(r"#define\s+(PKV_PLAN_\w+)\s+(\d+)u", text))
    assert flags == {"PKV_PLAN_EARLY_GATHER": str(pkv.PKV_PLAN_EARLY_GATHER),
                     "PKV_PLAN_PERSISTENT": str(pkv.PKV_PLAN_PERSISTENT),
                     "PKV_PLAN_SINGLE_LAUNCH": str(pkv.PKV_PLAN_SINGLE_LAUNCH)}
    codes = dict(re.findall(r"(PKV_(?:OK|ERR_\w+))\s*=\s*(-?\d+)", text))
    assert codes and all(getattr(pkv, k) == int(v) for k, v in codes.items())


def check_plan(indptr, n_kv_heads, head_dim, ctas, plan, hpc=0, shared=None, rpu=None):
    """Every (request, head group, token) is attended exactly once; units, partial
    slots and merge records are consistent. shared = (shared_indptr, shared_len),
    rpu = requests per shared-prefix unit."""
    indptr = np.asarray(indptr, np.int64)
    B = indptr.size - 1
    lengths = np.diff(indptr)
    hpg = hpc or min(n_kv_heads, 512 // head_dim)
    groups = n_kv_heads // hpg
    units, cta_begin, merges, chunk = plan["units"], plan["cta_begin"], plan["merges"], plan["chunk"]
    part_list = plan["part_list"]
    n = len(units)
    assert cta_begin[0] == 0 and cta_begin[-1] == n
    assert np.all(np.diff(cta_begin) >= 0)
    assert len(cta_begin) - 1 == ctas, "every CTA of the grid has an entry"
    assert plan["ctas_used"] <= ctas
    prefix = np.zeros(B, np.int64)
    run_size = np.ones(B, np.int64)  # members of the sharing run of each request
    if shared is not None:
        sp, sl = shared
        for s in range(len(sp) - 1):
            prefix[sp[s]:sp[s + 1]] = sl[s]
            run_size[sp[s]:sp[s + 1]] = sp[s + 1] - sp[s]
    covered = {(b, g): np.zeros(lengths[b], np.int32) for b in range(B) for g in range(groups)}
    direct, slot_owner = set(), {}
    for b, hg, t0, t1, part, nreq, idx_begin, length in units:
        assert 0 <= b and b + nreq <= B and nreq >= 1 and 0 <= hg < groups and 0 <= t0 <= t1
        assert idx_begin == indptr[b] + t0
        if nreq > 1 or length < 0:  # a shared prefix
            assert length in (-1, -2) and part >= 0
            if rpu is not None:  # -2: other units of the run read the same slots
                assert length == (-2 if run_size[b] > rpu else -1)
            for r in range(nreq):
                assert t1 <= prefix[b + r], "prefix unit beyond the shared prefix"
        else:
            assert length == lengths[b] and t1 <= lengths[b]
        for r in range(nreq):
            covered[(b + r, hg)][t0:t1] += 1
        if part < 0:
            assert nreq == 1 and (t0, t1) == (0, lengths[b])
            assert (b, hg) not in direct
            direct.add((b, hg))
        else:
            for r in range(nreq):
                assert part + r not in slot_owner
                slot_owner[part + r] = (b + r, hg, t0, t1)
            assert t1 > t0
    for key, cov in covered.items():
        assert np.all(cov == 1), f"{key}: tokens not covered exactly once"
    merged = set()
    for b, hg, first, count in merges:
        assert count >= 1 and (b, hg) not in merged and (b, hg) not in direct
        merged.add((b, hg))
        ps = [slot_owner[part_list[first + c]] for c in range(count)]
        assert all(pb == b and ph == hg for pb, ph, _, _ in ps)
        assert sum(t1 - t0 for _, _, t0, t1 in ps) == lengths[b]
    assert merged | direct == set(covered)
    assert len(slot_owner) == plan["partials"] == sum(int(c) for *_, c in merges)
    assert sorted(part_list.tolist()) == list(range(plan["partials"]))
    assert n <= 2 * ctas + 2 * B * groups
    # Costed as the kernel spends its time (whole pipeline stages of st tokens plus
    # a fixed cost per unit), no CTA exceeds the larger of the average cost and the
    # cost of a context too short to split by more than one CTA's possible slack:
    # a minimum piece, a stage and a unit.
    st = 16 * (512 // (hpg * head_dim))
    uc = max(1, st // 4)

    def cost(t):
        return -(-int(t) // st) * st + uc if t > 0 else 0

    for b, hg, t0, t1, part, nreq, idx_begin, length in units:
        if t1 > t0 and part >= 0:
            # pieces of split contexts start on a stage boundary of their item and
            # are never shorter than the minimum piece, except an item's whole run
            start = 0 if (nreq > 1 or length < 0) else int(prefix[b])
            item_len = (int(prefix[b]) if (nreq > 1 or length < 0) else lengths[b] - start)
            assert (t0 - start) % st == 0, "a split falls inside a pipeline stage"
            assert t1 - t0 >= min(64, item_len), "a piece shorter than the minimum"
    cta_cost = [sum(cost(u[3] - u[2]) for u in units[a:b]) for a, b in zip(cta_begin[:-1], cta_begin[1:])]
    # the planner's items: per head group, one per plain request; with shared
    # prefixes, ceil(run / rpu) prefix items per run and a suffix item per member
    item_lens = []
    if shared is None:
        item_lens = [int(L) for L in lengths]
    elif rpu is not None:
        sp, sl = shared
        in_run = np.zeros(B, bool)
        for s in range(len(sp) - 1):
            if sl[s] > 0 and sp[s + 1] > sp[s]:
                in_run[sp[s]:sp[s + 1]] = True
                item_lens += [int(sl[s])] * (-(-(sp[s + 1] - sp[s]) // rpu))
                item_lens += [int(lengths[m] - sl[s]) for m in range(sp[s], sp[s + 1])]
        item_lens += [int(lengths[b]) for b in range(B) if not in_run[b]]
    if item_lens:
        whole = sum(cost(L) for L in item_lens) * groups
        short = max([cost(L) for L in item_lens if L < 2 * 64 + st] + [0])
        assert max(cta_cost) <= max(whole / ctas, short) + 64 + st + uc


@pytest.mark.parametrize("seed", range(8))
def test_planner_with_shared_prefixes(pkv, seed):
    rng = np.random.default_rng(100 + seed)
    n_groups = int(rng.integers(1, 6))
    sizes = rng.integers(1, 10, n_groups)
    singles = rng.integers(0, 4, n_groups + 1)
    lengths, sp, sl = [], [], []
    for gi in range(n_groups):
        lengths += list(rng.integers(0, 3000, singles[gi]))
        P = int(rng.integers(0, 5000))
        sp.append(len(lengths))
        sl.append(P)
        lengths += list(P + rng.integers(1, 2000, sizes[gi]))
        sp.append(len(lengths))
    lengths += list(rng.integers(0, 3000, singles[-1]))
    # runs are given as [start, end) pairs collapsed into an indptr of groups
    starts, ends = sp[0::2], sp[1::2]
    shared_indptr, shared_len = [], []
    for s_, e_, P in zip(starts, ends, sl):
        shared_indptr.append((s_, e_, P))
    indptr = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    # the C API takes consecutive runs: build one run per group, with standalone
    # requests between runs expressed as runs of length 0 shared slots
    sp_arr, sl_arr = [0], []
    cursor = 0
    for s_, e_, P in shared_indptr:
        if s_ > cursor:
            sp_arr.append(s_)
            sl_arr.append(0)
        sp_arr.append(e_)
        sl_arr.append(P)
        cursor = e_
    if sp_arr[0] != 0 or len(sp_arr) < 2:
        pass
    rpu = [2, 4, 8, 16][seed % 4]
    ctas = 304
    plan = pkv.paged_decode_plan_host(indptr, 8, 128, ctas, shared_indptr=sp_arr, shared_len=sl_arr,
                                      requests_per_unit=rpu)
    check_plan(indptr, 8, 128, ctas, plan, shared=(np.array(sp_arr), np.array(sl_arr)), rpu=rpu)
    # a prefix unit serves at most requests_per_unit requests
    assert plan["units"][:, 5].max() <= rpu


def test_planner_rejects_bad_sharing(pkv):
    indptr = np.array([0, 100, 150, 300], np.int32)
    with pytest.raises(pkv.PkvError) as e:  # shared prefix as long as a member's context
        pkv.paged_decode_plan_host(indptr, 8, 128, 304, shared_indptr=[0, 2], shared_len=[50],
                                   requests_per_unit=4)
    assert e.value.code == pkv.PKV_ERR_INVALID_ARG
    with pytest.raises(pkv.PkvError) as e:  # run beyond the batch
        pkv.paged_decode_plan_host(indptr, 8, 128, 304, shared_indptr=[1, 5], shared_len=[10],
                                   requests_per_unit=4)
    assert e.value.code == pkv.PKV_ERR_INVALID_ARG


SHAPES = [(8, 128), (4, 256), (2, 128), (1, 256), (8, 256)]


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
    hkv, d = SHAPES[seed % len(SHAPES)]
    ctas = 152 * int(rng.integers(1, 3))
    hpc = [0, 1, 2][seed % 3] if min(hkv, 512 // d) >= 2 else 0
    plan = pkv.paged_decode_plan_host(indptr, hkv, d, ctas, heads_per_cta=hpc)
    check_plan(indptr, hkv, d, ctas, plan, hpc)


def test_planner_edge_cases(pkv):
    # empty batch
    p = pkv.paged_decode_plan_host(np.zeros(1, np.int32), 8, 128, 304)
    assert len(p["units"]) == 0 and len(p["merges"]) == 0
    # all contexts empty: one (empty) direct unit per (request, head group)
    p = pkv.paged_decode_plan_host(np.zeros(5, np.int32), 8, 128, 304)
    assert len(p["units"]) == 8 and all(u[2] == u[3] == 0 and u[4] == -1 for u in p["units"])
    check_plan(np.zeros(5, np.int32), 8, 128, 304, p)
    # a single huge context is spread over the whole device
    p = pkv.paged_decode_plan_host(np.array([0, 131072], np.int32), 8, 128, 304)
    check_plan([0, 131072], 8, 128, 304, p)
    assert len(p["merges"]) == 2 and p["ctas_used"] == 304
    # a tiny step: contexts too short for two minimum pieces stay whole, and the
    # two 30-token ones share a CTA (their stages cost less than the 100-token one's)
    p = pkv.paged_decode_plan_host(np.array([0, 100, 130], np.int32), 8, 128, 304)
    check_plan([0, 100, 130], 8, 128, 304, p)
    assert p["ctas_used"] == 3 and all(u[4] == -1 for u in p["units"])
    # the skewed 128-request long-context batch
    rng = np.random.default_rng(5)
    L = np.rint(np.exp(rng.uniform(np.log(128), np.log(32768), 127))).astype(np.int64)
    L = np.append(L, 131072)
    ip = np.concatenate([[0], np.cumsum(L)]).astype(np.int32)
    p = pkv.paged_decode_plan_host(ip, 8, 128, 304)
    check_plan(ip, 8, 128, 304, p)
    assert p["ctas_used"] == 304
    # a split context has few parts (range boundaries only)
    assert max(m[3] for m in p["merges"]) <= 2 * 131072 // (2 * L.sum() // 304) + 2


def test_planner_rejects_bad_input(pkv):
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_decode_plan_host(np.array([0, 5, 3], np.int32), 8, 128, 304)
    assert e.value.code == pkv.PKV_ERR_INVALID_ARG
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_decode_plan_host(np.array([1, 5], np.int32), 8, 128, 304)
    assert e.value.code == pkv.PKV_ERR_INVALID_ARG
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_decode_plan_host(np.array([0, 100000], np.int32), 8, 128, 304, max_units=1)
    assert e.value.code == pkv.PKV_ERR_PLAN
    with pytest.raises(pkv.PkvError) as e:  # 4 heads of dim 256 do not fit a 1 KB row
        pkv.paged_decode_plan_host(np.array([0, 10], np.int32), 4, 256, 304, heads_per_cta=4)
    assert e.value.code == pkv.PKV_ERR_UNSUPPORTED


# ---------------------------------------------------------------------------
# the chunked-prefill planner (host only)
# ---------------------------------------------------------------------------

def check_prefill_plan(qo, kv, hq, hkv, plan, split_target):
    """Every (query row, KV head) is planned exactly once; split units' pieces
    partition their range at ring-tile cuts at or below the first query's position."""
    qo, kv = np.asarray(qo, np.int64), np.asarray(kv, np.int64)
    G = hq // hkv
    tile = 128 // G
    units, merges = plan["units"], plan["merges"]
    covered = np.zeros((int(qo[-1]), hkv), np.int32)
    req_of_row = np.repeat(np.arange(len(qo) - 1), np.diff(qo))
    lengths = [int(x) for x in units[:, 7] - units[:, 6]]
    assert lengths == sorted(lengths, reverse=True), "longest range first"
    by_block = {}
    for part, g, q_row0, n_q, kv_begin, pos0, kv_lo, kv_hi in units:
        assert 1 <= n_q <= tile and 0 <= g < hkv
        b = req_of_row[q_row0]
        C, L = qo[b + 1] - qo[b], kv[b + 1] - kv[b]
        t0 = q_row0 - qo[b]
        assert t0 % tile == 0 and kv_begin == kv[b] and pos0 == L - C + t0
        assert 0 <= kv_lo < kv_hi <= pos0 + n_q
        if part < 0:
            assert kv_lo == 0 and kv_hi == pos0 + n_q
            covered[q_row0:q_row0 + n_q, g] += 1
        else:
            assert part not in by_block
            by_block[part] = (q_row0, n_q, g, pos0, kv_lo, kv_hi)
    assert sorted(by_block) == list(range(plan["blocks"]))
    for q_row0, n_q, g, first, count, *_ in merges:
        assert 2 <= count <= 16
        pieces = [by_block[first + c] for c in range(count)]
        assert all(p[:3] == (q_row0, n_q, g) for p in pieces)
        pos0 = pieces[0][3]
        ranges = sorted((p[4], p[5]) for p in pieces)
        assert ranges[0][0] == 0 and ranges[-1][1] == pos0 + n_q
        for (lo, hi), (lo2, _) in zip(ranges, ranges[1:]):
            assert hi == lo2 and hi % 64 == 0 and hi <= pos0, "cut on a tile edge at or below pos0"
        covered[q_row0:q_row0 + n_q, g] += 1
    assert np.all(covered == 1)
    n_tile_units = sum(-(-int(qo[b + 1] - qo[b]) // tile) for b in range(len(qo) - 1)) * hkv
    if n_tile_units >= split_target:
        assert len(merges) == 0, "enough units: no split"


@pytest.mark.parametrize("seed", range(10))
def test_prefill_planner_properties(pkv, seed):
    rng = np.random.default_rng(seed)
    B = int(rng.integers(1, 12))
    chunks = rng.choice([0, 1, 17, 64, 300, 512], B)
    contexts = chunks + rng.integers(0, [20000, 3000, 50][seed % 3], B)
    qo = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    kv = np.concatenate([[0], np.cumsum(contexts)]).astype(np.int32)
    hq, hkv, d = [(32, 8, 128), (16, 4, 256), (8, 8, 128), (64, 8, 128)][seed % 4]
    for target in (0, 100, 912, 100000):
        plan = pkv.paged_prefill_plan_host(qo, kv, hq, hkv, d, target)
        check_prefill_plan(qo, kv, hq, hkv, plan, target)


def test_prefill_planner_splits_a_short_step(pkv):
    # 8 requests x 64-token chunks over long contexts: far fewer units than the target
    qo = np.arange(0, 9 * 64, 64, dtype=np.int32)
    kv = np.concatenate([[0], np.cumsum([16000, 9000, 64, 300, 15000, 7000, 2000, 12000])]).astype(np.int32)
    plan = pkv.paged_prefill_plan_host(qo, kv, 32, 8, 128, 912)
    check_prefill_plan(qo, kv, 32, 8, plan, 912)
    assert len(plan["merges"]) > 0 and len(plan["units"]) > 256


def test_prefill_planner_rejects_bad_input(pkv):
    with pytest.raises(pkv.PkvError) as e:  # chunk longer than the slot list
        pkv.paged_prefill_plan_host(np.array([0, 10], np.int32), np.array([0, 9], np.int32),
                                    32, 8, 128, 0)
    assert e.value.code == pkv.PKV_ERR_INVALID_ARG
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_prefill_plan_host(np.array([0, 10], np.int32), np.array([0, 90], np.int32),
                                    32, 8, 128, 0, max_units=1)
    assert e.value.code == pkv.PKV_ERR_PLAN
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_prefill_plan_host(np.array([0, 1], np.int32), np.array([0, 9], np.int32),
                                    30, 8, 128, 0)
    assert e.value.code == pkv.PKV_ERR_UNSUPPORTED


def _fill_count(items, T, st, uc, min_piece=64):
    """CTAs the documented greedy fill needs at budget T (None when a piece cannot fit
    an empty CTA): whole items while they fit, then whole stages of the next item,
    never leaving or taking less than a minimum piece of a split item."""
    def cost(t):
        return -(-t // st) * st + uc
    n, budget = 0, T
    for length in items:
        r = length
        while r > 0:
            if cost(r) <= budget:
                budget -= cost(r)
                break
            p = (budget - uc) // st * st if budget > uc else 0
            if r - p < min_piece:
                p = (r - min_piece) // st * st if r >= min_piece else 0
            if p >= min_piece:
                r -= p
            elif budget == T:
                return None
            n += 1
            budget = T
    return n + (budget < T)


@pytest.mark.parametrize("seed", range(40))
def test_planner_budget_is_the_smallest_that_fits(pkv, seed):
    """No smaller budget than the plan's costliest CTA lets the greedy fill fit the
    grid: the bisection found the least one."""
    rng = np.random.default_rng(700 + seed)
    B = int(rng.integers(1, 40))
    lengths = rng.integers(0, [300, 3000, 20000][seed % 3], B)
    ctas = int(rng.integers(1, 64))
    hkv, d = SHAPES[seed % len(SHAPES)]
    indptr = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    plan = pkv.paged_decode_plan_host(indptr, hkv, d, ctas)
    check_plan(indptr, hkv, d, ctas, plan)
    hpg = min(hkv, 512 // d)
    st = 16 * (512 // (hpg * d))
    uc = max(1, st // 4)
    units, cb = plan["units"], plan["cta_begin"]
    costs = [sum(-(-int(u[3] - u[2]) // st) * st + uc for u in units[a:b] if u[3] > u[2])
             for a, b in zip(cb[:-1], cb[1:])]
    if max(costs) == 0:
        return
    items = [int(L) for L in lengths for _ in range(hkv // hpg)]
    items = [L for L in items if L > 0]
    n = _fill_count(items, max(costs) - 1, st, uc)
    assert n is None or n > ctas, f"budget {max(costs) - 1} fits in {n} of {ctas} CTAs"
