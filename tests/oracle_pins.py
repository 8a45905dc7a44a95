"""Pins that tie the fp64 oracle to something other than itself.

Each ``pin_*`` takes an oracle object (``oracle.OracleLib``) and raises
AssertionError when the oracle disagrees with:
  * a library routine on a dense gather: torch's fp64 scaled_dot_product_attention
    and torch.logsumexp, with K/V heads expanded by repeat_interleave (contiguous
    GQA groups, query head h -> KV head h / G, the grouping of "Pegainfer:
    纯Rust+CUDA构建的LLM推理引擎", section "1. 注意力机制优化");
  * closed forms: hand-derived examples (tests/golden/hand_examples.json), a
    single-token context (out = that V row, lse = s_0), a zero query (uniform
    weights: out = mean of the V rows, lse = ln L), identical V rows;
  * invariants: moving the listed rows anywhere in the pool (page size 1: a
    request only sees its slot list, "Agent-Infer: 纯 Rust 编写的高性能 LLM 推理引擎",
    section "分页 KV 缓存"), splitting a context and merging the halves by
    log-sum-exp, equal queries in a GQA group, Hq = Hkv reducing to MHA;
  * the mean of lse over many N(0,1) heads (ln L + sigma^2 / 2);
  * numpy's scatter for the append.
The mutation test plants mistakes in copies of the oracle and checks that some
pin fails for each.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                      "hand_examples.json")


def bf16_bits_of(x) -> np.ndarray:
    t = torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def widen(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def random_case(rng, lengths, hq, hkv, d, extra_slots=7, scale=None):
    lengths = list(lengths)
    n = sum(lengths)
    S = n + extra_slots
    perm = rng.permutation(S)
    indices = perm[:n].astype(np.int32)
    indptr = np.zeros(len(lengths) + 1, np.int32)
    indptr[1:] = np.cumsum(lengths)
    q = bf16_bits_of(rng.standard_normal((len(lengths), hq, d)))
    k = bf16_bits_of(rng.standard_normal((S, hkv, d)))
    v = bf16_bits_of(rng.standard_normal((S, hkv, d)))
    if scale is None:
        scale = float(np.float32(1.0 / math.sqrt(d)))
    return q, k, v, indptr, indices, scale


def sdpa_reference(q, k, v, indptr, indices, hq, hkv, d, scale):
    """Dense fp64 attention by torch's library routines, request by request."""
    G = hq // hkv
    B = len(indptr) - 1
    out = np.zeros((B, hq, d))
    lse = np.full((B, hq), -np.inf)
    qd, kd, vd = widen(q), widen(k), widen(v)
    for b in range(B):
        idx = indices[indptr[b]:indptr[b + 1]]
        if idx.size == 0:
            continue
        Q = torch.from_numpy(qd[b]).reshape(1, hq, 1, d)
        K = torch.from_numpy(kd[idx]).permute(1, 0, 2).repeat_interleave(G, dim=0)[None]
        V = torch.from_numpy(vd[idx]).permute(1, 0, 2).repeat_interleave(G, dim=0)[None]
        o = torch.nn.functional.scaled_dot_product_attention(Q, K, V, scale=float(scale))
        out[b] = o[0, :, 0].numpy()
        scores = (Q @ K.transpose(-1, -2))[0, :, 0] * float(scale)
        lse[b] = torch.logsumexp(scores, dim=-1).numpy()
    return out, lse


def _close(a, b, atol, rtol=0.0, what=""):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    with np.errstate(invalid="ignore"):
        both_inf = np.isinf(a) & np.isinf(b) & (np.sign(a) == np.sign(b))
        err = np.where(both_inf, 0.0, np.abs(a - b))
        ok = both_inf | (err <= atol + rtol * np.where(np.isfinite(b), np.abs(b), 0.0))
    assert ok.all(), f"{what}: max err {np.nanmax(err) if err.size else 0}"


def pin_golden(orc):
    data = json.load(open(GOLDEN))
    for case in data["cases"]:
        hq, hkv, d = case["n_qo_heads"], case["n_kv_heads"], case["head_dim"]
        out, lse = orc.decode(bf16_bits_of(case["q"]), bf16_bits_of(case["k_pool"]),
                              bf16_bits_of(case["v_pool"]), case["kv_indptr"],
                              case["kv_indices"], hq, hkv, d, case["sm_scale"])
        exp_lse = np.array([[float(x) for x in row] for row in case["lse"]])
        _close(lse, exp_lse, 1e-14, what=case["name"] + " lse")
        _close(out, np.array(case["out"]), 1e-14, what=case["name"] + " out")


def pin_golden_derivations():
    """The stored golden numbers equal their written closed forms."""
    e = math.e
    data = {c["name"]: c for c in json.load(open(GOLDEN))["cases"]}
    c = data["two_tokens_mha"]
    assert c["lse"][0][0] == math.log(1 + e)
    _close(c["out"][0][0], [1 + 2 / (1 + e), 2 + 2 / (1 + e)], 1e-15)
    c = data["three_tokens_gqa2"]
    z0 = math.exp(0.5) + e + 1
    z1 = math.exp(-0.25) + math.exp(0.5) + 1
    _close(c["lse"][0], [math.log(z0), math.log(z1)], 1e-15)
    _close(c["out"][0][0], [(math.exp(0.5) + 2) / z0, (e + 2) / z0], 1e-15)
    _close(c["out"][0][1], [(math.exp(-0.25) + 2) / z1, (math.exp(0.5) + 2) / z1], 1e-15)


def pin_sdpa(orc, seed=0):
    rng = np.random.default_rng(seed)
    for lengths, hq, hkv, d in [([1, 5, 3], 4, 4, 8), ([7, 0, 12, 2], 8, 2, 16),
                                ([33, 17], 32, 8, 128), ([9, 40], 16, 4, 256),
                                ([5, 6], 8, 1, 4)]:
        q, k, v, indptr, indices, scale = random_case(rng, lengths, hq, hkv, d)
        out, lse = orc.decode(q, k, v, indptr, indices, hq, hkv, d, scale)
        rout, rlse = sdpa_reference(q, k, v, indptr, indices, hq, hkv, d, scale)
        _close(out, rout, 1e-12, 1e-12, what=f"sdpa out {lengths},{hq}/{hkv},{d}")
        _close(lse, rlse, 1e-12, 1e-12, what=f"sdpa lse {lengths},{hq}/{hkv},{d}")


def pin_single_token(orc, seed=1):
    rng = np.random.default_rng(seed)
    hq, hkv, d = 8, 2, 128
    q, k, v, indptr, indices, scale = random_case(rng, [1, 1, 1], hq, hkv, d)
    out, lse = orc.decode(q, k, v, indptr, indices, hq, hkv, d, scale)
    qd, kd, vd = widen(q), widen(k), widen(v)
    for b in range(3):
        slot = indices[b]
        for h in range(hq):
            g = h // (hq // hkv)
            assert np.array_equal(out[b, h], vd[slot, g]), "L=1 must return the V row"
            s0 = float(np.float64(scale) * np.dot(qd[b, h], kd[slot, g]))
            assert abs(lse[b, h] - s0) <= 1e-12 * max(1.0, abs(s0)), "L=1: lse = s_0"


def pin_zero_query(orc, seed=2):
    rng = np.random.default_rng(seed)
    hq, hkv, d = 4, 2, 16
    q, k, v, indptr, indices, scale = random_case(rng, [1, 6, 31], hq, hkv, d)
    q[:] = 0
    out, lse = orc.decode(q, k, v, indptr, indices, hq, hkv, d, scale)
    vd = widen(v)
    for b in range(3):
        idx = indices[indptr[b]:indptr[b + 1]]
        for h in range(hq):
            g = h // (hq // hkv)
            _close(out[b, h], vd[idx, g].mean(axis=0), 1e-14, 1e-13, what="q=0 mean")
            _close(lse[b, h], math.log(len(idx)), 1e-14, what="q=0 lse")


def pin_identical_v(orc, seed=3):
    rng = np.random.default_rng(seed)
    hq, hkv, d = 8, 2, 32
    q, k, v, indptr, indices, scale = random_case(rng, [4, 19], hq, hkv, d)
    row = bf16_bits_of(rng.standard_normal((hkv, d)))
    v[indices] = row
    out, _ = orc.decode(q, k, v, indptr, indices, hq, hkv, d, scale)
    vd = widen(row)
    for b in range(2):
        for h in range(hq):
            _close(out[b, h], vd[h // (hq // hkv)], 1e-14, 1e-13, what="identical V")


def pin_permutation(orc, seed=4):
    rng = np.random.default_rng(seed)
    hq, hkv, d = 8, 4, 16
    q, k, v, indptr, indices, scale = random_case(rng, [3, 11, 8], hq, hkv, d, extra_slots=20)
    S = k.shape[0]
    pi = rng.permutation(S)
    k2 = np.empty_like(k)
    v2 = np.empty_like(v)
    k2[pi] = k
    v2[pi] = v
    out1, lse1 = orc.decode(q, k, v, indptr, indices, hq, hkv, d, scale)
    out2, lse2 = orc.decode(q, k2, v2, indptr, pi[indices].astype(np.int32), hq, hkv, d, scale)
    assert np.array_equal(out1, out2) and np.array_equal(lse1, lse2), "slot placement"


def pin_split_merge(orc, seed=5):
    rng = np.random.default_rng(seed)
    hq, hkv, d = 8, 2, 32
    lengths = [40, 13]
    q, k, v, indptr, indices, scale = random_case(rng, lengths, hq, hkv, d)
    whole_o, whole_l = orc.decode(q, k, v, indptr, indices, hq, hkv, d, scale)
    for b, L in enumerate(lengths):
        idx = indices[indptr[b]:indptr[b + 1]]
        for cut in (1, L // 3, L - 1):
            parts_o, parts_l = [], []
            for sub in (idx[:cut], idx[cut:]):
                o, l = orc.decode(q[b:b + 1], k, v, [0, len(sub)], sub, hq, hkv, d, scale)
                parts_o.append(o[0])
                parts_l.append(l[0])
            mo, ml = orc.lse_merge(np.stack(parts_o), np.stack(parts_l))
            _close(mo, whole_o[b], 1e-12, what="split/merge out")
            _close(ml, whole_l[b], 1e-12, what="split/merge lse")
    # an empty part contributes nothing
    o, l = orc.decode(q[:1], k, v, [0, 0], np.zeros(0, np.int32), hq, hkv, d, scale)
    mo, ml = orc.lse_merge(np.stack([o[0], whole_o[0]]), np.stack([l[0], whole_l[0]]))
    _close(mo, whole_o[0], 1e-15, what="merge with empty part")
    _close(ml, whole_l[0], 1e-15, what="merge with empty part lse")


def pin_gqa_equal_queries(orc, seed=6):
    rng = np.random.default_rng(seed)
    hq, hkv, d = 16, 4, 16
    q, k, v, indptr, indices, scale = random_case(rng, [9, 2], hq, hkv, d)
    G = hq // hkv
    for g in range(hkv):
        q[:, g * G:(g + 1) * G] = q[:, g * G][:, None]
    out, lse = orc.decode(q, k, v, indptr, indices, hq, hkv, d, scale)
    for g in range(hkv):
        for j in range(1, G):
            assert np.array_equal(out[:, g * G + j], out[:, g * G])
            assert np.array_equal(lse[:, g * G + j], lse[:, g * G])
    # distinct KV heads give distinct results (the group really selects a head)
    assert not np.allclose(out[:, 0], out[:, G])


def pin_empty(orc, seed=7):
    rng = np.random.default_rng(seed)
    q, k, v, indptr, indices, scale = random_case(rng, [0, 3, 0], 4, 2, 8)
    out, lse = orc.decode(q, k, v, indptr, indices, 4, 2, 8, scale)
    assert np.all(out[[0, 2]] == 0) and np.all(np.isneginf(lse[[0, 2]]))
    assert np.all(np.isfinite(lse[1]))


def pin_lse_statistics(orc, seed=8):
    """s ~ N(0, sigma^2) given the query, so E[lse] ~ ln L + sigma^2 / 2 for large L."""
    rng = np.random.default_rng(seed)
    for hq, hkv, d, kscale, L in [(32, 8, 128, 1.0, 4096), (16, 4, 256, 0.5, 4096)]:
        S = L * 4
        indices = rng.permutation(S)[: 4 * L].astype(np.int32)
        indptr = np.arange(0, 4 * L + 1, L, dtype=np.int32)
        q = bf16_bits_of(rng.standard_normal((4, hq, d)))
        k = bf16_bits_of(rng.standard_normal((S, hkv, d)) * kscale)
        v = bf16_bits_of(rng.standard_normal((S, hkv, d)))
        scale = float(np.float32(1.0 / math.sqrt(d)))
        _, lse = orc.decode(q, k, v, indptr, indices, hq, hkv, d, scale)
        sigma2 = kscale ** 2
        assert abs(lse.mean() - (math.log(L) + sigma2 / 2)) < 0.08, lse.mean()


def pin_append(orc, seed=9):
    rng = np.random.default_rng(seed)
    S, hkv, d = 50, 2, 8
    pool = bf16_bits_of(rng.standard_normal((S, hkv, d)))
    ids = rng.permutation(S)[:13].astype(np.int32)
    rows = bf16_bits_of(rng.standard_normal((13, hkv, d)))
    got = orc.append(pool, ids, rows)
    want = pool.copy()
    want[ids] = rows
    assert np.array_equal(got, want)
    untouched = np.setdiff1d(np.arange(S), ids)
    assert np.array_equal(got[untouched], pool[untouched])
    assert np.array_equal(orc.append(pool, np.zeros(0, np.int32), rows[:0]), pool)


ALL_PINS = [pin_golden, pin_sdpa, pin_single_token, pin_zero_query, pin_identical_v,
            pin_permutation, pin_split_merge, pin_gqa_equal_queries, pin_empty,
            pin_lse_statistics, pin_append]
