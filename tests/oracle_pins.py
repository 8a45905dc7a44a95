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
  * numpy's scatter for the append;
  * for chunked prefill (causal attention of a request's newest C tokens over its
    L listed slots, "Agent-Infer", section "连续批处理"): torch's fp64
    scaled_dot_product_attention with an explicit causal mask, a brute-force
    loop on a tiny case, the first token of a chunk with no prefix (out = its V
    row), causality (rows after a query's position do not matter to it, the row
    at it does), a chunk cut in two giving the same rows, and chunks of one token
    reducing to decode.
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


def pin_numpy_brute_force(orc, seed=10):
    """Tiny random cases (B <= 3, L <= 5, head_dim 4 or 8) against the definition
    written out with numpy, request by request and head by head."""
    rng = np.random.default_rng(seed)
    for lengths, hq, hkv, d in [([1, 5, 3], 2, 1, 4), ([4, 2], 4, 2, 8), ([5], 8, 2, 8),
                                ([3, 0, 2], 2, 2, 4)]:
        q, k, v, indptr, indices, scale = random_case(rng, lengths, hq, hkv, d)
        out, lse = orc.decode(q, k, v, indptr, indices, hq, hkv, d, scale)
        qd, kd, vd = widen(q), widen(k), widen(v)
        G = hq // hkv
        for b in range(len(lengths)):
            idx = indices[indptr[b]:indptr[b + 1]]
            for h in range(hq):
                if idx.size == 0:
                    assert lse[b, h] == -np.inf and np.all(out[b, h] == 0)
                    continue
                s = np.array([scale * np.dot(qd[b, h], kd[j, h // G]) for j in idx])
                m = s.max()
                want_lse = m + np.log(np.exp(s - m).sum())
                want = (np.exp(s - want_lse)[:, None] * vd[idx, h // G]).sum(axis=0)
                assert abs(lse[b, h] - want_lse) < 1e-12, (lengths, b, h)
                assert np.max(np.abs(out[b, h] - want)) < 1e-12, (lengths, b, h)


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


# ---------------------------------------------------------------------------
# chunked prefill
# ---------------------------------------------------------------------------

def prefill_case(rng, chunks, contexts, hq, hkv, d, extra_slots=5):
    """Request b lists contexts[b] slots; its newest chunks[b] tokens are the chunk."""
    assert all(0 <= c <= l for c, l in zip(chunks, contexts))
    n = sum(contexts)
    S = n + extra_slots
    indices = rng.permutation(S)[:n].astype(np.int32)
    kv_indptr = np.concatenate([[0], np.cumsum(contexts)]).astype(np.int32)
    qo_indptr = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    q = bf16_bits_of(rng.standard_normal((int(qo_indptr[-1]), hq, d)))
    k = bf16_bits_of(rng.standard_normal((S, hkv, d)))
    v = bf16_bits_of(rng.standard_normal((S, hkv, d)))
    scale = float(np.float32(1.0 / math.sqrt(d)))
    return q, k, v, qo_indptr, kv_indptr, indices, scale


def sdpa_prefill_reference(q, k, v, qo_indptr, kv_indptr, indices, hq, hkv, d, scale):
    """Dense fp64 causal attention per request by torch's library routines, with the
    mask built from positions: query c of a chunk of C over L entries sees j <= L-C+c."""
    G = hq // hkv
    NQ = int(qo_indptr[-1])
    out = np.zeros((NQ, hq, d))
    lse = np.zeros((NQ, hq))
    qd, kd, vd = widen(q), widen(k), widen(v)
    for b in range(len(kv_indptr) - 1):
        C = int(qo_indptr[b + 1] - qo_indptr[b])
        if C == 0:
            continue
        idx = indices[kv_indptr[b]:kv_indptr[b + 1]]
        L = idx.size
        Q = torch.from_numpy(qd[qo_indptr[b]:qo_indptr[b + 1]]).permute(1, 0, 2)[None]
        K = torch.from_numpy(kd[idx]).permute(1, 0, 2).repeat_interleave(G, dim=0)[None]
        V = torch.from_numpy(vd[idx]).permute(1, 0, 2).repeat_interleave(G, dim=0)[None]
        allowed = torch.arange(L)[None, :] <= (L - C + torch.arange(C))[:, None]
        o = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=allowed,
                                                             scale=float(scale))
        out[qo_indptr[b]:qo_indptr[b + 1]] = o[0].permute(1, 0, 2).numpy()
        scores = (Q @ K.transpose(-1, -2))[0] * float(scale)
        scores = scores.masked_fill(~allowed[None], float("-inf"))
        lse[qo_indptr[b]:qo_indptr[b + 1]] = torch.logsumexp(scores, dim=-1).T.numpy()
    return out, lse


def pin_prefill_sdpa(orc, seed=21):
    rng = np.random.default_rng(seed)
    for chunks, contexts, hq, hkv, d in [
        ([5, 1, 0, 7], [9, 6, 4, 7], 8, 2, 16),     # prefix + chunk, one token, none, no prefix
        ([16, 3], [40, 3], 4, 4, 8),                 # G = 1
        ([6], [11], 16, 2, 32),                      # G = 8
    ]:
        q, k, v, qo, kvp, idx, scale = prefill_case(rng, chunks, contexts, hq, hkv, d)
        out, lse = orc.prefill(q, k, v, qo, kvp, idx, hq, hkv, d, scale)
        ro, rl = sdpa_prefill_reference(q, k, v, qo, kvp, idx, hq, hkv, d, scale)
        _close(out, ro, 1e-12, 1e-12, what="prefill vs sdpa out")
        _close(lse, rl, 1e-12, 1e-12, what="prefill vs sdpa lse")


def pin_prefill_brute_force(orc):
    """Two query tokens over three listed slots, one KV head shared by two query
    heads, head_dim 4: the definition written out with math.exp."""
    rng = np.random.default_rng(31)
    q, k, v, qo, kvp, idx, scale = prefill_case(rng, [2], [3], 2, 1, 4, extra_slots=2)
    out, lse = orc.prefill(q, k, v, qo, kvp, idx, 2, 1, 4, scale)
    qd, kd, vd = widen(q), widen(k), widen(v)
    for c in range(2):
        pos = 3 - 2 + c
        for h in range(2):
            s = [scale * sum(qd[c, h, t] * kd[idx[j], 0, t] for t in range(4))
                 for j in range(pos + 1)]
            m = max(s)
            tot = sum(math.exp(x - m) for x in s)
            want_lse = m + math.log(tot)
            assert abs(lse[c, h] - want_lse) < 1e-12, (c, h)
            for t in range(4):
                want = sum(math.exp(s[j] - want_lse) * vd[idx[j], 0, t] for j in range(pos + 1))
                assert abs(out[c, h, t] - want) < 1e-12, (c, h, t)


def pin_prefill_first_token(orc):
    """A chunk with no prefix (C = L): its first query sees only entry 0."""
    rng = np.random.default_rng(32)
    q, k, v, qo, kvp, idx, scale = prefill_case(rng, [4], [4], 4, 2, 8)
    out, lse = orc.prefill(q, k, v, qo, kvp, idx, 4, 2, 8, scale)
    qd, kd, vd = widen(q), widen(k), widen(v)
    for h in range(4):
        g = h // 2
        assert np.array_equal(out[0, h], vd[idx[0], g]), h
        s0 = scale * float(np.dot(qd[0, h], kd[idx[0], g]))
        assert abs(lse[0, h] - s0) < 1e-12


def pin_prefill_causality(orc, seed=33):
    """Rows after a query's position do not change its result; the row at it does."""
    rng = np.random.default_rng(seed)
    chunks, contexts = [3], [8]
    q, k, v, qo, kvp, idx, scale = prefill_case(rng, chunks, contexts, 4, 2, 8)
    base_o, base_l = orc.prefill(q, k, v, qo, kvp, idx, 4, 2, 8, scale)
    pos0 = 8 - 3  # position of the chunk's first query
    k2, v2 = k.copy(), v.copy()
    for j in range(pos0 + 1, 8):
        k2[idx[j]] = bf16_bits_of(rng.standard_normal(k.shape[1:]) * 3)
        v2[idx[j]] = bf16_bits_of(rng.standard_normal(v.shape[1:]) * 3)
    o2, l2 = orc.prefill(q, k2, v2, qo, kvp, idx, 4, 2, 8, scale)
    assert np.array_equal(o2[0], base_o[0]) and np.array_equal(l2[0], base_l[0])
    assert not np.allclose(o2[1:], base_o[1:]), "later queries see those rows"
    v3 = v.copy()
    v3[idx[pos0]] = bf16_bits_of(rng.standard_normal(v.shape[1:]) * 3)
    o3, _ = orc.prefill(q, k, v3, qo, kvp, idx, 4, 2, 8, scale)
    assert not np.allclose(o3[0], base_o[0]), "a query sees the row at its own position"


def pin_prefill_chunk_cut(orc, seed=34):
    """Cutting a chunk in two gives the same rows: the last C2 queries of a chunk of
    C over L entries equal a chunk of C2 over the same L entries."""
    rng = np.random.default_rng(seed)
    q, k, v, qo, kvp, idx, scale = prefill_case(rng, [9], [20], 8, 2, 16)
    full_o, full_l = orc.prefill(q, k, v, qo, kvp, idx, 8, 2, 16, scale)
    tail_o, tail_l = orc.prefill(q[5:], k, v, np.array([0, 4], np.int32), kvp, idx, 8, 2, 16,
                                 scale)
    assert np.array_equal(tail_o, full_o[5:]) and np.array_equal(tail_l, full_l[5:])


def pin_prefill_one_token_chunks(orc, seed=35):
    """Chunks of one token are decode (whose own pins hold on the decode oracle)."""
    rng = np.random.default_rng(seed)
    q, k, v, qo, kvp, idx, scale = prefill_case(rng, [1, 1, 1], [5, 1, 12], 8, 2, 16)
    po, pl = orc.prefill(q, k, v, qo, kvp, idx, 8, 2, 16, scale)
    do, dl = orc.decode(q, k, v, kvp, idx, 8, 2, 16, scale)
    assert np.array_equal(po, do) or np.allclose(po, do, rtol=1e-14, atol=1e-14)
    assert np.allclose(pl, dl, rtol=1e-14, atol=1e-14)


PREFILL_PINS = [pin_prefill_sdpa, pin_prefill_brute_force, pin_prefill_first_token,
                pin_prefill_causality, pin_prefill_chunk_cut, pin_prefill_one_token_chunks]

ALL_PINS = [pin_golden, pin_sdpa, pin_numpy_brute_force, pin_single_token, pin_zero_query, pin_identical_v,
            pin_permutation, pin_split_merge, pin_gqa_equal_queries, pin_empty,
            pin_lse_statistics, pin_append] + PREFILL_PINS
