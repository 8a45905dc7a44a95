"""Chunked-prefill attention on the GPU against the fp64 oracle (parity tests).

Every case follows a prefill step's flow: the chunk's K/V rows are appended to the
pool with kvpool_append, the step is planned (paged_prefill_plan) and the chunk
attends causally over its request's slot list (paged_prefill_attn). Pool slots no
request lists hold bf16 NaN, and so do the chunk's slots before the append, so a
stray or early read shows as NaN. Tolerances are those of the decode parity tests.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from test_gpu_parity import assert_parity, bits, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_gqa_tokentokvpool_gb300 import build
    build.build()
    import paged_kv_gqa_tokentokvpool_gb300 as m
    return m


def run_prefill(pkv, pw, layer=0, debug=False):
    """GPU out/lse of one layer of a prefill workload, and the pools after the append."""
    q, kp, vp, kn, vn = workloads.prefill_tensors(pw, layer, device="cpu",
                                                  poison_unreferenced=True)
    dev = torch.device("cuda")
    B, Hq, Hkv, D, NQ = pw.batch, pw.n_qo_heads, pw.n_kv_heads, pw.head_dim, pw.total_q
    kp_d, vp_d = kp.to(dev), vp.to(dev)
    slots = torch.from_numpy(pw.chunk_slots).to(dev)
    if NQ:
        pkv.kvpool_append(kp_d, vp_d, slots, kn.to(dev), vn.to(dev))
    plan = pkv.paged_prefill_plan_create(max(B, 1), max(NQ, 1), Hq, Hkv, D)
    pkv.paged_prefill_plan(plan, pw.qo_indptr, pw.kv_indptr)
    out = torch.full((max(NQ, 1), Hq, D), float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full((max(NQ, 1), Hq), float("nan"), dtype=torch.float32, device=dev)
    idx = torch.from_numpy(pw.kv_indices if pw.kv_indices.size else np.zeros(1, np.int32)).to(dev)
    pkv.pkv_set_debug_checks(debug)
    try:
        pkv.paged_prefill_attn(q.to(dev) if NQ else out, kp_d, vp_d,
                               torch.from_numpy(pw.qo_indptr).to(dev),
                               torch.from_numpy(pw.kv_indptr).to(dev), idx, B, Hq, Hkv, D,
                               pw.sm_scale, out, lse, plan)
    finally:
        pkv.pkv_set_debug_checks(False)
    torch.cuda.synchronize()
    assert plan.status() == 0, "a pipeline wait of the prefill kernel expired"
    return out[:NQ], lse[:NQ], (q, kp, vp, kn, vn), (kp_d, vp_d)


def oracle_prefill(pw, tensors, rows=None):
    """Oracle out/lse (all chunk rows) from the generated pre-append tensors."""
    q, kp, vp, kn, vn = tensors
    k_after = oracle.append(bits(kp), pw.chunk_slots, bits(kn))
    v_after = oracle.append(bits(vp), pw.chunk_slots, bits(vn))
    return oracle.prefill(bits(q), k_after, v_after, pw.qo_indptr, pw.kv_indptr, pw.kv_indices,
                          pw.n_qo_heads, pw.n_kv_heads, pw.head_dim, pw.sm_scale)


PREFILL_CASES = [
    # (chunks, contexts, Hq, Hkv, D)
    ([64], [64], 32, 8, 128),                            # whole prompt, no prefix
    ([512, 64, 1, 0, 100], [700, 64, 3000, 5, 100], 32, 8, 128),
    ([17, 33], [40, 200], 8, 8, 128),                    # G = 1
    ([9, 70], [9, 500], 16, 8, 128),                     # G = 2
    ([13, 5], [100, 5], 64, 8, 128),                     # G = 8
    ([1, 1, 1], [5, 1, 300], 32, 8, 128),                # one-token chunks
    ([64, 31], [1000, 31], 16, 4, 256),                  # head_dim 256, G = 4
    ([8, 3], [40, 8], 8, 1, 256),                        # head_dim 256, G = 8, one KV head
    ([40], [40], 4, 4, 256),                             # head_dim 256, G = 1
    ([200, 7], [4000, 2500], 16, 2, 128),                # G = 8, long ranges split
    ([300, 5], [5000, 3000], 16, 4, 256),                # head_dim 256, long ranges split
    ([100], [6000], 8, 8, 128),                          # G = 1, long range split
    # K/V tiles are 128 entries at head_dim 128 and 64 at 256, units 128 / G tokens:
    # contexts at and around tile edges, chunks one token over a unit
    ([33, 32, 31], [128, 129, 127], 32, 8, 128),         # G = 4: units of 32 tokens
    ([17, 16], [256, 255], 64, 8, 128),                  # G = 8: units of 16 tokens
    ([129, 128], [257, 384], 8, 8, 128),                 # G = 1: units of 128 tokens
    ([65, 64], [64 + 65, 192], 16, 8, 128),              # G = 2: units of 64 tokens
    ([33, 1], [65, 63], 16, 4, 256),                     # head_dim 256 around 64-entry tiles
    ([65, 64], [129, 64], 8, 4, 256),                    # head_dim 256, G = 2
]


@pytest.mark.parametrize("case", range(len(PREFILL_CASES)))
def test_prefill_small_cases(pkv, case):
    chunks, contexts, hq, hkv, d = PREFILL_CASES[case]
    pw = workloads.prefill_workload(chunks, contexts, n_qo_heads=hq, n_kv_heads=hkv,
                                    head_dim=d, seed=900 + case)
    out, lse, tensors, (kp_d, _) = run_prefill(pkv, pw, debug=True)
    ref_out, ref_lse = oracle_prefill(pw, tensors)
    assert_parity(to_f64(out), lse.cpu().numpy(), ref_out, ref_lse, what=f"prefill case {case}")
    # the append wrote the chunk's rows bit-exactly
    k_after = oracle.append(bits(tensors[1]), pw.chunk_slots, bits(tensors[3]))
    assert np.array_equal(bits(kp_d), k_after)


def test_prefill_plan_reused_across_layers(pkv):
    """One plan serves every layer of the step (different q and pools per layer)."""
    pw = workloads.prefill_workload([100, 37], [300, 37], layers=3, seed=77)
    dev = torch.device("cuda")
    plan = pkv.paged_prefill_plan_create(2, pw.total_q, 32, 8, 128)
    pkv.paged_prefill_plan(plan, pw.qo_indptr, pw.kv_indptr)
    qo = torch.from_numpy(pw.qo_indptr).to(dev)
    kv = torch.from_numpy(pw.kv_indptr).to(dev)
    idx = torch.from_numpy(pw.kv_indices).to(dev)
    for layer in range(3):
        q, kp, vp, kn, vn = workloads.prefill_tensors(pw, layer, poison_unreferenced=True)
        kp_d, vp_d = kp.to(dev), vp.to(dev)
        pkv.kvpool_append(kp_d, vp_d, torch.from_numpy(pw.chunk_slots).to(dev), kn.to(dev),
                          vn.to(dev))
        out = torch.empty(pw.total_q, 32, 128, dtype=torch.bfloat16, device=dev)
        pkv.paged_prefill_attn(q.to(dev), kp_d, vp_d, qo, kv, idx, 2, 32, 8, 128, pw.sm_scale,
                               out, None, plan)
        torch.cuda.synchronize()
        ref_out, ref_lse = oracle_prefill(pw, (q, kp, vp, kn, vn))
        assert_parity(to_f64(out), ref_lse, ref_out, ref_lse, what=f"layer {layer}")
    assert plan.status() == 0


def test_prefill_rejects_bad_calls(pkv):
    plan = pkv.paged_prefill_plan_create(4, 1000, 32, 8, 128)
    with pytest.raises(pkv.PkvError) as e:  # chunk longer than the slot list
        pkv.paged_prefill_plan(plan, np.array([0, 10], np.int32), np.array([0, 9], np.int32))
    assert e.value.code == pkv.PKV_ERR_INVALID_ARG
    with pytest.raises(pkv.PkvError) as e:  # more query tokens than the plan holds
        pkv.paged_prefill_plan(plan, np.array([0, 1001], np.int32), np.array([0, 2000], np.int32))
    assert e.value.code == pkv.PKV_ERR_PLAN
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_prefill_plan_create(4, 1000, 30, 8, 128)
    assert e.value.code == pkv.PKV_ERR_UNSUPPORTED
    pkv.paged_prefill_plan(plan, np.array([0, 5, 9], np.int32), np.array([0, 50, 60], np.int32))
    dev = torch.device("cuda")
    z = torch.zeros(16, 32, 128, dtype=torch.bfloat16, device=dev)
    pool = torch.zeros(64, 8, 128, dtype=torch.bfloat16, device=dev)
    ip = torch.zeros(3, dtype=torch.int32, device=dev)
    with pytest.raises(pkv.PkvError) as e:  # batch differs from the plan's
        pkv.paged_prefill_attn(z, pool, pool, ip, ip, ip, 3, 32, 8, 128, 0.1, z, None, plan)
    assert e.value.code == pkv.PKV_ERR_PLAN
    with pytest.raises(pkv.PkvError) as e:  # shape differs from the plan's
        pkv.paged_prefill_attn(z, pool, pool, ip, ip, ip, 2, 16, 8, 128, 0.1, z, None, plan)
    assert e.value.code == pkv.PKV_ERR_PLAN
    pkv.pkv_set_debug_checks(True)
    try:  # device offsets that disagree with the plan's host copies
        with pytest.raises(pkv.PkvError) as e:
            pkv.paged_prefill_attn(z, pool, pool, ip, ip, ip, 2, 32, 8, 128, 0.1, z, None, plan)
        assert e.value.code == pkv.PKV_ERR_INDEX
    finally:
        pkv.pkv_set_debug_checks(False)
    torch.cuda.synchronize()
    assert torch.all(z == 0), "a rejected call must not have launched"


def test_prefill_empty_step(pkv):
    pw = workloads.prefill_workload([0, 0], [5, 0], seed=3)
    out, lse, _, _ = run_prefill(pkv, pw)
    assert out.numel() == 0


@pytest.mark.parametrize("config_no", [1, 2, 3])
def test_prefill_full_size_sampled(pkv, config_no):
    """The benchmark's prefill workloads at full size (layer 0): every row of the
    chunk of the request with the longest context (every unit of it at the full
    tile count, and for the 64-token chunks of config 2 its split ranges and their
    merge), every row of the smallest request's chunk, and the first and last 16
    rows of every other chunk (by causality, the first rows need only the list up
    to their positions and the last rows only a shorter chunk over the whole
    list)."""
    pw = workloads.prefill_config(config_no)
    out, lse, tensors, _ = run_prefill(pkv, pw)
    q, kp, vp, kn, vn = tensors
    k_after = oracle.append(bits(kp), pw.chunk_slots, bits(kn))
    v_after = oracle.append(bits(vp), pw.chunk_slots, bits(vn))
    qb = bits(q)
    smallest = int(np.argmin(pw.contexts))
    longest = int(np.argmax(pw.contexts))
    for b in range(pw.batch):
        C, L = int(pw.chunks[b]), int(pw.contexts[b])
        q0, k0 = int(pw.qo_indptr[b]), int(pw.kv_indptr[b])
        idx = pw.kv_indices[k0:k0 + L]
        whole = b == longest or (b == smallest and config_no == 1)
        pieces = [(0, C)] if whole else [(0, 16), (C - 16, C)]
        for c0, c1 in pieces:
            # rows c0 .. c1 of the chunk: a chunk of c1 - c0 tokens over the first
            # L - C + c1 list entries
            ref_o, ref_l = oracle.prefill(qb[q0 + c0:q0 + c1], k_after, v_after,
                                          np.array([0, c1 - c0], np.int32),
                                          np.array([0, L - C + c1], np.int32), idx[:L - C + c1],
                                          pw.n_qo_heads, pw.n_kv_heads, pw.head_dim, pw.sm_scale)
            assert_parity(to_f64(out[q0 + c0:q0 + c1]), lse[q0 + c0:q0 + c1].cpu().numpy(),
                          ref_o, ref_l, what=f"prefill config {config_no} request {b} rows {c0}-{c1}")


def test_prefill_graph_replay_steps(pkv):
    """Several steps of back-to-back layers replayed from a CUDA graph, as the
    benchmark runs them (64-token chunks over long contexts: split ranges and the
    merge kernel): every layer's results equal the oracle's and no pipeline wait
    expires."""
    pw = workloads.prefill_workload([64, 64, 64], [9000, 3000, 700], layers=3, seed=31)
    dev = torch.device("cuda")
    plan = pkv.paged_prefill_plan_create(pw.batch, pw.total_q, 32, 8, 128)
    qo = torch.from_numpy(pw.qo_indptr).to(dev)
    kv = torch.from_numpy(pw.kv_indptr).to(dev)
    idx = torch.from_numpy(pw.kv_indices).to(dev)
    slots = torch.from_numpy(pw.chunk_slots).to(dev)
    layers = [workloads.prefill_tensors(pw, l, poison_unreferenced=True) for l in range(3)]
    dev_t = [tuple(x.to(dev) for x in t) for t in layers]
    outs = [torch.empty(pw.total_q, 32, 128, dtype=torch.bfloat16, device=dev) for _ in range(3)]
    lses = [torch.empty(pw.total_q, 32, dtype=torch.float32, device=dev) for _ in range(3)]

    def step_layers():
        for (q, kp, vp, kn, vn), o, l in zip(dev_t, outs, lses):
            pkv.kvpool_append(kp, vp, slots, kn, vn)
            pkv.paged_prefill_attn(q, kp, vp, qo, kv, idx, pw.batch, 32, 8, 128, pw.sm_scale, o,
                                   l, plan)

    pkv.paged_prefill_plan(plan, pw.qo_indptr, pw.kv_indptr)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step_layers()  # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step_layers()
    for _ in range(4):
        pkv.paged_prefill_plan(plan, pw.qo_indptr, pw.kv_indptr)
        g.replay()
    torch.cuda.synchronize()
    assert plan.status() == 0, "a pipeline wait of the prefill kernel expired"
    for layer in range(3):
        ref_out, ref_lse = oracle_prefill(pw, layers[layer])
        assert_parity(to_f64(outs[layer]), lses[layer].cpu().numpy(), ref_out, ref_lse,
                      what=f"graph layer {layer}")


def test_prefill_and_decode_overlap_on_two_streams(pkv):
    """A mixed batch's two paths at once: decode steps of one model's layers on one
    stream and chunked-prefill steps of another's on a second stream, enqueued
    alternately with no host wait, so the kernels overlap on the GPU (each with its
    own plan). Both results must equal the oracle's and both status words stay 0."""
    dev = torch.device("cuda")
    # decode: 16 requests of 300-5000 tokens
    wl = workloads.scattered_workload([300 + 311 * i for i in range(16)], seed=71)
    t = workloads.layer_tensors(wl, 0, device="cpu", poison_unreferenced=True)
    kp_dec, vp_dec = t.k_pool.to(dev), t.v_pool.to(dev)
    q_dec = t.q.to(dev)
    ip = torch.from_numpy(wl.kv_indptr).to(dev)
    idx = torch.from_numpy(wl.kv_indices).to(dev)
    slots = torch.from_numpy(wl.append_slots).to(dev)
    k_new, v_new = t.k_new.to(dev), t.v_new.to(dev)
    out_dec = torch.full((wl.batch, 32, 128), float("nan"), dtype=torch.bfloat16, device=dev)
    lse_dec = torch.full((wl.batch, 32), float("nan"), dtype=torch.float32, device=dev)
    dplan = pkv.paged_decode_plan_create(wl.batch, wl.total_tokens, 32, 8, 128)
    # prefill: two chunks of 200 and 64 tokens over contexts of 3000 and 900
    pw = workloads.prefill_workload([200, 64], [3000, 900], seed=72)
    q, kp, vp, kn, vn = workloads.prefill_tensors(pw, 0, device="cpu", poison_unreferenced=True)
    kp_pf, vp_pf = kp.to(dev), vp.to(dev)
    pslots = torch.from_numpy(pw.chunk_slots).to(dev)
    kn_d, vn_d, q_pf = kn.to(dev), vn.to(dev), q.to(dev)
    out_pf = torch.full((pw.total_q, 32, 128), float("nan"), dtype=torch.bfloat16, device=dev)
    lse_pf = torch.full((pw.total_q, 32), float("nan"), dtype=torch.float32, device=dev)
    pplan = pkv.paged_prefill_plan_create(pw.batch, pw.total_q, 32, 8, 128)
    qo_d = torch.from_numpy(pw.qo_indptr).to(dev)
    kv_d = torch.from_numpy(pw.kv_indptr).to(dev)
    pidx = torch.from_numpy(pw.kv_indices).to(dev)
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    for _ in range(6):  # repeated steps (the appends rewrite the same rows)
        pkv.paged_decode_plan(dplan, wl.kv_indptr, stream=s1)
        pkv.paged_prefill_plan(pplan, pw.qo_indptr, pw.kv_indptr, stream=s2)
        for _layer in range(4):
            pkv.paged_decode_append_attn(q_dec, kp_dec, vp_dec, ip, idx, slots, k_new, v_new,
                                         wl.batch, 32, 8, 128, wl.sm_scale, out_dec, lse_dec,
                                         dplan, stream=s1)
            pkv.kvpool_append(kp_pf, vp_pf, pslots, kn_d, vn_d, stream=s2)
            pkv.paged_prefill_attn(q_pf, kp_pf, vp_pf, qo_d, kv_d, pidx, pw.batch, 32, 8, 128,
                                   pw.sm_scale, out_pf, lse_pf, pplan, stream=s2)
    torch.cuda.synchronize()
    assert dplan.status() == 0 and pplan.status() == 0
    from test_gpu_parity import oracle_reference
    ref_out, ref_lse = oracle_reference(wl, t)
    assert_parity(to_f64(out_dec), lse_dec.cpu().numpy(), ref_out, ref_lse, what="decode beside prefill")
    ref_out, ref_lse = oracle_prefill(pw, (q, kp, vp, kn, vn))
    assert_parity(to_f64(out_pf), lse_pf.cpu().numpy(), ref_out, ref_lse, what="prefill beside decode")
