"""CUDA path vs the fp64 oracle, through the C ABI (needs a GPU).

Tolerances (the decode contract): |out - ref| <= 1e-2 + 1e-2 * |ref| elementwise on
bf16 out, |lse - ref| <= 1e-3 on fp32 lse, and bit-exact pool rows after append.
Pools are NaN-poisoned outside the listed slots, so any stray read shows up as a
NaN output. The oracle always works from the generated inputs and applies its own
append; nothing the CUDA path wrote is fed to it.
"""
import math

import numpy as np
import pytest
import torch

import workloads
import oracle

pytestmark = pytest.mark.gpu

OUT_ATOL, OUT_RTOL, LSE_ATOL = 1e-2, 1e-2, 1e-3


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_gqa_tokentokvpool_gb300 import build
    build.build()
    import paged_kv_gqa_tokentokvpool_gb300 as m
    return m


def bits(t):
    return workloads.bf16_bits(t)


def to_f64(t_bf16):
    return t_bf16.float().double().cpu().numpy()


def assert_parity(out, lse, ref_out, ref_lse, what=""):
    out = np.asarray(out, np.float64)
    lse = np.asarray(lse, np.float64)
    assert out.shape == ref_out.shape and lse.shape == ref_lse.shape
    empty = np.isneginf(ref_lse)
    assert np.all(np.isneginf(lse[empty])), f"{what}: empty contexts need lse = -inf"
    assert np.all(out[empty] == 0), f"{what}: empty contexts need out = 0"
    assert np.all(np.isfinite(out)), f"{what}: non-finite out (stray read of a poisoned slot?)"
    assert np.all(np.isfinite(lse[~empty])), f"{what}: non-finite lse"
    err = np.abs(out - ref_out)
    bad = err > OUT_ATOL + OUT_RTOL * np.abs(ref_out)
    assert not bad.any(), (f"{what}: out mismatch at {np.argwhere(bad)[:5].tolist()}, "
                           f"max err {err.max():.3g}")
    lerr = np.abs(lse[~empty] - ref_lse[~empty])
    assert lerr.size == 0 or lerr.max() <= LSE_ATOL, f"{what}: lse max err {lerr.max():.3g}"


def oracle_reference(wl, t, layer_pools=None):
    """Oracle out/lse for one layer from generated (pre-append) tensors."""
    k_bits = bits(t.k_pool) if layer_pools is None else layer_pools[0]
    v_bits = bits(t.v_pool) if layer_pools is None else layer_pools[1]
    k_after = oracle.append(k_bits, wl.append_slots, bits(t.k_new))
    v_after = oracle.append(v_bits, wl.append_slots, bits(t.v_new))
    return oracle.decode(bits(t.q), k_after, v_after, wl.kv_indptr, wl.kv_indices,
                         wl.n_qo_heads, wl.n_kv_heads, wl.head_dim, wl.sm_scale)


def run_small(pkv, wl, layer=0, debug=False, persistent=False):
    """Append + plan + attention for one layer of a small workload; returns GPU
    results, generated tensors and the GPU pools after append. persistent: keep the
    persistent grid even when the plan is small enough for single-launch mode."""
    t = workloads.layer_tensors(wl, layer, device="cpu", poison_unreferenced=True)
    dev = torch.device("cuda")
    k_pool, v_pool = t.k_pool.to(dev), t.v_pool.to(dev)
    q = t.q.to(dev)
    out = torch.full((wl.batch, wl.n_qo_heads, wl.head_dim), float("nan"),
                     dtype=torch.bfloat16, device=dev)
    lse = torch.full((wl.batch, wl.n_qo_heads), float("nan"), dtype=torch.float32, device=dev)
    indptr = torch.from_numpy(wl.kv_indptr).to(dev)
    indices = torch.from_numpy(wl.kv_indices).to(dev)
    if indices.numel() == 0:
        indices = torch.zeros(1, dtype=torch.int32, device=dev)
    slots = torch.from_numpy(wl.append_slots).to(dev)
    pkv.pkv_set_debug_checks(debug)
    try:
        pkv.kvpool_append(k_pool, v_pool, slots, t.k_new.to(dev), t.v_new.to(dev))
        plan = pkv.paged_decode_plan_create(max(wl.batch, 1), max(wl.total_tokens, 1),
                                            wl.n_qo_heads, wl.n_kv_heads, wl.head_dim)
        if persistent:
            plan.set_flags(pkv.PKV_PLAN_PERSISTENT)
        pkv.paged_decode_plan(plan, wl.kv_indptr)
        pkv.paged_decode_attn(q, k_pool, v_pool, indptr, indices, wl.batch, wl.n_qo_heads,
                              wl.n_kv_heads, wl.head_dim, wl.sm_scale, out, lse, plan)
        torch.cuda.synchronize()
    finally:
        pkv.pkv_set_debug_checks(False)
    return out, lse, t, k_pool, v_pool, plan


SMALL_CASES = [
    # (lengths, Hq, Hkv, D)
    ([1], 32, 8, 128),
    ([0], 32, 8, 128),
    ([0, 1, 0, 2, 3], 32, 8, 128),
    ([17, 300, 1000, 5, 64, 65, 31, 33], 32, 8, 128),
    ([4097], 32, 8, 128),
    ([20000, 7, 3000], 32, 8, 128),
    ([1, 255, 256, 257, 12345], 16, 4, 256),
    ([9000, 0, 40], 16, 4, 256),
    ([100, 2000], 8, 8, 128),
    ([100, 2000], 16, 8, 128),
    ([100, 5000], 64, 8, 128),
    ([77, 3001], 8, 1, 256),
    ([513] * 40, 32, 8, 128),
    (list(range(0, 3000, 15)), 32, 8, 128),
    ([131072], 32, 8, 128),
    ([60000, 1, 16, 17, 15], 16, 2, 256),
    ([3000, 70], 4, 4, 128),
    # groups of fewer than four KV heads at head_dim 128 (two and four consumer warps
    # per head) and of one at head_dim 256
    ([300, 4000, 1], 4, 2, 128),
    ([2500, 9, 700], 8, 1, 128),
    ([5000, 33], 4, 1, 256),
    # large batches of short contexts: many whole units per CTA, empty ones among them
    ([1] * 4096, 32, 8, 128),
    ([(7 * i) % 65 for i in range(2000)], 16, 4, 256),
]


@pytest.mark.parametrize("persistent", [False, True], ids=["auto", "persistent"])
@pytest.mark.parametrize("case", range(len(SMALL_CASES)))
def test_decode_small_cases(pkv, case, persistent):
    """Every case planned by default (single launch where the plan is small enough)
    and on the persistent grid."""
    lengths, hq, hkv, d = SMALL_CASES[case]
    wl = workloads.scattered_workload(lengths, n_qo_heads=hq, n_kv_heads=hkv, head_dim=d,
                                      seed=100 + case, k_scale=1.0)
    out, lse, t, _, _, plan = run_small(pkv, wl, debug=(case % 2 == 0), persistent=persistent)
    ref_out, ref_lse = oracle_reference(wl, t)
    assert_parity(to_f64(out), lse.cpu().numpy(), ref_out, ref_lse, what=f"case {case}")
    assert plan.status() == 0


def test_append_bit_exact(pkv):
    wl = workloads.scattered_workload([3, 0, 700, 1, 64] * 7, seed=7)
    out, lse, t, k_pool, v_pool, _ = run_small(pkv, wl)
    want_k = oracle.append(bits(t.k_pool), wl.append_slots, bits(t.k_new))
    want_v = oracle.append(bits(t.v_pool), wl.append_slots, bits(t.v_new))
    assert np.array_equal(bits(k_pool), want_k)
    assert np.array_equal(bits(v_pool), want_v)


def test_append_zero_rows_is_noop(pkv):
    dev = torch.device("cuda")
    pool = torch.randn(64, 8, 128, device=dev).to(torch.bfloat16)
    before = pool.clone()
    empty_rows = torch.empty(0, 8, 128, dtype=torch.bfloat16, device=dev)
    pkv.kvpool_append(pool, pool, torch.empty(0, dtype=torch.int32, device=dev), empty_rows,
                      empty_rows)
    torch.cuda.synchronize()
    assert torch.equal(pool.view(torch.int16), before.view(torch.int16))


def test_plan_reused_across_layers_and_steps(pkv):
    """One plan per step serves every layer; re-planning with other lengths works."""
    dev = torch.device("cuda")
    plan = pkv.paged_decode_plan_create(6, 40000, 32, 8, 128)
    for step, lengths in enumerate([[5000, 3, 900], [1, 1, 1, 1, 1, 30000], [0, 2048]]):
        wl = workloads.scattered_workload(lengths, layers=3, seed=200 + step)
        pkv.paged_decode_plan(plan, wl.kv_indptr)
        indptr = torch.from_numpy(wl.kv_indptr).to(dev)
        indices = torch.from_numpy(wl.kv_indices).to(dev)
        for layer in range(3):
            t = workloads.layer_tensors(wl, layer, device="cpu", poison_unreferenced=True)
            kp, vp = t.k_pool.to(dev), t.v_pool.to(dev)
            slots = torch.from_numpy(wl.append_slots).to(dev)
            pkv.kvpool_append(kp, vp, slots, t.k_new.to(dev), t.v_new.to(dev))
            out = torch.empty(wl.batch, 32, 128, dtype=torch.bfloat16, device=dev)
            lse = torch.empty(wl.batch, 32, dtype=torch.float32, device=dev)
            pkv.paged_decode_attn(t.q.to(dev), kp, vp, indptr, indices, wl.batch, 32, 8, 128,
                                  wl.sm_scale, out, lse, plan)
            torch.cuda.synchronize()
            ref_out, ref_lse = oracle_reference(wl, t)
            assert_parity(to_f64(out), lse.cpu().numpy(), ref_out, ref_lse,
                          what=f"step {step} layer {layer}")


def test_lse_optional(pkv):
    wl = workloads.scattered_workload([300, 5000], seed=9)
    t = workloads.layer_tensors(wl, 0, device="cpu")
    dev = torch.device("cuda")
    kp, vp = t.k_pool.to(dev), t.v_pool.to(dev)
    out = torch.empty(2, 32, 128, dtype=torch.bfloat16, device=dev)
    plan = pkv.paged_decode_plan_create(2, wl.total_tokens, 32, 8, 128)
    pkv.paged_decode_plan(plan, wl.kv_indptr)
    pkv.paged_decode_attn(t.q.to(dev), kp, vp, torch.from_numpy(wl.kv_indptr).to(dev),
                          torch.from_numpy(wl.kv_indices).to(dev), 2, 32, 8, 128, wl.sm_scale,
                          out, None, plan)
    torch.cuda.synchronize()
    ref_out, _ = oracle.decode(bits(t.q), bits(t.k_pool), bits(t.v_pool), wl.kv_indptr,
                               wl.kv_indices, 32, 8, 128, wl.sm_scale)
    got = to_f64(out)
    assert np.all(np.abs(got - ref_out) <= OUT_ATOL + OUT_RTOL * np.abs(ref_out))


def test_errors_do_not_launch(pkv):
    dev = torch.device("cuda")
    plan = pkv.paged_decode_plan_create(4, 1000, 32, 8, 128)
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_decode_plan(plan, np.array([0, 10, 5], np.int32))
    assert e.value.code == pkv.PKV_ERR_INVALID_ARG
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_decode_plan(plan, np.array([0, 10, 2000], np.int32))
    assert e.value.code == pkv.PKV_ERR_PLAN
    pkv.paged_decode_plan(plan, np.array([0, 10, 20], np.int32))
    q = torch.zeros(3, 32, 128, dtype=torch.bfloat16, device=dev)
    pool = torch.zeros(64, 8, 128, dtype=torch.bfloat16, device=dev)
    ip = torch.tensor([0, 10, 20, 20], dtype=torch.int32, device=dev)
    idx = torch.arange(20, dtype=torch.int32, device=dev)
    out = torch.zeros(3, 32, 128, dtype=torch.bfloat16, device=dev)
    with pytest.raises(pkv.PkvError) as e:  # batch differs from the plan's
        pkv.paged_decode_attn(q, pool, pool, ip, idx, 3, 32, 8, 128, 0.1, out, None, plan)
    assert e.value.code == pkv.PKV_ERR_PLAN
    with pytest.raises(pkv.PkvError) as e:  # shape differs from the plan's
        pkv.paged_decode_attn(q[:2], pool, pool, ip[:3], idx, 2, 16, 8, 128, 0.1, out, None, plan)
    assert e.value.code == pkv.PKV_ERR_PLAN
    # debug checks catch an indptr that disagrees with the plan and a bad slot
    pkv.pkv_set_debug_checks(True)
    try:
        with pytest.raises(pkv.PkvError) as e:
            pkv.paged_decode_attn(q[:2], pool, pool, torch.tensor([0, 10, 19], dtype=torch.int32,
                                  device=dev), idx, 2, 32, 8, 128, 0.1, out, None, plan)
        assert e.value.code == pkv.PKV_ERR_INDEX
        with pytest.raises(pkv.PkvError) as e:
            pkv.kvpool_append(pool, pool, torch.tensor([3, 64], dtype=torch.int32, device=dev),
                              pool[:2], pool[:2])
        assert e.value.code == pkv.PKV_ERR_INDEX
        with pytest.raises(pkv.PkvError) as e:
            pkv.kvpool_append(pool, pool, torch.tensor([3, 3], dtype=torch.int32, device=dev),
                              pool[:2], pool[:2])
        assert e.value.code == pkv.PKV_ERR_INDEX
        # a host array where device memory belongs (it would fault the kernel); the
        # binding refuses CPU tensors itself, so these go through the C ABI directly
        import ctypes
        lib = pkv.library()
        vp = lambda t: ctypes.c_void_p(t.data_ptr())
        stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        q_host = torch.zeros(2, 32, 128, dtype=torch.bfloat16)
        rc = lib.paged_decode_attn(vp(q_host), vp(pool), vp(pool), vp(ip), vp(idx), 2, 32, 8, 128,
                                   ctypes.c_float(0.1), vp(out), None, plan.handle, stream)
        assert rc == pkv.PKV_ERR_INVALID_ARG and "q is not device memory" in pkv.pkv_last_error()
        pool_host = pool.cpu()
        rc = lib.kvpool_append(vp(pool_host), vp(pool), vp(idx), vp(pool), vp(pool), 1, 8, 128, 64,
                               stream)
        assert rc == pkv.PKV_ERR_INVALID_ARG and "k_pool" in pkv.pkv_last_error()
        pw = workloads.prefill_workload([5], [9], seed=3)
        pplan = pkv.paged_prefill_plan_create(1, 5, 32, 8, 128)
        pkv.paged_prefill_plan(pplan, pw.qo_indptr, pw.kv_indptr)
        pout = torch.zeros(5, 32, 128, dtype=torch.bfloat16, device=dev)
        qo_d = torch.from_numpy(pw.qo_indptr).to(dev)
        kv_d = torch.from_numpy(pw.kv_indptr).to(dev)
        rc = lib.paged_prefill_attn(vp(torch.zeros(5, 32, 128, dtype=torch.bfloat16)), vp(pool),
                                    vp(pool), vp(qo_d), vp(kv_d), vp(idx), 1, 32, 8, 128,
                                    ctypes.c_float(0.1), vp(pout), None, pplan.handle, stream)
        assert rc == pkv.PKV_ERR_INVALID_ARG and "q is not device memory" in pkv.pkv_last_error()
        assert torch.all(pout == 0)
    finally:
        pkv.pkv_set_debug_checks(False)
    torch.cuda.synchronize()
    assert torch.all(out == 0), "a rejected call must not have launched"


# ---------------------------------------------------------------------------
# the benchmark's five workloads at full size, in the benchmark's launch setup
# ---------------------------------------------------------------------------

FULL = {1: None, 2: None, 3: [0, 35], 4: [0, 7], 5: None}


@pytest.mark.parametrize("fused", [True, False], ids=["fused_append", "separate_append"])
@pytest.mark.parametrize("config_no", sorted(FULL))
def test_full_size_config(pkv, config_no, fused):
    import bench
    wl = workloads.config_workload(config_no)
    st = bench.StepState(wl, layers=FULL[config_no], poison_unreferenced=True, fused=fused)
    assert st.fused == fused
    assert (st.sharing is not None) == (config_no == 3)
    uniq, inv = np.unique(wl.kv_indices, return_inverse=True)
    compact = inv.astype(np.int32)
    uniq_dev = torch.from_numpy(uniq.astype(np.int64)).cuda()
    # the appended slots' positions in the compacted pool
    pos = {int(s): i for i, s in enumerate(uniq)}
    app_compact = np.array([pos[int(s)] for s in wl.append_slots], np.int32)
    before = []
    for i in range(len(st.layer_ids)):
        before.append((bits(st.k_pool[i].index_select(0, uniq_dev)),
                       bits(st.v_pool[i].index_select(0, uniq_dev))))
    st.run()
    torch.cuda.synchronize()
    for i, layer in enumerate(st.layer_ids):
        kb, vb = before[i]
        k_after = oracle.append(kb, app_compact, bits(st.k_new[i]))
        v_after = oracle.append(vb, app_compact, bits(st.v_new[i]))
        # append: bit-exact on every listed row (appended and untouched alike)
        assert np.array_equal(bits(st.k_pool[i].index_select(0, uniq_dev)), k_after)
        assert np.array_equal(bits(st.v_pool[i].index_select(0, uniq_dev)), v_after)
        ref_out, ref_lse = oracle.decode(bits(st.q[i]), k_after, v_after, wl.kv_indptr, compact,
                                         wl.n_qo_heads, wl.n_kv_heads, wl.head_dim, wl.sm_scale)
        assert_parity(to_f64(st.out[i]), st.lse[i].cpu().numpy(), ref_out, ref_lse,
                      what=f"config {config_no} layer {layer}")
        # loose statistical sanity of the generator scaling: E[lse] ~ ln L + sigma^2/2
        sigma2 = wl.k_scale ** 2
        expect = np.log(wl.lengths)[:, None] + sigma2 / 2
        assert abs(float(np.mean(ref_lse - expect))) < 0.2
    assert st.plan.status() == 0


def test_end_to_end_host_path_matches_device_path(pkv):
    import bench
    wl = workloads.config_workload(2)
    st = bench.StepState(wl, layers=[0, 1])
    st.run()
    torch.cuda.synchronize()
    dev_out = [o.clone() for o in st.out]
    io = bench.HostIO(st)
    io.run()
    torch.cuda.synchronize()
    for a, b in zip(io.out, dev_out):
        assert torch.equal(a.view(torch.int16), b.cpu().view(torch.int16))


def test_graph_replay_after_replanning(pkv):
    """A CUDA graph of the layer loop stays valid when the next step re-plans with
    other context lengths: the grid is fixed and the kernel reads the plan from
    the plan's own device buffers."""
    dev = torch.device("cuda")
    B, layers, S = 4, 2, 1 << 16
    steps = [[3000, 17, 0, 9000], [1, 20000, 513, 64], [700, 700, 700, 700]]
    max_tokens = max(sum(s) for s in steps)
    plan = pkv.paged_decode_plan_create(B, max_tokens, 32, 8, 128)
    q = torch.empty(layers, B, 32, 128, dtype=torch.bfloat16, device=dev)
    kp = torch.empty(layers, S, 8, 128, dtype=torch.bfloat16, device=dev)
    vp = torch.empty_like(kp)
    kn = torch.empty(layers, B, 8, 128, dtype=torch.bfloat16, device=dev)
    vn = torch.empty_like(kn)
    out = torch.empty(layers, B, 32, 128, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(layers, B, 32, dtype=torch.float32, device=dev)
    indptr = torch.zeros(B + 1, dtype=torch.int32, device=dev)
    indices = torch.zeros(max_tokens, dtype=torch.int32, device=dev)
    slots = torch.zeros(B, dtype=torch.int32, device=dev)
    graph = None
    for step, lengths in enumerate(steps):
        wl = workloads.scattered_workload(lengths, pool_slots=S, layers=layers, seed=300 + step)
        tens = [workloads.layer_tensors(wl, l, device="cpu") for l in range(layers)]
        nonempty = [b for b in range(B) if lengths[b] > 0]
        for l, t in enumerate(tens):
            q[l].copy_(t.q)
            kp[l].copy_(t.k_pool)
            vp[l].copy_(t.v_pool)
            kn[l].zero_()
            vn[l].zero_()
            kn[l][nonempty] = t.k_new.to(dev)
            vn[l][nonempty] = t.v_new.to(dev)
        unused = np.setdiff1d(np.arange(S), wl.kv_indices)[:B].astype(np.int32)
        app = unused.copy()  # rows of empty requests land on slots nobody lists
        app[nonempty] = wl.append_slots
        slots.copy_(torch.from_numpy(app))
        indptr.copy_(torch.from_numpy(wl.kv_indptr))
        indices[:wl.total_tokens].copy_(torch.from_numpy(wl.kv_indices))
        pkv.paged_decode_plan(plan, wl.kv_indptr)
        if graph is None:
            def body():
                for l in range(layers):
                    pkv.kvpool_append(kp[l], vp[l], slots, kn[l], vn[l])
                    pkv.paged_decode_attn(q[l], kp[l], vp[l], indptr, indices, B, 32, 8, 128,
                                          wl.sm_scale, out[l], lse[l], plan)
            body()
            torch.cuda.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                body()
            # the capture did not run the body; make it run from a fresh pool state
            for l, t in enumerate(tens):
                kp[l].copy_(t.k_pool)
                vp[l].copy_(t.v_pool)
        graph.replay()
        torch.cuda.synchronize()
        for l, t in enumerate(tens):
            ref_out, ref_lse = oracle_reference(wl, t)
            assert_parity(to_f64(out[l]), lse[l].cpu().numpy(), ref_out, ref_lse,
                          what=f"graph step {step} layer {l}")
    assert plan.status() == 0


@pytest.mark.parametrize("shared", [False, True], ids=["plain", "shared_prefix"])
def test_early_gather_graph_steps(pkv, shared):
    """PKV_PLAN_EARLY_GATHER with the fused append, layer loop in a CUDA graph,
    re-planned every step: each step's rows are written before its plan upload, as
    the flag requires. Results equal the oracle's and, bit for bit, those of the
    same plan without the flag."""
    dev = torch.device("cuda")
    layers = 3
    if shared:
        wls = [workloads.prefix_shared_workload([1500, 40], [3, 700, 1, 90, 2000, 5, 17, 64], 4,
                                                pool_slots=1 << 15, layers=layers, seed=700 + i)
               for i in range(2)]
    else:
        wls = [workloads.scattered_workload(l, pool_slots=1 << 15, layers=layers, seed=700 + i)
               for i, l in enumerate([[3000, 17, 1, 9000], [1, 20000, 513, 64]])]
    B = wls[0].batch
    max_tokens = max(w.total_tokens for w in wls)
    S = wls[0].pool_slots
    q = torch.empty(layers, B, 32, 128, dtype=torch.bfloat16, device=dev)
    kp = torch.empty(layers, S, 8, 128, dtype=torch.bfloat16, device=dev)
    vp = torch.empty_like(kp)
    kn = torch.empty(layers, B, 8, 128, dtype=torch.bfloat16, device=dev)
    vn = torch.empty_like(kn)
    out = torch.empty(layers, B, 32, 128, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(layers, B, 32, dtype=torch.float32, device=dev)
    indptr = torch.zeros(B + 1, dtype=torch.int32, device=dev)
    indices = torch.zeros(max_tokens, dtype=torch.int32, device=dev)
    slots = torch.zeros(B, dtype=torch.int32, device=dev)
    plans = {}
    for early in (True, False):
        plans[early] = pkv.paged_decode_plan_create(B, max_tokens, 32, 8, 128)
        if early:
            plans[early].set_flags(pkv.PKV_PLAN_EARLY_GATHER)

    def plan_step(plan, wl):
        if shared:
            gs = wl.meta["group_size"]
            sp = np.arange(0, B + 1, gs, dtype=np.int32)
            pkv.paged_decode_plan_shared(plan, wl.kv_indptr, sp,
                                         np.array(wl.meta["prefix_lens"], np.int32))
        else:
            pkv.paged_decode_plan(plan, wl.kv_indptr)

    def body(plan):
        for l in range(layers):
            pkv.paged_decode_append_attn(q[l], kp[l], vp[l], indptr, indices, slots, kn[l], vn[l],
                                         B, 32, 8, 128, wls[0].sm_scale, out[l], lse[l], plan)

    results = {}
    for early in (True, False):
        graph = None
        for step, wl in enumerate(wls):
            tens = [workloads.layer_tensors(wl, l, device="cpu") for l in range(layers)]

            def load_inputs():
                for l, t in enumerate(tens):  # every row written before the plan upload
                    q[l].copy_(t.q)
                    kp[l].copy_(t.k_pool)
                    vp[l].copy_(t.v_pool)
                    kn[l].copy_(t.k_new)
                    vn[l].copy_(t.v_new)
                slots.copy_(torch.from_numpy(wl.append_slots))
                indptr.copy_(torch.from_numpy(wl.kv_indptr))
                indices[:wl.total_tokens].copy_(torch.from_numpy(wl.kv_indices))

            load_inputs()
            plan_step(plans[early], wl)
            if graph is None:
                body(plans[early])
                torch.cuda.synchronize()
                graph = torch.cuda.CUDAGraph()
                with torch.cuda.graph(graph):
                    body(plans[early])
                load_inputs()
                plan_step(plans[early], wl)
            graph.replay()
            torch.cuda.synchronize()
            for l, t in enumerate(tens):
                ref_out, ref_lse = oracle_reference(wl, t)
                assert_parity(to_f64(out[l]), lse[l].cpu().numpy(), ref_out, ref_lse,
                              what=f"early={early} step {step} layer {l}")
                k_after = oracle.append(bits(t.k_pool), wl.append_slots, bits(t.k_new))
                assert np.array_equal(bits(kp[l]), k_after)
            results[(early, step)] = (out.clone(), lse.clone())
        assert plans[early].status() == 0
    for step in range(len(wls)):
        assert torch.equal(results[(True, step)][0].view(torch.int16),
                           results[(False, step)][0].view(torch.int16))
        assert torch.equal(results[(True, step)][1], results[(False, step)][1])


FUSED_CASES = [
    ([1], 32, 8, 128),
    ([1, 2, 3, 17, 300, 1000, 5, 64, 65], 32, 8, 128),
    ([20000, 7, 3000], 32, 8, 128),
    ([1, 255, 256, 257, 12345], 16, 4, 256),
    ([100, 2000], 8, 8, 128),
    ([100, 5000], 64, 8, 128),
    ([77, 3001], 8, 1, 256),
    ([513] * 40, 32, 8, 128),
]


@pytest.mark.parametrize("case", range(len(FUSED_CASES)))
def test_fused_append_attention(pkv, case):
    """paged_decode_append_attn == kvpool_append then paged_decode_attn (oracle side:
    the oracle's append, then the oracle's attention)."""
    lengths, hq, hkv, d = FUSED_CASES[case]
    wl = workloads.scattered_workload(lengths, n_qo_heads=hq, n_kv_heads=hkv, head_dim=d,
                                      seed=400 + case)
    t = workloads.layer_tensors(wl, 0, device="cpu", poison_unreferenced=True)
    dev = torch.device("cuda")
    kp, vp = t.k_pool.to(dev), t.v_pool.to(dev)
    out = torch.full((wl.batch, hq, d), float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full((wl.batch, hq), float("nan"), dtype=torch.float32, device=dev)
    plan = pkv.paged_decode_plan_create(wl.batch, wl.total_tokens, hq, hkv, d)
    pkv.paged_decode_plan(plan, wl.kv_indptr)
    pkv.pkv_set_debug_checks(case % 2 == 0)
    try:
        pkv.paged_decode_append_attn(t.q.to(dev), kp, vp, torch.from_numpy(wl.kv_indptr).to(dev),
                                     torch.from_numpy(wl.kv_indices).to(dev),
                                     torch.from_numpy(wl.append_slots).to(dev), t.k_new.to(dev),
                                     t.v_new.to(dev), wl.batch, hq, hkv, d, wl.sm_scale, out, lse,
                                     plan)
        torch.cuda.synchronize()
    finally:
        pkv.pkv_set_debug_checks(False)
    k_ref = oracle.append(bits(t.k_pool), wl.append_slots, bits(t.k_new))
    v_ref = oracle.append(bits(t.v_pool), wl.append_slots, bits(t.v_new))
    assert np.array_equal(bits(kp), k_ref) and np.array_equal(bits(vp), v_ref)
    ref_out, ref_lse = oracle.decode(bits(t.q), k_ref, v_ref, wl.kv_indptr, wl.kv_indices, hq,
                                     hkv, d, wl.sm_scale)
    assert_parity(to_f64(out), lse.cpu().numpy(), ref_out, ref_lse, what=f"fused case {case}")
    assert plan.status() == 0


def test_fused_append_rejects_bad_calls(pkv):
    dev = torch.device("cuda")
    wl = workloads.scattered_workload([5, 0, 7], seed=5)
    plan = pkv.paged_decode_plan_create(3, 20, 32, 8, 128)
    pkv.paged_decode_plan(plan, wl.kv_indptr)
    z = torch.zeros(3, 32, 128, dtype=torch.bfloat16, device=dev)
    pool = torch.zeros(64, 8, 128, dtype=torch.bfloat16, device=dev)
    rows = torch.zeros(3, 8, 128, dtype=torch.bfloat16, device=dev)
    ip = torch.from_numpy(wl.kv_indptr).to(dev)
    idx = torch.from_numpy(wl.kv_indices).to(dev)
    slots = torch.zeros(3, dtype=torch.int32, device=dev)
    with pytest.raises(pkv.PkvError) as e:  # request 1 has no newest token
        pkv.paged_decode_append_attn(z, pool, pool, ip, idx, slots, rows, rows, 3, 32, 8, 128,
                                     0.1, z, None, plan)
    assert e.value.code == pkv.PKV_ERR_INVALID_ARG
    wl = workloads.scattered_workload([5, 3, 7], pool_slots=64, seed=6)
    pkv.paged_decode_plan(plan, wl.kv_indptr)
    ip = torch.from_numpy(wl.kv_indptr).to(dev)
    idx = torch.from_numpy(wl.kv_indices).to(dev)
    bad = torch.from_numpy(wl.append_slots[::-1].copy()).to(dev)  # not each request's last slot
    pkv.pkv_set_debug_checks(True)
    try:
        with pytest.raises(pkv.PkvError) as e:
            pkv.paged_decode_append_attn(z, pool, pool, ip, idx, bad, rows, rows, 3, 32, 8, 128,
                                         0.1, z, None, plan)
        assert e.value.code == pkv.PKV_ERR_INDEX
    finally:
        pkv.pkv_set_debug_checks(False)


SHARED_CASES = [
    # (prefix lengths, group size, suffix lengths, Hq, Hkv, D)
    ([300], 4, [5, 1, 700, 64], 32, 8, 128),
    ([3000, 17], 5, [1, 2, 3, 400, 9000, 16, 17, 1, 2, 3], 32, 8, 128),
    ([5000], 8, [64] * 8, 32, 8, 128),
    ([777, 2048], 3, [100, 1, 50, 3000, 2, 8], 64, 8, 128),
    ([4100], 9, list(range(1, 10)), 16, 8, 128),
    ([1000], 17, [1] * 17, 8, 8, 128),
    ([2500], 4, [1, 90, 300, 2], 16, 4, 256),
    # runs longer than one prefix unit (32 / G requests): several units read the prefix
    ([2000], 12, [3, 1, 800, 64, 5, 17, 2, 100, 1, 9, 33, 250], 32, 8, 128),
    ([600, 1500], 9, [1 + 37 * i for i in range(18)], 64, 8, 128),
    ([900], 40, [1 + (7 * i) % 50 for i in range(40)], 8, 8, 128),
    ([1200], 20, [2 + 11 * i for i in range(20)], 16, 8, 128),
    ([3333], 10, [1 + 91 * i for i in range(10)], 16, 4, 128),
]


@pytest.mark.parametrize("fused", [False, True], ids=["attn", "append_attn"])
@pytest.mark.parametrize("case", range(len(SHARED_CASES)))
def test_shared_prefix_plan(pkv, case, fused):
    """paged_decode_plan_shared: prefix units serve several requests; results must
    equal the oracle's (which knows nothing about sharing)."""
    prefixes, gsize, suffixes, hq, hkv, d = SHARED_CASES[case]
    wl = workloads.prefix_shared_workload(prefixes, suffixes, gsize, n_qo_heads=hq,
                                          n_kv_heads=hkv, head_dim=d, seed=500 + case)
    t = workloads.layer_tensors(wl, 0, device="cpu", poison_unreferenced=True)
    dev = torch.device("cuda")
    kp, vp = t.k_pool.to(dev), t.v_pool.to(dev)
    out = torch.full((wl.batch, hq, d), float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full((wl.batch, hq), float("nan"), dtype=torch.float32, device=dev)
    ip = torch.from_numpy(wl.kv_indptr).to(dev)
    idx = torch.from_numpy(wl.kv_indices).to(dev)
    slots = torch.from_numpy(wl.append_slots).to(dev)
    plan = pkv.paged_decode_plan_create(wl.batch, wl.total_tokens, hq, hkv, d)
    plan.set_flags(pkv.PKV_PLAN_PERSISTENT)  # the shared-prefix kernel runs on the persistent grid
    shared_indptr = np.arange(0, gsize * len(prefixes) + 1, gsize, dtype=np.int32)
    pkv.paged_decode_plan_shared(plan, wl.kv_indptr, shared_indptr, np.array(prefixes, np.int32))
    if fused:
        pkv.paged_decode_append_attn(t.q.to(dev), kp, vp, ip, idx, slots, t.k_new.to(dev),
                                     t.v_new.to(dev), wl.batch, hq, hkv, d, wl.sm_scale, out, lse,
                                     plan)
    else:
        pkv.kvpool_append(kp, vp, slots, t.k_new.to(dev), t.v_new.to(dev))
        pkv.paged_decode_attn(t.q.to(dev), kp, vp, ip, idx, wl.batch, hq, hkv, d, wl.sm_scale,
                              out, lse, plan)
    torch.cuda.synchronize()
    ref_out, ref_lse = oracle_reference(wl, t)
    assert_parity(to_f64(out), lse.cpu().numpy(), ref_out, ref_lse, what=f"shared case {case}")
    assert plan.status() == 0
    if d == 128 and hkv == 8:
        assert plan.info()["n_merges"] >= wl.batch  # every member merged its parts


def test_false_sharing_description_is_rejected_with_debug_checks(pkv):
    """paged_decode_plan_shared's precondition (members list the same prefix slot
    ids) is verified by the attention call when debug checks are on: a description
    that kv_indices does not bear out gives PKV_ERR_INDEX and launches nothing."""
    wl = workloads.scattered_workload([400, 500, 300, 600], seed=77)  # nothing shared
    dev = torch.device("cuda")
    t = workloads.layer_tensors(wl, 0, device=dev)
    out = torch.full((wl.batch, 32, 128), float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full((wl.batch, 32), float("nan"), dtype=torch.float32, device=dev)
    ip = torch.from_numpy(wl.kv_indptr).to(dev)
    idx = torch.from_numpy(wl.kv_indices).to(dev)
    slots = torch.from_numpy(wl.append_slots).to(dev)
    plan = pkv.paged_decode_plan_create(wl.batch, wl.total_tokens, 32, 8, 128)
    plan.set_flags(pkv.PKV_PLAN_PERSISTENT)  # the shared-prefix kernel runs on the persistent grid
    # claims requests 0-3 share their first 200 slots
    pkv.paged_decode_plan_shared(plan, wl.kv_indptr, np.array([0, 4], np.int32),
                                 np.array([200], np.int32))
    pkv.pkv_set_debug_checks(True)
    try:
        for fused in (False, True):
            with pytest.raises(pkv.PkvError) as e:
                if fused:
                    pkv.paged_decode_append_attn(t.q, t.k_pool, t.v_pool, ip, idx, slots, t.k_new,
                                                 t.v_new, wl.batch, 32, 8, 128, wl.sm_scale, out,
                                                 lse, plan)
                else:
                    pkv.paged_decode_attn(t.q, t.k_pool, t.v_pool, ip, idx, wl.batch, 32, 8, 128,
                                          wl.sm_scale, out, lse, plan)
            assert e.value.code == pkv.PKV_ERR_INDEX
            assert "shared" in e.value.message
        torch.cuda.synchronize()
        assert torch.isnan(out.float()).all() and torch.isnan(lse).all()  # nothing launched
        # a true description passes the check: requests 0-1 made to share 100 slots
        shared = wl.kv_indices.copy()
        shared[wl.kv_indptr[1]:wl.kv_indptr[1] + 100] = shared[:100]
        idx2 = torch.from_numpy(shared).to(dev)
        pkv.paged_decode_plan_shared(plan, wl.kv_indptr, np.array([0, 2], np.int32),
                                     np.array([100], np.int32))
        pkv.paged_decode_attn(t.q, t.k_pool, t.v_pool, ip, idx2, wl.batch, 32, 8, 128,
                              wl.sm_scale, out, lse, plan)
        torch.cuda.synchronize()
    finally:
        pkv.pkv_set_debug_checks(False)
    assert plan.status() == 0
    assert torch.isfinite(out.float()).all()


def test_host_tier_round_trip_then_attention(pkv):
    """kvpool_offload + kvpool_prefetch are bit-exact row moves through pinned host
    memory; attention over the prefetched slots equals the oracle on the original."""
    dev = torch.device("cuda")
    wl = workloads.scattered_workload([3000, 700, 12000], seed=41)
    t = workloads.layer_tensors(wl, 0, device="cpu", poison_unreferenced=True)
    kp, vp = t.k_pool.to(dev), t.v_pool.to(dev)
    # the cold part of each context: its first half
    cold = np.concatenate([wl.kv_indices[wl.kv_indptr[b]:wl.kv_indptr[b] + wl.lengths[b] // 2]
                           for b in range(wl.batch)]).astype(np.int32)
    n = cold.size
    H = n + 100
    kh = torch.zeros(H, 8, 128, dtype=torch.bfloat16).pin_memory()
    vh = torch.zeros(H, 8, 128, dtype=torch.bfloat16).pin_memory()
    host_slots = np.random.default_rng(3).permutation(H)[:n].astype(np.int32)
    pkv.pkv_set_debug_checks(True)
    try:
        pkv.kvpool_offload(kp, vp, torch.from_numpy(cold).to(dev), kh, vh,
                           torch.from_numpy(host_slots).to(dev))
        torch.cuda.synchronize()
        assert np.array_equal(bits(kh)[host_slots], bits(t.k_pool)[cold])
        assert np.array_equal(bits(vh)[host_slots], bits(t.v_pool)[cold])
        # the device copies are gone (NaN); the rows come back to fresh slots
        kp.view(torch.int16)[torch.from_numpy(cold).long().to(dev)] = workloads.BF16_NAN_BITS
        vp.view(torch.int16)[torch.from_numpy(cold).long().to(dev)] = workloads.BF16_NAN_BITS
        free = np.setdiff1d(np.arange(wl.pool_slots), wl.kv_indices)[:n].astype(np.int32)
        pkv.kvpool_prefetch(kp, vp, torch.from_numpy(free).to(dev), kh, vh,
                            torch.from_numpy(host_slots).to(dev))
        torch.cuda.synchronize()
    finally:
        pkv.pkv_set_debug_checks(False)
    assert np.array_equal(bits(kp)[free], bits(t.k_pool)[cold])
    assert np.array_equal(bits(vp)[free], bits(t.v_pool)[cold])
    remap = dict(zip(cold.tolist(), free.tolist()))
    new_indices = np.array([remap.get(int(s), int(s)) for s in wl.kv_indices], np.int32)
    # attention over the remapped lists (no append here: pools as generated)
    out = torch.empty(wl.batch, 32, 128, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(wl.batch, 32, dtype=torch.float32, device=dev)
    plan = pkv.paged_decode_plan_create(wl.batch, wl.total_tokens, 32, 8, 128)
    pkv.paged_decode_plan(plan, wl.kv_indptr)
    k_ref = bits(t.k_pool).copy()
    v_ref = bits(t.v_pool).copy()
    # the appended slots were never filled here: give them their generated new rows
    k_ref = oracle.append(k_ref, wl.append_slots, bits(t.k_new))
    v_ref = oracle.append(v_ref, wl.append_slots, bits(t.v_new))
    kp.view(torch.int16)[torch.from_numpy(wl.append_slots).long().to(dev)] = \
        torch.from_numpy(bits(t.k_new).view(np.int16)).to(dev)
    vp.view(torch.int16)[torch.from_numpy(wl.append_slots).long().to(dev)] = \
        torch.from_numpy(bits(t.v_new).view(np.int16)).to(dev)
    pkv.paged_decode_attn(t.q.to(dev), kp, vp, torch.from_numpy(wl.kv_indptr).to(dev),
                          torch.from_numpy(new_indices).to(dev), wl.batch, 32, 8, 128, wl.sm_scale,
                          out, lse, plan)
    torch.cuda.synchronize()
    ref_out, ref_lse = oracle.decode(bits(t.q), k_ref, v_ref, wl.kv_indptr, wl.kv_indices, 32, 8,
                                     128, wl.sm_scale)
    assert_parity(to_f64(out), lse.cpu().numpy(), ref_out, ref_lse, what="after prefetch")


SINGLE_LAUNCH_CASES = [
    # (lengths, Hq, Hkv, D): plans small enough for the single-launch cluster kernel
    ([512], 32, 8, 128),
    ([1], 32, 8, 128),
    ([0, 5, 1500], 32, 8, 128),
    ([17, 300, 33], 16, 4, 256),
    ([2000, 1], 8, 8, 128),      # G = 1
    ([700, 64], 64, 8, 128),     # G = 8
    ([100, 2000], 4, 2, 128),    # two KV heads per group
    ([1000], 8, 1, 256),         # one KV head, G = 8
]


@pytest.mark.parametrize("persistent", [False, True], ids=["single_launch", "persistent"])
@pytest.mark.parametrize("fused", [False, True], ids=["attn", "append_attn"])
@pytest.mark.parametrize("case", range(len(SINGLE_LAUNCH_CASES)))
def test_small_step_modes(pkv, case, fused, persistent):
    """A small plan runs its steps as one launch of the cluster kernel (slot-list
    shares per CTA, merged in distributed shared memory); PKV_PLAN_PERSISTENT runs
    the same step on the persistent grid. Both must equal the oracle."""
    lengths, hq, hkv, d = SINGLE_LAUNCH_CASES[case]
    if fused and 0 in lengths:
        pytest.skip("the fused append needs a newest token in every request")
    wl = workloads.scattered_workload(lengths, n_qo_heads=hq, n_kv_heads=hkv, head_dim=d,
                                      seed=700 + case)
    t = workloads.layer_tensors(wl, 0, device="cpu", poison_unreferenced=True)
    dev = torch.device("cuda")
    kp, vp = t.k_pool.to(dev), t.v_pool.to(dev)
    out = torch.full((wl.batch, hq, d), float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full((wl.batch, hq), float("nan"), dtype=torch.float32, device=dev)
    ip = torch.from_numpy(wl.kv_indptr).to(dev)
    idx = torch.from_numpy(wl.kv_indices if wl.kv_indices.size else np.zeros(1, np.int32)).to(dev)
    slots = torch.from_numpy(wl.append_slots).to(dev)
    plan = pkv.paged_decode_plan_create(wl.batch, max(wl.total_tokens, 1), hq, hkv, d)
    flags = pkv.PKV_PLAN_EARLY_GATHER if fused else 0
    plan.set_flags(flags | (pkv.PKV_PLAN_PERSISTENT if persistent else 0))
    assert plan.single_launch() == (not persistent)
    pkv.paged_decode_plan(plan, wl.kv_indptr)
    pkv.pkv_set_debug_checks(True)
    try:
        if fused:
            pkv.paged_decode_append_attn(t.q.to(dev), kp, vp, ip, idx, slots, t.k_new.to(dev),
                                         t.v_new.to(dev), wl.batch, hq, hkv, d, wl.sm_scale, out,
                                         lse, plan)
        else:
            pkv.kvpool_append(kp, vp, slots, t.k_new.to(dev), t.v_new.to(dev))
            pkv.paged_decode_attn(t.q.to(dev), kp, vp, ip, idx, wl.batch, hq, hkv, d, wl.sm_scale,
                                  out, lse, plan)
        torch.cuda.synchronize()
    finally:
        pkv.pkv_set_debug_checks(False)
    assert plan.status() == 0
    ref_out, ref_lse = oracle_reference(wl, t)
    assert_parity(to_f64(out), lse.cpu().numpy(), ref_out, ref_lse,
                  what=f"small case {case} fused={fused} persistent={persistent}")
    k_after = oracle.append(bits(t.k_pool), wl.append_slots, bits(t.k_new))
    assert np.array_equal(bits(kp), k_after)


@pytest.mark.parametrize("lengths", [[1024] * 4, [9000, 5], [1, 2048, 0, 700], [512] * 8,
                                     [300 + 97 * i for i in range(12)],
                                     [200 + 37 * i for i in range(24)]],
                         ids=["four_1k", "one_long", "mixed", "eight_short", "twelve",
                              "twenty_four"])
def test_single_launch_flag(pkv, lengths):
    """PKV_PLAN_SINGLE_LAUNCH: a plan whose max_tokens is beyond the automatic
    single-launch limit runs its steps in that mode all the same (each request split 16
    ways, a CTA's share of 9000 tokens is 36 stages; 8 or 4 ways on clusters of 8 or 4
    for the batches whose clusters of 16 do not all fit); results equal the oracle's."""
    wl = workloads.scattered_workload(lengths, seed=81)
    t = workloads.layer_tensors(wl, 0, device="cpu", poison_unreferenced=True)
    dev = torch.device("cuda")
    kp, vp = t.k_pool.to(dev), t.v_pool.to(dev)
    plan = pkv.paged_decode_plan_create(wl.batch, wl.total_tokens, 32, 8, 128)
    assert not plan.single_launch()  # more than 2048 tokens
    with pytest.raises(pkv.PkvError) as e:
        plan.set_flags(pkv.PKV_PLAN_SINGLE_LAUNCH | pkv.PKV_PLAN_PERSISTENT)
    assert e.value.code == pkv.PKV_ERR_INVALID_ARG
    plan.set_flags(pkv.PKV_PLAN_SINGLE_LAUNCH)
    assert plan.single_launch()
    pkv.paged_decode_plan(plan, wl.kv_indptr)
    out = torch.full((wl.batch, 32, 128), float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full((wl.batch, 32), float("nan"), dtype=torch.float32, device=dev)
    ip = torch.from_numpy(wl.kv_indptr).to(dev)
    idx = torch.from_numpy(wl.kv_indices).to(dev)
    slots = torch.from_numpy(wl.append_slots).to(dev)
    if all(L > 0 for L in lengths):
        pkv.paged_decode_append_attn(t.q.to(dev), kp, vp, ip, idx, slots, t.k_new.to(dev),
                                     t.v_new.to(dev), wl.batch, 32, 8, 128, wl.sm_scale, out, lse,
                                     plan)
    else:
        pkv.kvpool_append(kp, vp, slots, t.k_new.to(dev), t.v_new.to(dev))
        pkv.paged_decode_attn(t.q.to(dev), kp, vp, ip, idx, wl.batch, 32, 8, 128, wl.sm_scale,
                              out, lse, plan)
    torch.cuda.synchronize()
    assert plan.status() == 0
    ref_out, ref_lse = oracle_reference(wl, t)
    assert_parity(to_f64(out), lse.cpu().numpy(), ref_out, ref_lse, what=f"single launch {lengths}")


def test_single_launch_flag_needs_the_clusters(pkv):
    """A plan whose max_batch x KV-head groups exceed the resident clusters refuses the
    flag and keeps its mode."""
    plan = pkv.paged_decode_plan_create(128, 1 << 16, 32, 8, 128)
    with pytest.raises(pkv.PkvError) as e:
        plan.set_flags(pkv.PKV_PLAN_SINGLE_LAUNCH)
    assert e.value.code == pkv.PKV_ERR_UNSUPPORTED
    assert not plan.single_launch()


def test_single_launch_graph_steps(pkv):
    """Small-step mode under CUDA-graph replay: three layers captured once, replayed
    for several steps, each step re-planned on the host (nothing uploaded); every
    layer equals the oracle and no bounded wait expires."""
    wl = workloads.scattered_workload([300, 1200, 40], layers=3, seed=41)
    dev = torch.device("cuda")
    plan = pkv.paged_decode_plan_create(wl.batch, wl.total_tokens, 32, 8, 128)
    plan.set_flags(pkv.PKV_PLAN_EARLY_GATHER)
    assert plan.single_launch()
    ip = torch.from_numpy(wl.kv_indptr).to(dev)
    idx = torch.from_numpy(wl.kv_indices).to(dev)
    slots = torch.from_numpy(wl.append_slots).to(dev)
    layers = [workloads.layer_tensors(wl, l, poison_unreferenced=True) for l in range(3)]
    dt = [(t.q.to(dev), t.k_pool.to(dev), t.v_pool.to(dev), t.k_new.to(dev), t.v_new.to(dev))
          for t in layers]
    outs = [torch.empty(wl.batch, 32, 128, dtype=torch.bfloat16, device=dev) for _ in range(3)]
    lses = [torch.empty(wl.batch, 32, dtype=torch.float32, device=dev) for _ in range(3)]

    def step_layers():
        for (q, kp, vp, kn, vn), o, l in zip(dt, outs, lses):
            pkv.paged_decode_append_attn(q, kp, vp, ip, idx, slots, kn, vn, wl.batch, 32, 8, 128,
                                         wl.sm_scale, o, l, plan)

    pkv.paged_decode_plan(plan, wl.kv_indptr)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step_layers()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step_layers()
    for _ in range(4):
        pkv.paged_decode_plan(plan, wl.kv_indptr)
        g.replay()
    torch.cuda.synchronize()
    assert plan.status() == 0
    for layer in range(3):
        ref_out, ref_lse = oracle_reference(wl, layers[layer])
        assert_parity(to_f64(outs[layer]), lses[layer].cpu().numpy(), ref_out, ref_lse,
                      what=f"single-launch graph layer {layer}")


TIERED_CASES = [
    # (lengths, Hq, Hkv, D, fraction of listed rows kept in host memory)
    ([3000, 17, 900, 5000, 1], 32, 8, 128, 0.4),
    ([1, 700, 12000, 9], 16, 4, 256, 0.25),
    ([4097, 2, 300], 8, 1, 128, 1.0),
    ([20000], 32, 8, 128, 0.05),
]


@pytest.mark.parametrize("case", range(len(TIERED_CASES)))
def test_tiered_attention_reads_host_rows_in_place(pkv, case):
    """paged_decode_attn_tiered: lists that mix HBM slots and host slots (-1 - h). The
    HBM copies of the host-resident rows are NaN, so any read of them from HBM shows;
    results must equal the oracle on the original placement."""
    lengths, hq, hkv, d, frac = TIERED_CASES[case]
    wl = workloads.scattered_workload(lengths, n_qo_heads=hq, n_kv_heads=hkv, head_dim=d,
                                      seed=610 + case)
    t = workloads.layer_tensors(wl, 0, device="cpu", poison_unreferenced=True)
    k_bits = oracle.append(bits(t.k_pool), wl.append_slots, bits(t.k_new))
    v_bits = oracle.append(bits(t.v_pool), wl.append_slots, bits(t.v_new))
    ref_out, ref_lse = oracle.decode(bits(t.q), k_bits, v_bits, wl.kv_indptr, wl.kv_indices,
                                     hq, hkv, d, wl.sm_scale)
    rng = np.random.default_rng(case)
    n = wl.total_tokens
    moved = np.sort(rng.choice(n, size=max(1, int(frac * n)), replace=False))
    host_rows = rng.permutation(len(moved) + 7)[:len(moved)]  # scattered in a larger host pool
    as_bf16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    k_host = torch.full((len(moved) + 7, hkv, d), float("nan"), dtype=torch.bfloat16).pin_memory()
    v_host = torch.full((len(moved) + 7, hkv, d), float("nan"), dtype=torch.bfloat16).pin_memory()
    slots = wl.kv_indices[moved]
    k_host[torch.from_numpy(host_rows)] = as_bf16(k_bits[slots])
    v_host[torch.from_numpy(host_rows)] = as_bf16(v_bits[slots])
    k_dev, v_dev = k_bits.copy(), v_bits.copy()
    k_dev[slots] = workloads.BF16_NAN_BITS
    v_dev[slots] = workloads.BF16_NAN_BITS
    indices = wl.kv_indices.copy()
    indices[moved] = -1 - host_rows.astype(np.int32)
    dev = torch.device("cuda")
    kp, vp = as_bf16(k_dev).to(dev), as_bf16(v_dev).to(dev)
    out = torch.full((wl.batch, hq, d), float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full((wl.batch, hq), float("nan"), dtype=torch.float32, device=dev)
    ip = torch.from_numpy(wl.kv_indptr).to(dev)
    idx = torch.from_numpy(indices).to(dev)
    plan = pkv.paged_decode_plan_create(wl.batch, wl.total_tokens, hq, hkv, d)
    pkv.paged_decode_plan(plan, wl.kv_indptr)
    pkv.pkv_set_debug_checks(True)
    try:
        pkv.paged_decode_attn_tiered(t.q.to(dev), kp, vp, k_host, v_host, ip, idx, wl.batch, hq,
                                     hkv, d, wl.sm_scale, out, lse, plan)
        torch.cuda.synchronize()
    finally:
        pkv.pkv_set_debug_checks(False)
    assert plan.status() == 0
    assert_parity(to_f64(out), lse.cpu().numpy(), ref_out, ref_lse, what=f"tiered case {case}")
    # a second call without debug checks (no host synchronisation in between)
    out2 = torch.full_like(out, float("nan"))
    pkv.paged_decode_attn_tiered(t.q.to(dev), kp, vp, k_host, v_host, ip, idx, wl.batch, hq, hkv,
                                 d, wl.sm_scale, out2, None, plan)
    torch.cuda.synchronize()
    assert torch.equal(out2, out)
    assert plan.status() == 0


@pytest.mark.parametrize("case", range(2))
def test_tiered_attention_with_shared_prefixes(pkv, case):
    """paged_decode_attn_tiered with a paged_decode_plan_shared plan: a third of the
    listed slots (shared prefix rows and private rows alike) live in the host pools,
    their HBM copies NaN, and every member names a moved slot by the same host row, so
    the prefix lists still agree."""
    prefixes, gsize, suffixes = [([2000], 8, [1 + 97 * i for i in range(8)]),
                                 ([700, 3100], 9, [1 + 31 * i for i in range(18)])][case]
    wl = workloads.prefix_shared_workload(prefixes, suffixes, gsize, seed=660 + case)
    t = workloads.layer_tensors(wl, 0, device="cpu", poison_unreferenced=True)
    k_bits = oracle.append(bits(t.k_pool), wl.append_slots, bits(t.k_new))
    v_bits = oracle.append(bits(t.v_pool), wl.append_slots, bits(t.v_new))
    ref_out, ref_lse = oracle.decode(bits(t.q), k_bits, v_bits, wl.kv_indptr, wl.kv_indices,
                                     32, 8, 128, wl.sm_scale)
    rng = np.random.default_rng(case)
    slots = np.unique(wl.kv_indices)
    moved = np.sort(rng.choice(slots, size=len(slots) // 3, replace=False))
    host_row = {int(s): i for i, s in enumerate(rng.permutation(moved))}
    as_bf16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    rows = np.array([host_row[int(s)] for s in moved])
    k_host = torch.full((len(moved), 8, 128), float("nan"), dtype=torch.bfloat16).pin_memory()
    v_host = torch.full((len(moved), 8, 128), float("nan"), dtype=torch.bfloat16).pin_memory()
    k_host[torch.from_numpy(rows)] = as_bf16(k_bits[moved])
    v_host[torch.from_numpy(rows)] = as_bf16(v_bits[moved])
    k_dev, v_dev = k_bits.copy(), v_bits.copy()
    k_dev[moved] = workloads.BF16_NAN_BITS
    v_dev[moved] = workloads.BF16_NAN_BITS
    indices = np.array([-1 - host_row[int(s)] if int(s) in host_row else int(s)
                        for s in wl.kv_indices], np.int32)
    dev = torch.device("cuda")
    out = torch.full((wl.batch, 32, 128), float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full((wl.batch, 32), float("nan"), dtype=torch.float32, device=dev)
    plan = pkv.paged_decode_plan_create(wl.batch, wl.total_tokens, 32, 8, 128)
    plan.set_flags(pkv.PKV_PLAN_PERSISTENT)  # the shared-prefix kernel runs on the persistent grid
    shared_indptr = np.arange(0, gsize * len(prefixes) + 1, gsize, dtype=np.int32)
    pkv.paged_decode_plan_shared(plan, wl.kv_indptr, shared_indptr, np.array(prefixes, np.int32))
    pkv.pkv_set_debug_checks(True)  # also checks that the members' prefix ids agree
    try:
        pkv.paged_decode_attn_tiered(t.q.to(dev), as_bf16(k_dev).to(dev), as_bf16(v_dev).to(dev),
                                     k_host, v_host, torch.from_numpy(wl.kv_indptr).to(dev),
                                     torch.from_numpy(indices).to(dev), wl.batch, 32, 8, 128,
                                     wl.sm_scale, out, lse, plan)
        torch.cuda.synchronize()
    finally:
        pkv.pkv_set_debug_checks(False)
    assert plan.status() == 0
    assert_parity(to_f64(out), lse.cpu().numpy(), ref_out, ref_lse, what=f"tiered shared {case}")


def test_tiered_attention_rejects_bad_host_arguments(pkv):
    wl = workloads.scattered_workload([50, 60], seed=5)
    dev = torch.device("cuda")
    t = workloads.layer_tensors(wl, 0, device=dev)
    ip = torch.from_numpy(wl.kv_indptr).to(dev)
    idx_np = wl.kv_indices.copy()
    idx_np[3] = -20  # host row 19 of a 10-row host pool
    idx = torch.from_numpy(idx_np).to(dev)
    out = torch.full((wl.batch, 32, 128), float("nan"), dtype=torch.bfloat16, device=dev)
    plan = pkv.paged_decode_plan_create(wl.batch, wl.total_tokens, 32, 8, 128)
    pkv.paged_decode_plan(plan, wl.kv_indptr)
    pinned = torch.zeros(10, 8, 128, dtype=torch.bfloat16).pin_memory()
    pageable = torch.zeros(10, 8, 128, dtype=torch.bfloat16)
    with pytest.raises(pkv.PkvError) as e:
        pkv.paged_decode_attn_tiered(t.q, t.k_pool, t.v_pool, pageable, pageable, ip, idx,
                                     wl.batch, 32, 8, 128, wl.sm_scale, out, None, plan)
    assert e.value.code == pkv.PKV_ERR_INVALID_ARG
    pkv.pkv_set_debug_checks(True)
    try:
        with pytest.raises(pkv.PkvError) as e:
            pkv.paged_decode_attn_tiered(t.q, t.k_pool, t.v_pool, pinned, pinned, ip, idx,
                                         wl.batch, 32, 8, 128, wl.sm_scale, out, None, plan)
        assert e.value.code == pkv.PKV_ERR_INDEX
    finally:
        pkv.pkv_set_debug_checks(False)
    torch.cuda.synchronize()
    assert torch.isnan(out.float()).all()  # nothing launched


def test_host_tier_rejects_pageable_and_duplicate_destinations(pkv):
    dev = torch.device("cuda")
    kp = torch.zeros(64, 8, 128, dtype=torch.bfloat16, device=dev)
    pageable = torch.zeros(16, 8, 128, dtype=torch.bfloat16)
    slots = torch.arange(4, dtype=torch.int32, device=dev)
    with pytest.raises(pkv.PkvError) as e:
        pkv.kvpool_offload(kp, kp, slots, pageable, pageable, slots)
    assert e.value.code == pkv.PKV_ERR_INVALID_ARG
    pinned = torch.zeros(16, 8, 128, dtype=torch.bfloat16).pin_memory()
    pkv.pkv_set_debug_checks(True)
    try:
        with pytest.raises(pkv.PkvError) as e:
            pkv.kvpool_prefetch(kp, kp, torch.tensor([1, 1], dtype=torch.int32, device=dev),
                                pinned, pinned, torch.tensor([0, 1], dtype=torch.int32, device=dev))
        assert e.value.code == pkv.PKV_ERR_INDEX
        with pytest.raises(pkv.PkvError) as e:
            pkv.kvpool_offload(kp, kp, slots, pinned, pinned,
                               torch.tensor([0, 1, 2, 16], dtype=torch.int32, device=dev))
        assert e.value.code == pkv.PKV_ERR_INDEX
    finally:
        pkv.pkv_set_debug_checks(False)
