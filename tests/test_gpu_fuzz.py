"""Seeded random parity sweep on the GPU: decode and chunked-prefill steps of random
shapes (every supported head_dim, group size and KV-head count), random batch sizes,
log-uniform context lengths with empty contexts among them, random plan modes (the
automatic choice, the persistent grid, single launch, early gather), fused or separate
append, and sometimes shared prefixes. Each case is checked against the fp64 oracle with
the tolerances of the other parity tests; pool slots no request lists hold NaN.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from test_gpu_parity import assert_parity, bits, oracle_reference, to_f64

pytestmark = pytest.mark.gpu

SHAPES = [  # (n_qo_heads, n_kv_heads, head_dim)
    (32, 8, 128), (64, 8, 128), (16, 8, 128), (8, 8, 128), (16, 4, 128), (8, 2, 128),
    (4, 1, 128), (16, 4, 256), (32, 4, 256), (8, 2, 256), (8, 1, 256), (4, 4, 256),
]


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_gqa_tokentokvpool_gb300 import build
    build.build()
    import paged_kv_gqa_tokentokvpool_gb300 as m
    return m


def random_lengths(rng, batch, longest):
    lengths = np.rint(np.exp(rng.uniform(0, np.log(longest), batch))).astype(np.int64)
    lengths[rng.random(batch) < 0.1] = 0  # some empty contexts
    return lengths


@pytest.mark.parametrize("seed", range(24))
def test_decode_random_steps(pkv, seed):
    rng = np.random.default_rng(7000 + seed)
    hq, hkv, d = SHAPES[seed % len(SHAPES)]
    batch = int(rng.integers(1, 48))
    dev = torch.device("cuda")
    shared = None
    if d == 128 and hkv in (4, 8) and seed % 3 == 0:  # shapes with a shared-prefix kernel
        n_groups = int(rng.integers(1, 4))
        gsize = int(rng.integers(2, 12))
        prefixes = [int(x) for x in rng.integers(1, 4000, n_groups)]
        suffixes = [int(x) for x in rng.integers(1, 1500, n_groups * gsize)]
        wl = workloads.prefix_shared_workload(prefixes, suffixes, gsize, n_qo_heads=hq,
                                              n_kv_heads=hkv, head_dim=d, seed=seed)
        shared = (np.arange(0, gsize * n_groups + 1, gsize, dtype=np.int32),
                  np.array(prefixes, np.int32))
    else:
        lengths = random_lengths(rng, batch, [600, 6000, 40000][seed % 3])
        wl = workloads.scattered_workload(lengths, n_qo_heads=hq, n_kv_heads=hkv, head_dim=d,
                                          seed=seed)
    t = workloads.layer_tensors(wl, 0, device="cpu", poison_unreferenced=True)
    kp, vp = t.k_pool.to(dev), t.v_pool.to(dev)
    out = torch.full((wl.batch, hq, d), float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full((wl.batch, hq), float("nan"), dtype=torch.float32, device=dev)
    ip = torch.from_numpy(wl.kv_indptr).to(dev)
    idx = torch.from_numpy(wl.kv_indices if wl.kv_indices.size else np.zeros(1, np.int32)).to(dev)
    slots = torch.from_numpy(wl.append_slots).to(dev)
    plan = pkv.paged_decode_plan_create(wl.batch, max(wl.total_tokens, 1), hq, hkv, d)
    mode = ["auto", "persistent", "single_launch"][int(rng.integers(0, 3))]
    flags = {"auto": 0, "persistent": pkv.PKV_PLAN_PERSISTENT,
             "single_launch": pkv.PKV_PLAN_SINGLE_LAUNCH}[mode]
    fused = bool(rng.integers(0, 2)) and len(wl.append_slots) == wl.batch
    if fused and rng.integers(0, 2):
        flags |= pkv.PKV_PLAN_EARLY_GATHER  # the pool rows and ids are final before the plan
    try:
        plan.set_flags(flags)
    except pkv.PkvError as e:  # too many requests for the resident clusters
        assert e.code == pkv.PKV_ERR_UNSUPPORTED and mode == "single_launch"
        plan.set_flags(flags & ~pkv.PKV_PLAN_SINGLE_LAUNCH)
    if shared is not None:
        pkv.paged_decode_plan_shared(plan, wl.kv_indptr, shared[0], shared[1])
    else:
        pkv.paged_decode_plan(plan, wl.kv_indptr)
    if fused:
        pkv.paged_decode_append_attn(t.q.to(dev), kp, vp, ip, idx, slots, t.k_new.to(dev),
                                     t.v_new.to(dev), wl.batch, hq, hkv, d, wl.sm_scale, out, lse,
                                     plan)
    else:
        if len(wl.append_slots):
            pkv.kvpool_append(kp, vp, slots, t.k_new.to(dev), t.v_new.to(dev))
        pkv.paged_decode_attn(t.q.to(dev), kp, vp, ip, idx, wl.batch, hq, hkv, d, wl.sm_scale,
                              out, lse, plan)
    torch.cuda.synchronize()
    assert plan.status() == 0
    ref_out, ref_lse = oracle_reference(wl, t)
    assert_parity(to_f64(out), lse.cpu().numpy(), ref_out, ref_lse,
                  what=f"seed {seed} ({hq}/{hkv}/{d}, batch {wl.batch}, {mode}, fused {fused}, "
                       f"shared {shared is not None})")


@pytest.mark.parametrize("seed", range(12))
def test_prefill_random_steps(pkv, seed):
    rng = np.random.default_rng(8000 + seed)
    hq, hkv, d = SHAPES[(5 * seed) % len(SHAPES)]
    batch = int(rng.integers(1, 6))
    chunks = [int(x) for x in rng.choice([1, 7, 33, 64, 200, 512], batch)]
    contexts = [c + int(rng.integers(0, [300, 3000, 12000][seed % 3])) for c in chunks]
    pw = workloads.prefill_workload(chunks, contexts, n_qo_heads=hq, n_kv_heads=hkv, head_dim=d,
                                    seed=seed)
    q, kp, vp, kn, vn = workloads.prefill_tensors(pw, 0, device="cpu", poison_unreferenced=True)
    dev = torch.device("cuda")
    kp_d, vp_d = kp.to(dev), vp.to(dev)
    pkv.kvpool_append(kp_d, vp_d, torch.from_numpy(pw.chunk_slots).to(dev), kn.to(dev), vn.to(dev))
    plan = pkv.paged_prefill_plan_create(pw.batch, pw.total_q, hq, hkv, d)
    pkv.paged_prefill_plan(plan, pw.qo_indptr, pw.kv_indptr)
    out = torch.full((pw.total_q, hq, d), float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full((pw.total_q, hq), float("nan"), dtype=torch.float32, device=dev)
    pkv.paged_prefill_attn(q.to(dev), kp_d, vp_d, torch.from_numpy(pw.qo_indptr).to(dev),
                           torch.from_numpy(pw.kv_indptr).to(dev),
                           torch.from_numpy(pw.kv_indices).to(dev), pw.batch, hq, hkv, d,
                           pw.sm_scale, out, lse, plan)
    torch.cuda.synchronize()
    assert plan.status() == 0
    k_after = oracle.append(bits(kp), pw.chunk_slots, bits(kn))
    v_after = oracle.append(bits(vp), pw.chunk_slots, bits(vn))
    ref_out, ref_lse = oracle.prefill(bits(q), k_after, v_after, pw.qo_indptr, pw.kv_indptr,
                                      pw.kv_indices, hq, hkv, d, pw.sm_scale)
    assert_parity(to_f64(out), lse.cpu().numpy(), ref_out, ref_lse,
                  what=f"prefill seed {seed} ({hq}/{hkv}/{d}, chunks {chunks})")
