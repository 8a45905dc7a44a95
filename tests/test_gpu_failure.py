"""Failure detection on the GPU without a fault: an injected stall makes every
pipeline wait of one attention launch run out (each is bounded at 1 s). The launch
must end on its own, report through the plan's status word, and leave the context
usable: the next launch with the same plan is correct and reports 0."""
import time

import numpy as np
import pytest
import torch

import workloads
from test_gpu_parity import assert_parity, oracle_reference, to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_gqa_tokentokvpool_gb300 import build
    build.build()
    import paged_kv_gqa_tokentokvpool_gb300 as m
    return m


@pytest.mark.parametrize("lengths", [[3000, 17, 900, 1], [500, 17, 900, 1], [100] * 8],
                         ids=["persistent_grid", "single_launch", "single_launch_8"])
def test_expired_waits_set_the_status_word_and_the_context_survives(pkv, lengths):
    """The second and third workloads' plans are small enough for the single-launch
    cluster kernel (the third, 8 requests, on clusters of 8 where clusters of 16 for
    all of them do not fit), whose CTAs also meet at cluster barriers after the bounded
    waits have run out."""
    wl = workloads.scattered_workload(lengths, seed=61)
    t = workloads.layer_tensors(wl, 0, device="cpu", poison_unreferenced=True)
    dev = torch.device("cuda")
    kp, vp = t.k_pool.to(dev), t.v_pool.to(dev)
    ip = torch.from_numpy(wl.kv_indptr).to(dev)
    idx = torch.from_numpy(wl.kv_indices).to(dev)
    slots = torch.from_numpy(wl.append_slots).to(dev)
    pkv.kvpool_append(kp, vp, slots, t.k_new.to(dev), t.v_new.to(dev))
    plan = pkv.paged_decode_plan_create(wl.batch, wl.total_tokens, 32, 8, 128)
    assert plan.single_launch() == (wl.total_tokens <= 2048)
    pkv.paged_decode_plan(plan, wl.kv_indptr)
    q = t.q.to(dev)
    out = torch.zeros(wl.batch, 32, 128, dtype=torch.bfloat16, device=dev)
    lse = torch.zeros(wl.batch, 32, dtype=torch.float32, device=dev)
    torch.cuda.synchronize()
    assert plan.status() == 0
    pkv.pkv_inject_stall(1)
    try:
        t0 = time.perf_counter()
        pkv.paged_decode_attn(q, kp, vp, ip, idx, wl.batch, 32, 8, 128, wl.sm_scale, out, lse,
                              plan)
        torch.cuda.synchronize()  # ends by itself once the bounded waits expire
        waited = time.perf_counter() - t0
    finally:
        pkv.pkv_inject_stall(0)
    assert plan.status() != 0, "an expired wait must be reported"
    assert waited > 0.5, "the waits should have run to their bound"
    # the same plan and context still work, and report a clean launch
    pkv.paged_decode_attn(q, kp, vp, ip, idx, wl.batch, 32, 8, 128, wl.sm_scale, out, lse, plan)
    torch.cuda.synchronize()
    assert plan.status() == 0
    ref_out, ref_lse = oracle_reference(wl, t)
    assert_parity(to_f64(out), lse.cpu().numpy(), ref_out, ref_lse, what="after the stall")


def test_prefill_expired_waits_set_the_status_word_and_the_context_survives(pkv):
    """The same for the chunked-prefill kernel (tcgen05, tensor memory): the stalled
    launch ends by itself, frees its tensor memory on that path (the next launch
    allocates it again), and the next launch is correct with status 0."""
    import oracle
    from test_gpu_parity import bits
    pw = workloads.prefill_workload([40, 7], [300, 50], seed=62)
    q, kp, vp, kn, vn = workloads.prefill_tensors(pw, 0, device="cpu", poison_unreferenced=True)
    dev = torch.device("cuda")
    kp_d, vp_d = kp.to(dev), vp.to(dev)
    pkv.kvpool_append(kp_d, vp_d, torch.from_numpy(pw.chunk_slots).to(dev), kn.to(dev), vn.to(dev))
    plan = pkv.paged_prefill_plan_create(pw.batch, pw.total_q, 32, 8, 128)
    pkv.paged_prefill_plan(plan, pw.qo_indptr, pw.kv_indptr)
    args = (q.to(dev), kp_d, vp_d, torch.from_numpy(pw.qo_indptr).to(dev),
            torch.from_numpy(pw.kv_indptr).to(dev), torch.from_numpy(pw.kv_indices).to(dev),
            pw.batch, 32, 8, 128, pw.sm_scale)
    out = torch.zeros(pw.total_q, 32, 128, dtype=torch.bfloat16, device=dev)
    lse = torch.zeros(pw.total_q, 32, dtype=torch.float32, device=dev)
    torch.cuda.synchronize()
    assert plan.status() == 0
    pkv.pkv_inject_stall(1)
    try:
        t0 = time.perf_counter()
        pkv.paged_prefill_attn(*args, out, lse, plan)
        torch.cuda.synchronize()  # ends by itself once the bounded waits expire
        waited = time.perf_counter() - t0
    finally:
        pkv.pkv_inject_stall(0)
    assert plan.status() != 0, "an expired wait must be reported"
    assert waited > 0.5, "the waits should have run to their bound"
    pkv.paged_prefill_attn(*args, out, lse, plan)
    torch.cuda.synchronize()
    assert plan.status() == 0
    ref_out, ref_lse = oracle.prefill(
        bits(q), oracle.append(bits(kp), pw.chunk_slots, bits(kn)),
        oracle.append(bits(vp), pw.chunk_slots, bits(vn)), pw.qo_indptr, pw.kv_indptr,
        pw.kv_indices, 32, 8, 128, pw.sm_scale)
    assert_parity(to_f64(out), lse.cpu().numpy(), ref_out, ref_lse, what="prefill after the stall")
