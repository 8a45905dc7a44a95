"""paged_decode_attn_static, the entry point for callers that cannot allocate device
memory (an engine whose KV pool already holds all free HBM, a runtime whose allocator
must own every buffer, a path that must not hit cudaMalloc's implicit synchronisation).

It is checked through the C ABI against the planned entry point, paged_decode_attn,
on two calls in a row whose work lists and split workspaces differ, so a second call
that read stale scratch left by the first would show up. Tolerances are the ones of
the parity tests: |out - ref| <= 1e-2 + 1e-2 |ref|, |lse - ref| <= 1e-3, and empty
contexts give out = 0, lse = -inf on both. This file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_gqa_tokentokvpool_gb300 import build
    build.build()
    import paged_kv_gqa_tokentokvpool_gb300 as m
    return m


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def test_static_scratch_entry_matches_planned_entry(pkv):
    lib = pkv.library()
    dev = torch.device("cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    calls = [([5000, 3, 900, 0, 20000, 64], 32, 8, 128, 11),
             ([1, 700, 12000, 9, 4097], 16, 4, 256, 12)]
    for i, (lengths, hq, hkv, d, seed) in enumerate(calls):
        wl = workloads.scattered_workload(lengths, n_qo_heads=hq, n_kv_heads=hkv, head_dim=d,
                                          seed=seed)
        t = workloads.layer_tensors(wl, 0, device="cpu")
        q, kp, vp = t.q.to(dev), t.k_pool.to(dev), t.v_pool.to(dev)
        indptr = torch.from_numpy(wl.kv_indptr).to(dev)
        indices = torch.from_numpy(wl.kv_indices).to(dev)
        B = wl.batch
        out_ref = torch.empty(B, hq, d, dtype=torch.bfloat16, device=dev)
        lse_ref = torch.empty(B, hq, dtype=torch.float32, device=dev)
        out = torch.full((B, hq, d), float("nan"), dtype=torch.bfloat16, device=dev)
        lse = torch.full((B, hq), float("nan"), dtype=torch.float32, device=dev)

        plan = pkv.paged_decode_plan_create(B, wl.total_tokens, hq, hkv, d)
        pkv.paged_decode_plan(plan, wl.kv_indptr)
        pkv.paged_decode_attn(q, kp, vp, indptr, indices, B, hq, hkv, d, wl.sm_scale, out_ref,
                              lse_ref, plan)

        ip_host = np.ascontiguousarray(wl.kv_indptr, dtype=np.int32)
        rc = lib.paged_decode_attn_static(
            _p(q), _p(kp), _p(vp), ip_host.ctypes.data_as(ctypes.c_void_p), _p(indptr),
            _p(indices), B, hq, hkv, d, ctypes.c_float(wl.sm_scale), _p(out), _p(lse), stream)
        assert rc == 0, pkv.pkv_last_error()
        torch.cuda.synchronize()

        ref = out_ref.double().cpu().numpy()
        got = out.double().cpu().numpy()
        rl = lse_ref.double().cpu().numpy()
        gl = lse.double().cpu().numpy()
        empty = np.isneginf(rl)
        assert np.array_equal(np.isneginf(gl), empty), f"call {i}: empty contexts differ"
        assert np.all(got[empty] == 0)
        assert np.all(np.isfinite(got))
        assert np.all(np.abs(got - ref) <= 1e-2 + 1e-2 * np.abs(ref)), f"call {i}: out differs"
        assert np.all(np.abs(gl[~empty] - rl[~empty]) <= 1e-3), f"call {i}: lse differs"
        assert plan.status() == 0


def test_static_scratch_entry_rejects_oversized_steps(pkv):
    lib = pkv.library()
    dev = torch.device("cuda")
    buf = torch.zeros(64, dtype=torch.bfloat16, device=dev)
    ip = torch.zeros(5001, dtype=torch.int32, device=dev)
    ip_host = np.zeros(5001, np.int32)  # 5000 empty requests x 2 head groups > 4096 pairs
    rc = lib.paged_decode_attn_static(_p(buf), _p(buf), _p(buf),
                                      ip_host.ctypes.data_as(ctypes.c_void_p), _p(ip), _p(ip),
                                      5000, 32, 8, 128, ctypes.c_float(0.1), _p(buf), None,
                                      ctypes.c_void_p(0))
    assert rc == pkv.PKV_ERR_PLAN
    assert "static maximum" in pkv.pkv_last_error()
