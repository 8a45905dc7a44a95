"""paged_decode_attn_static, the entry point for callers that cannot allocate device
memory (an engine whose KV pool already holds all free HBM, a runtime whose allocator
must own every buffer, a path that must not hit cudaMalloc's implicit synchronisation).

It is checked through the C ABI against the planned entry point, paged_decode_attn,
and against the fp64 oracle, on two calls in a row whose work lists and split
workspaces differ, so a second call that read stale scratch left by the first would
show up; then on calls queued back to back on one stream with no host wait between
them; then that a call under stream capture is refused; then for its status word (an
injected stall must be reported and cleared); and
for allocation: in a fresh process, calls after the first leave the device's free
memory unchanged, and with eager module loading so does the first. Tolerances are the
ones of the parity tests: |out - ref| <= 1e-2 + 1e-2 |ref|, |lse - ref| <= 1e-3, and
empty contexts give out = 0, lse = -inf. This file is named to be collected last.
"""
import ctypes
import os
import subprocess
import sys
import textwrap

import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (lengths, n_qo_heads, n_kv_heads, head_dim, seed): different shapes, so the second
# call's work list, partial slots and workspace layout differ from the first's
CALLS = [([5000, 3, 900, 0, 20000, 64], 32, 8, 128, 11),
         ([1, 700, 12000, 9, 4097], 16, 4, 256, 12)]


@pytest.fixture(scope="module")
def pkv():
    from paged_kv_gqa_tokentokvpool_gb300 import build
    build.build()
    import paged_kv_gqa_tokentokvpool_gb300 as m
    return m


@pytest.fixture(scope="module")
def orc():
    import oracle
    return oracle.default()


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


class Case:
    """Device inputs of one call, the planned entry point's outputs and the oracle's."""

    def __init__(self, pkv, orc, lengths, hq, hkv, d, seed):
        dev = torch.device("cuda")
        wl = workloads.scattered_workload(lengths, n_qo_heads=hq, n_kv_heads=hkv, head_dim=d,
                                          seed=seed)
        t = workloads.layer_tensors(wl, 0, device="cpu", poison_unreferenced=True)
        bits = workloads.bf16_bits
        # the step's new rows written into their slots by the oracle's append (the
        # rest of the pool, unlisted, stays NaN so a stray read shows)
        k_bits = orc.append(bits(t.k_pool), wl.append_slots, bits(t.k_new))
        v_bits = orc.append(bits(t.v_pool), wl.append_slots, bits(t.v_new))
        as_bf16 = lambda a: torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(dev)
        self.wl, self.hq, self.hkv, self.d = wl, hq, hkv, d
        self.q, self.kp, self.vp = t.q.to(dev), as_bf16(k_bits), as_bf16(v_bits)
        self.indptr = torch.from_numpy(wl.kv_indptr).to(dev)
        self.indices = torch.from_numpy(wl.kv_indices).to(dev)
        self.ip_host = np.ascontiguousarray(wl.kv_indptr, dtype=np.int32)
        B = wl.batch
        self.out_plan = torch.empty(B, hq, d, dtype=torch.bfloat16, device=dev)
        self.lse_plan = torch.empty(B, hq, dtype=torch.float32, device=dev)
        plan = pkv.paged_decode_plan_create(B, wl.total_tokens, hq, hkv, d)
        pkv.paged_decode_plan(plan, wl.kv_indptr)
        pkv.paged_decode_attn(self.q, self.kp, self.vp, self.indptr, self.indices, B, hq, hkv, d,
                              wl.sm_scale, self.out_plan, self.lse_plan, plan)
        torch.cuda.synchronize()
        assert plan.status() == 0
        self.ref_out, self.ref_lse = orc.decode(bits(t.q), k_bits, v_bits,
                                                wl.kv_indptr, wl.kv_indices, hq, hkv, d,
                                                wl.sm_scale)

    def fresh_outputs(self):
        B = self.wl.batch
        out = torch.full((B, self.hq, self.d), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((B, self.hq), float("nan"), dtype=torch.float32, device="cuda")
        return out, lse

    def call_static(self, lib, out, lse, stream):
        rc = lib.paged_decode_attn_static(
            _p(self.q), _p(self.kp), _p(self.vp), self.ip_host.ctypes.data_as(ctypes.c_void_p),
            _p(self.indptr), _p(self.indices), self.wl.batch, self.hq, self.hkv, self.d,
            ctypes.c_float(self.wl.sm_scale), _p(out), _p(lse), stream)
        return rc

    def check(self, out, lse, what):
        got = out.double().cpu().numpy()
        gl = lse.double().cpu().numpy()
        for name, ref, rl in (("planned entry", self.out_plan.double().cpu().numpy(),
                               self.lse_plan.double().cpu().numpy()),
                              ("oracle", self.ref_out, self.ref_lse)):
            empty = np.isneginf(rl)
            assert np.array_equal(np.isneginf(gl), empty), f"{what}: empty contexts differ ({name})"
            assert np.all(got[empty] == 0), what
            assert np.all(np.isfinite(got)), f"{what}: non-finite output"
            assert np.all(np.abs(got - ref) <= 1e-2 + 1e-2 * np.abs(ref)), \
                f"{what}: out differs from the {name}"
            assert np.all(np.abs(gl[~empty] - rl[~empty]) <= 1e-3), \
                f"{what}: lse differs from the {name}"


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def test_static_scratch_entry_matches_planned_entry(pkv, orc):
    lib = pkv.library()
    for i, args in enumerate(CALLS):
        c = Case(pkv, orc, *args)
        out, lse = c.fresh_outputs()
        assert c.call_static(lib, out, lse, _stream()) == 0, pkv.pkv_last_error()
        torch.cuda.synchronize()
        c.check(out, lse, f"call {i}")
    assert pkv.paged_decode_attn_static_status() == 0


def test_static_calls_queued_back_to_back(pkv, orc):
    """Calls with different shapes and work lists queued on one stream without a host
    wait between them (the per-layer use): each reads the work list uploaded for it
    and the workspace its own decode kernel wrote."""
    lib = pkv.library()
    cases = [Case(pkv, orc, *args) for args in CALLS]
    outs = [c.fresh_outputs() for c in cases]
    outs2 = [c.fresh_outputs() for c in cases]
    s = _stream()
    for c, (o, l) in zip(cases + cases, outs + outs2):
        assert c.call_static(lib, o, l, s) == 0, pkv.pkv_last_error()
    torch.cuda.synchronize()
    for i, (c, (o, l)) in enumerate(zip(cases + cases, outs + outs2)):
        c.check(o, l, f"queued call {i}")
    assert pkv.paged_decode_attn_static_status() == 0


@pytest.mark.filterwarnings("ignore:The CUDA Graph is empty")
def test_static_call_refuses_stream_capture(pkv, orc):
    """A call on a stream being captured returns PKV_ERR_UNSUPPORTED and enqueues
    nothing (its work list lives in one shared host array, which a graph would replay);
    the capture then ends with an empty graph, and the next eager call is correct."""
    lib = pkv.library()
    c = Case(pkv, orc, *CALLS[0])
    out, lse = c.fresh_outputs()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    rc = None
    with torch.cuda.stream(side):
        g.capture_begin()
        try:
            rc = c.call_static(lib, out, lse, ctypes.c_void_p(side.cuda_stream))
            message = pkv.pkv_last_error()
        finally:
            g.capture_end()
    torch.cuda.current_stream().wait_stream(side)
    assert rc == pkv.PKV_ERR_UNSUPPORTED and "captured" in message
    assert c.call_static(lib, out, lse, _stream()) == 0, pkv.pkv_last_error()
    torch.cuda.synchronize()
    c.check(out, lse, "after the refused capture")


def test_static_status_reports_an_expired_wait(pkv, orc):
    """An injected stall (the producers issue no copies) makes the launch's bounded
    waits run out: the status accessor reports it once, and the next call is correct."""
    lib = pkv.library()
    c = Case(pkv, orc, *CALLS[0])
    out, lse = c.fresh_outputs()
    pkv.pkv_inject_stall(1)
    assert c.call_static(lib, out, lse, _stream()) == 0, pkv.pkv_last_error()
    assert pkv.paged_decode_attn_static_status() != 0
    assert pkv.paged_decode_attn_static_status() == 0  # read and cleared
    out, lse = c.fresh_outputs()
    assert c.call_static(lib, out, lse, _stream()) == 0, pkv.pkv_last_error()
    torch.cuda.synchronize()
    c.check(out, lse, "call after the stall")
    assert pkv.paged_decode_attn_static_status() == 0


_ALLOC_CHILD = textwrap.dedent(r"""
    import ctypes, sys
    import numpy as np
    sys.path.insert(0, sys.argv[1])
    import paged_kv_gqa_tokentokvpool_gb300 as pkv
    lib = pkv.library()          # loaded before the CUDA context exists
    import torch
    import workloads
    torch.cuda.init()
    dev = torch.device("cuda")
    def free():
        torch.cuda.synchronize()
        return torch.cuda.mem_get_info()[0]
    wl = workloads.scattered_workload([3000, 17, 700, 9000], seed=5)
    t = workloads.layer_tensors(wl, 0, device=dev)
    ip = torch.from_numpy(wl.kv_indptr).to(dev)
    idx = torch.from_numpy(wl.kv_indices).to(dev)
    out = torch.empty(wl.batch, 32, 128, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(wl.batch, 32, dtype=torch.float32, device=dev)
    ip_host = np.ascontiguousarray(wl.kv_indptr, dtype=np.int32)
    P = lambda x: ctypes.c_void_p(x.data_ptr())
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    # the library's own CUDA runtime starts here (a stream wait); under eager module
    # loading it loads the library's code and static array now
    assert pkv.paged_decode_attn_static_status() == 0
    def call(batch):
        rc = lib.paged_decode_attn_static(P(t.q), P(t.k_pool), P(t.v_pool),
                                          ip_host.ctypes.data_as(ctypes.c_void_p), P(ip), P(idx),
                                          batch, 32, 8, 128, ctypes.c_float(wl.sm_scale), P(out),
                                          P(lse), s)
        assert rc == 0, pkv.pkv_last_error()
    f0 = free()
    call(wl.batch)
    f1 = free()
    call(wl.batch - 1)
    call(wl.batch)
    f2 = free()
    print(f0, f1, f2)
""")


def _alloc_child(env_extra):
    env = dict(os.environ, **env_extra)
    r = subprocess.run([sys.executable, "-c", _ALLOC_CHILD, ROOT], capture_output=True,
                       text=True, env=env, timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    f0, f1, f2 = (int(x) for x in r.stdout.split()[-3:])
    return f0, f1, f2


def test_static_calls_allocate_no_device_memory():
    """In a fresh process: calls after the first leave the device's free memory
    unchanged. With lazy module loading (the CUDA default) the first call may load
    the library's code and its 32 MiB static array; with eager loading that happens
    when the context is created, and the first call leaves free memory unchanged too."""
    f0, f1, f2 = _alloc_child({})
    assert f2 == f1, f"later calls changed free device memory by {f1 - f2} bytes"
    assert 0 <= f0 - f1 <= (32 + 16) << 20, f"first call took {f0 - f1} bytes"
    f0, f1, f2 = _alloc_child({"CUDA_MODULE_LOADING": "EAGER"})
    assert f1 == f0, f"first call changed free device memory by {f0 - f1} bytes"
    assert f2 == f1, f"later calls changed free device memory by {f1 - f2} bytes"


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


def test_static_binding_checks_the_host_offsets(pkv):
    """The Python binding takes batch from the host offsets and refuses a batch the
    offsets do not cover (the C side would read past the end of the array)."""
    dev = torch.device("cuda")
    buf = torch.zeros(4, 8, 128, dtype=torch.bfloat16, device=dev)
    q = torch.zeros(2, 32, 128, dtype=torch.bfloat16, device=dev)
    ip = torch.zeros(3, dtype=torch.int32, device=dev)
    with pytest.raises(ValueError):
        pkv.paged_decode_attn_static(q, buf, buf, np.zeros(2, np.int32), ip, ip, 2, 32, 8, 128,
                                     0.1, q, None)
