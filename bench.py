"""Benchmark: one decode step of paged GQA attention over the token pool.

A step is the whole hot path for one batch: the per-step plan (host partition +
upload), then for every layer the KV append scatter and the split-KV decode
attention (with its LSE merge). Inputs are seeded synthetic tensors shaped like
the Qwen3-4B / Qwen3.5 decode workloads (see workloads.py), resident in HBM when
the timed region starts.

    python bench.py [--config N] [--gpus N --steps K --warmup W] [--impl reference]

Prints one JSON line (rank 0). Under torchrun (N > 1) every rank runs an
independent replica of the step (the path has no exchange step); the time is the
max over ranks and the value sums all ranks' bytes.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "paged GQA decode attn: HBM GB/s & % of peak; µs/step at batch 8/32/128"
DEFAULT_CONFIG = 2
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS_SUSTAINED = 1700.0
L2_BYTES = 129 * 1024 * 1024
NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e, nominal


# ---------------------------------------------------------------------------
# workload state and the step
# ---------------------------------------------------------------------------

class StepState:
    """Device tensors of one decode step for every layer, plus the plan."""

    def __init__(self, wl: workloads.Workload, device="cuda", layers=None,
                 poison_unreferenced=False, fused=None, share=True, early=True):
        import paged_kv_gqa_tokentokvpool_gb300 as pkv
        self.pkv = pkv
        self.wl = wl
        self.device = torch.device(device)
        self.layer_ids = list(range(wl.layers)) if layers is None else list(layers)
        # Every layer's q, new rows, out and lse live in one stacked buffer each
        # (the per-layer tensors are views), so a step's host transfers are a few
        # large copies; the pools are separate allocations per layer.
        B, Hq, Hkv, D = wl.batch, wl.n_qo_heads, wl.n_kv_heads, wl.head_dim
        n = len(self.layer_ids)
        n_app = len(wl.append_slots)
        bf16 = dict(dtype=torch.bfloat16, device=self.device)
        self.q_all = torch.empty(n, B, Hq, D, **bf16)
        self.k_new_all = torch.empty(n, n_app, Hkv, D, **bf16)
        self.v_new_all = torch.empty(n, n_app, Hkv, D, **bf16)
        self.out_all = torch.empty(n, B, Hq, D, **bf16)
        self.lse_all = torch.empty(n, B, Hq, dtype=torch.float32, device=self.device)
        self.k_pool, self.v_pool = [], []
        for i, l in enumerate(self.layer_ids):
            t = workloads.layer_tensors(wl, l, device=self.device,
                                        poison_unreferenced=poison_unreferenced)
            self.q_all[i].copy_(t.q)
            self.k_new_all[i].copy_(t.k_new)
            self.v_new_all[i].copy_(t.v_new)
            self.k_pool.append(t.k_pool)
            self.v_pool.append(t.v_pool)
        self.q = list(self.q_all.unbind(0))
        self.k_new = list(self.k_new_all.unbind(0))
        self.v_new = list(self.v_new_all.unbind(0))
        self.out = list(self.out_all.unbind(0))
        self.lse = list(self.lse_all.unbind(0))
        self.kv_indptr_host = torch.from_numpy(wl.kv_indptr.copy())
        self.kv_indptr = self.kv_indptr_host.to(self.device)
        self.kv_indices = torch.from_numpy(wl.kv_indices.copy()).to(self.device)
        self.slot_ids = torch.from_numpy(wl.append_slots.copy()).to(self.device)
        self.plan = pkv.paged_decode_plan_create(max(B, 1), max(wl.total_tokens, 1), Hq,
                                                 wl.n_kv_heads, D)
        self.launches_per_step = None
        self.graph = None
        self.plan_host_s, self.plan_calls = 0.0, 0  # host time of the per-step plan calls
        # The append runs inside the attention launch when every request has a
        # newest token that is its last listed slot (the decode steps here).
        can_fuse = len(wl.append_slots) == wl.batch and wl.batch > 0
        self.fused = can_fuse if fused is None else (fused and can_fuse)
        # With the append fused, every row a layer reads was written before the
        # step's plan upload (earlier steps, or inputs copied in before the plan),
        # so the attention kernel may start gathering before the kernel ahead of it
        # has finished (PKV_PLAN_EARLY_GATHER). A separate append kernel after the
        # plan would break that promise.
        self.early = bool(early and self.fused)
        if self.early:
            self.plan.set_flags(pkv.PKV_PLAN_EARLY_GATHER)
        # Requests that list the same prefix slots (the prefix-sharing workload) are
        # described to the planner, which then reads each shared slot once for
        # several requests.
        self.sharing = None
        if share and "prefix_lens" in wl.meta:
            gs = wl.meta["group_size"]
            n = len(wl.meta["prefix_lens"])
            self.sharing = (np.arange(0, gs * n + 1, gs, dtype=np.int32),
                            np.asarray(wl.meta["prefix_lens"], dtype=np.int32))

    def layers(self, attn_events=None):
        """Every layer's KV append and decode attention, on the current stream.
        attn_events: list to which (start, end) CUDA events around each attention
        call are appended."""
        pkv, wl = self.pkv, self.wl
        stream = torch.cuda.current_stream()
        for i in range(len(self.layer_ids)):
            if not self.fused:
                pkv.kvpool_append(self.k_pool[i], self.v_pool[i], self.slot_ids, self.k_new[i],
                                  self.v_new[i], stream=stream)
            if attn_events is not None:
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
            if self.fused:
                pkv.paged_decode_append_attn(self.q[i], self.k_pool[i], self.v_pool[i],
                                             self.kv_indptr, self.kv_indices, self.slot_ids,
                                             self.k_new[i], self.v_new[i], wl.batch,
                                             wl.n_qo_heads, wl.n_kv_heads, wl.head_dim,
                                             wl.sm_scale, self.out[i], self.lse[i], self.plan,
                                             stream=stream)
            else:
                pkv.paged_decode_attn(self.q[i], self.k_pool[i], self.v_pool[i], self.kv_indptr,
                                      self.kv_indices, wl.batch, wl.n_qo_heads, wl.n_kv_heads,
                                      wl.head_dim, wl.sm_scale, self.out[i], self.lse[i],
                                      self.plan, stream=stream)
            if attn_events is not None:
                e1.record(stream)
                attn_events.append((e0, e1))

    def run(self, attn_events=None):
        """One decode step: the per-step plan (host partition + upload), then every
        layer's append and attention -- replayed from the captured CUDA graph when
        there is one (and no per-call events are asked for)."""
        pkv = self.pkv
        stream = torch.cuda.current_stream()
        t0 = time.perf_counter()
        if self.sharing is not None:
            pkv.paged_decode_plan_shared(self.plan, self.kv_indptr_host.numpy(), self.sharing[0],
                                         self.sharing[1], stream=stream)
        else:
            pkv.paged_decode_plan(self.plan, self.kv_indptr_host.numpy(), stream=stream)
        self.plan_host_s += time.perf_counter() - t0
        self.plan_calls += 1
        if self.graph is not None and attn_events is None:
            self.graph.replay()
        else:
            self.layers(attn_events)
        if self.launches_per_step is None:
            # append (unless fused), then the decode kernel and the merge kernel (launched
            # even when nothing is split), or the one single-launch kernel of a small plan
            attn = 1 if self.plan.single_launch() else 2
            per_layer = (0 if self.fused or not len(self.wl.append_slots) else 1) + attn
            self.launches_per_step = per_layer * len(self.layer_ids)

    def capture(self):
        """Capture the layer loop (every layer's append + attention launch) into
        one CUDA graph; the plan stays outside it, so each step re-plans on the
        host and uploads into the plan's fixed device buffers before the replay."""
        self.run()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.layers()
        torch.cuda.synchronize()
        self.graph = g


class HostIO:
    """Pinned host copies of one step's inputs and outputs, for the end-to-end
    measurement: every step copies q, the new K/V rows and the slot/index arrays
    host->device, runs the step, and copies out and lse device->host. Each stacked
    array (all layers) is one copy."""

    def __init__(self, st: StepState):
        self.st = st
        self.ins = [(dev, dev.cpu().pin_memory()) for dev in
                    (st.q_all, st.k_new_all, st.v_new_all, st.kv_indices, st.kv_indptr,
                     st.slot_ids)]
        self.outs = [(dev, torch.empty(dev.shape, dtype=dev.dtype, pin_memory=True))
                     for dev in (st.out_all, st.lse_all)]
        self.out = list(self.outs[0][1].unbind(0))
        self.h2d_bytes = sum(h.numel() * h.element_size() for _, h in self.ins)
        self.d2h_bytes = sum(h.numel() * h.element_size() for _, h in self.outs)

    def run(self):
        for dev, host in self.ins:
            dev.copy_(host, non_blocking=True)
        self.st.run()
        for dev, host in self.outs:
            host.copy_(dev, non_blocking=True)


def step_bytes(wl: workloads.Workload) -> dict:
    """Algorithmic HBM bytes of one step: each distinct KV row read once per layer,
    the slot indices, q, out and lse, and the append's read + write of new rows."""
    B, Hq, Hkv, D = wl.batch, wl.n_qo_heads, wl.n_kv_heads, wl.head_dim
    row = Hkv * D * 2  # bytes of one slot's K (or V) for all heads
    n_unique = int(np.unique(wl.kv_indices).size)
    N = wl.total_tokens
    attn = n_unique * 2 * row + N * 4 + (B + 1) * 4 + B * Hq * D * 2 * 2 + B * Hq * 4
    attn_logical = N * 2 * row + N * 4 + (B + 1) * 4 + B * Hq * D * 2 * 2 + B * Hq * 4
    n_app = len(wl.append_slots)
    append = n_app * 2 * row * 2 + n_app * 4
    return {"attn_per_layer": attn, "attn_logical_per_layer": attn_logical,
            "append_per_layer": append,
            "step": wl.layers * (attn + append),
            "step_logical": wl.layers * (attn_logical + append)}


# ---------------------------------------------------------------------------
# measurement helpers
# ---------------------------------------------------------------------------

def measured_hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "of measured"
    except Exception:
        return FALLBACK_HBM_GBS, "of fallback"


class ClockSampler:
    """Samples the GPU's SM clock and clock-event (throttle) reasons while the
    timed region runs: NVML through ctypes, polled from a thread every ~2 ms
    (falls back to nvidia-smi at 200 ms if NVML cannot be loaded). Read only."""

    REASONS = {0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown", 0x4: "sw_power_cap"}

    def __init__(self, device_index: int):
        self.device_index = device_index
        self.samples = []
        self.max_mhz = None
        self._stop = None

    def _nvml(self):
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        props = torch.cuda.get_device_properties(self.device_index)
        handle = ctypes.c_void_p()
        uuid = getattr(props, "uuid", None)
        ok = False
        if uuid is not None:
            text = str(uuid)
            if not text.startswith("GPU-"):
                text = "GPU-" + text
            ok = lib.nvmlDeviceGetHandleByUUID(text.encode(), ctypes.byref(handle)) == 0
        if not ok:
            raise RuntimeError("no NVML handle for the device")
        return lib, handle

    def __enter__(self):
        import threading
        self._stop = threading.Event()
        try:
            import ctypes
            lib, handle = self._nvml()
            clk = ctypes.c_uint()
            if lib.nvmlDeviceGetMaxClockInfo(handle, 1, ctypes.byref(clk)) == 0:
                self.max_mhz = clk.value
            get_reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")

            def poll():
                while not self._stop.is_set():
                    c = ctypes.c_uint()
                    if lib.nvmlDeviceGetClockInfo(handle, 1, ctypes.byref(c)) == 0:
                        r = ctypes.c_ulonglong(0)
                        get_reasons(handle, ctypes.byref(r))
                        self.samples.append((c.value, r.value))
                    self._stop.wait(0.002)

            self._thread = threading.Thread(target=poll, daemon=True)
            self._thread.start()
            self._mode = "nvml"
        except Exception:
            self._mode = "smi"
            self._proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.device_index}",
                 "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.active",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        return self

    def __exit__(self, *exc):
        self._stop.set()
        if self._mode == "nvml":
            self._thread.join(timeout=2)
        else:
            self._proc.terminate()
            try:
                out, _ = self._proc.communicate(timeout=5)
            except Exception:
                self._proc.kill()
                out, _ = self._proc.communicate()
            for line in out.splitlines():
                parts = [x.strip() for x in line.split(",")]
                try:
                    self.samples.append((float(parts[0]), int(parts[2], 16)))
                    self.max_mhz = float(parts[1])
                except (ValueError, IndexError):
                    pass

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["unsampled"],
                    "samples": 0, "source": self._mode}
        mhz = [m for m, _ in self.samples]
        bits = 0
        for _, r in self.samples:
            bits |= r
        reasons = sorted(name for bit, name in self.REASONS.items() if bits & bit)
        return {"sm_mhz": statistics.median(mhz), "sm_min_mhz": min(mhz),
                "sm_max_mhz": self.max_mhz, "reasons": reasons, "samples": len(mhz),
                "source": self._mode}


def cpu_baseline(st: StepState, budget_s: float = 12.0, max_layers=None):
    """Time the fp64 oracle on the host cores over a bounded sample of the same
    step: whole layers (all requests), in order, until ~budget_s of oracle time is
    spent. A step that takes less than the budget is walked again (each layer's rows
    are fetched from the device afresh for every call, outside the timed region)."""
    import oracle
    orc = oracle.default()
    wl = st.wl
    threads = orc.max_threads()
    total_t, total_bytes, calls = 0.0, 0, 0
    per_layer = step_bytes(wl)["attn_per_layer"]
    uniq, inv = np.unique(wl.kv_indices, return_inverse=True)
    idx_dev = torch.from_numpy(uniq.astype(np.int64)).to(st.device)
    compact = inv.astype(np.int32)
    limit = len(st.layer_ids) if max_layers is None else min(max_layers, len(st.layer_ids))
    while total_t < budget_s:
        for i in range(limit):
            k = workloads.bf16_bits(st.k_pool[i].index_select(0, idx_dev))
            v = workloads.bf16_bits(st.v_pool[i].index_select(0, idx_dev))
            q = workloads.bf16_bits(st.q[i])
            t0 = time.perf_counter()
            orc.decode(q, k, v, wl.kv_indptr, compact, wl.n_qo_heads, wl.n_kv_heads,
                       wl.head_dim, wl.sm_scale)
            total_t += time.perf_counter() - t0
            total_bytes += per_layer
            calls += 1
            if total_t >= budget_s:
                break
    passes = f"{calls / limit:.1f} passes over " if calls > limit else ""
    return {"value": total_bytes / total_t / 1e9, "unit": "GB/s", "cores": threads,
            "kind": "oracle",
            "sample": f"{calls} layer calls ({passes}{min(calls, limit)} of {wl.layers} layers) of "
                      f"{wl.name} (all {wl.batch} requests, attention only), fp64 C++ oracle, "
                      f"{total_t:.1f} s"}


# ---------------------------------------------------------------------------
# main
# ---------------------------------------------------------------------------

def max_over_ranks(x: float, dist=None, device="cpu") -> float:
    """The largest of every rank's x (x itself without a process group)."""
    if dist is None:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_gbs(world: int, bytes_per_step: int, steps: int, elapsed_ms: float) -> float:
    """Whole-job throughput of `world` replicas that each ran `steps` steps in (at
    most) elapsed_ms: every rank's bytes over the slowest rank's time."""
    return world * bytes_per_step * steps / (elapsed_ms * 1e-3) / 1e9


def measure_tier(config_no: int, steps: int, warmup: int, host_frac: float = 0.1) -> dict:
    """The host KV tier on a workload's pool (NVLink-C2C on GB300): scattered row moves
    HBM <-> pinned host memory (kvpool_offload / kvpool_prefetch) against one contiguous
    copy of the same bytes by the copy engines, and one layer's attention with a
    fraction of its listed rows read in place from host memory
    (paged_decode_attn_tiered) against the same call with every row in HBM."""
    import paged_kv_gqa_tokentokvpool_gb300 as pkv
    wl = workloads.config_workload(config_no)
    dev = torch.device("cuda")
    stream = torch.cuda.current_stream()
    rows = min(wl.total_tokens, 1 << 18)
    t = workloads.layer_tensors(wl, 0, device=dev)
    Hkv, D = wl.n_kv_heads, wl.head_dim
    kh = torch.empty(rows, Hkv, D, dtype=torch.bfloat16).pin_memory()
    vh = torch.empty_like(kh).pin_memory()
    rng = np.random.default_rng(7)
    dev_slots = torch.from_numpy(wl.kv_indices[:rows].copy()).to(dev)
    host_slots = torch.from_numpy(rng.permutation(rows).astype(np.int32)).to(dev)
    row_bytes = 2 * Hkv * D * 2

    def event_ms(fn):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps

    res = {"rows": rows, "row_bytes": row_bytes, "workload": f"{wl.name}: {wl.description}"}
    for name, fn in (("offload", pkv.kvpool_offload), ("prefetch", pkv.kvpool_prefetch)):
        ms = event_ms(lambda: fn(t.k_pool, t.v_pool, dev_slots, kh, vh, host_slots))
        res[name] = {"us_per_call": ms * 1e3, "gbs_over_link": rows * row_bytes / (ms * 1e-3) / 1e9}
    # the link's rate for the same bytes as one contiguous copy each way (copy engines)
    host_flat = torch.empty(rows * row_bytes, dtype=torch.uint8).pin_memory()
    dev_flat = torch.empty(rows * row_bytes, dtype=torch.uint8, device=dev)
    for name, (dst, src) in (("contiguous_h2d", (dev_flat, host_flat)),
                             ("contiguous_d2h", (host_flat, dev_flat))):
        ms = event_ms(lambda: dst.copy_(src, non_blocking=True))
        res[name] = {"gbs": rows * row_bytes / (ms * 1e-3) / 1e9}
    del host_flat, dev_flat, kh, vh
    # attention over the layer with host_frac of its listed rows in host memory
    n = wl.total_tokens
    moved = np.sort(rng.choice(n, size=max(1, int(host_frac * n)), replace=False))
    moved_slots = torch.from_numpy(wl.kv_indices[moved].astype(np.int64)).to(dev)
    kh2 = t.k_pool.index_select(0, moved_slots).cpu().pin_memory()
    vh2 = t.v_pool.index_select(0, moved_slots).cpu().pin_memory()
    tiered_idx = wl.kv_indices.copy()
    tiered_idx[moved] = -1 - np.arange(len(moved), dtype=np.int32)
    ip = torch.from_numpy(wl.kv_indptr).to(dev)
    idx_dev = torch.from_numpy(wl.kv_indices).to(dev)
    idx_tier = torch.from_numpy(tiered_idx).to(dev)
    out = torch.empty(wl.batch, wl.n_qo_heads, D, dtype=torch.bfloat16, device=dev)
    plan = pkv.paged_decode_plan_create(wl.batch, n, wl.n_qo_heads, Hkv, D)
    pkv.paged_decode_plan(plan, wl.kv_indptr)
    args = (wl.batch, wl.n_qo_heads, Hkv, D, wl.sm_scale, out, None, plan)
    ms_dev = event_ms(lambda: pkv.paged_decode_attn(t.q, t.k_pool, t.v_pool, ip, idx_dev, *args))
    ms_tier = event_ms(lambda: pkv.paged_decode_attn_tiered(t.q, t.k_pool, t.v_pool, kh2, vh2, ip,
                                                            idx_tier, *args))
    if plan.status() != 0:
        raise RuntimeError("a decode pipeline wait exceeded its bound: the tier figures are invalid")
    host_bytes = len(moved) * row_bytes
    res["attention_in_place"] = {
        "host_fraction": len(moved) / n, "host_bytes": host_bytes,
        "us_all_rows_in_hbm": ms_dev * 1e3, "us_with_host_rows": ms_tier * 1e3,
        "host_gbs": host_bytes / (ms_tier * 1e-3) / 1e9,
        "note": "one layer's attention (all requests); host rows read over the link in place"}
    del plan, t
    torch.cuda.empty_cache()
    return res


def run_tier_bench(args):
    res = measure_tier(args.config, args.steps, args.warmup)
    print(json.dumps({"metric": "host KV tier: scattered row moves HBM <-> pinned host memory, "
                                "and attention reading host rows in place",
                      "unit": "GB/s", **res}), flush=True)
    return 0


def measured_tensor_peak():
    """Sustained dense bf16 rate (a kernel timed inside a long step)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["bf16_tflops_sustained"]), "of measured (sustained)"
    except Exception:
        return FALLBACK_BF16_TFLOPS_SUSTAINED, "of fallback (sustained)"


class PrefillState:
    """Device tensors of one chunked-prefill step for every layer, plus the plan.
    A layer is kvpool_append of the chunks' rows, then paged_prefill_attn."""

    def __init__(self, pw: workloads.PrefillWorkload, device="cuda", layers=None):
        import paged_kv_gqa_tokentokvpool_gb300 as pkv
        self.pkv, self.pw = pkv, pw
        dev = torch.device(device)
        self.layer_ids = list(range(pw.layers)) if layers is None else list(layers)
        self.t = [workloads.prefill_tensors(pw, l, device=dev) for l in self.layer_ids]
        self.out = [torch.empty(pw.total_q, pw.n_qo_heads, pw.head_dim, dtype=torch.bfloat16,
                                device=dev) for _ in self.layer_ids]
        self.lse = [torch.empty(pw.total_q, pw.n_qo_heads, dtype=torch.float32, device=dev)
                    for _ in self.layer_ids]
        self.qo = torch.from_numpy(pw.qo_indptr).to(dev)
        self.kv = torch.from_numpy(pw.kv_indptr).to(dev)
        self.idx = torch.from_numpy(pw.kv_indices).to(dev)
        self.slots = torch.from_numpy(pw.chunk_slots).to(dev)
        self.plan = pkv.paged_prefill_plan_create(pw.batch, pw.total_q, pw.n_qo_heads,
                                                  pw.n_kv_heads, pw.head_dim)
        self.graph = None

    def layers(self, events=None):
        pkv, pw = self.pkv, self.pw
        stream = torch.cuda.current_stream()
        for i in range(len(self.layer_ids)):
            q, kp, vp, kn, vn = self.t[i]
            pkv.kvpool_append(kp, vp, self.slots, kn, vn, stream=stream)
            if events is not None:
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
            pkv.paged_prefill_attn(q, kp, vp, self.qo, self.kv, self.idx, pw.batch,
                                   pw.n_qo_heads, pw.n_kv_heads, pw.head_dim, pw.sm_scale,
                                   self.out[i], self.lse[i], self.plan, stream=stream)
            if events is not None:
                e1.record(stream)
                events.append((e0, e1))

    def run(self, events=None):
        self.pkv.paged_prefill_plan(self.plan, self.pw.qo_indptr, self.pw.kv_indptr,
                                    stream=torch.cuda.current_stream())
        if self.graph is not None and events is None:
            self.graph.replay()
        else:
            self.layers(events)

    def capture(self):
        self.run()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.layers()
        torch.cuda.synchronize()
        self.graph = g


def measure_prefill(pf_no: int, steps: int, warmup: int, layers=None, cpu_budget=None):
    """Chunked prefill (the pages' 512- and 64-token chunks): useful causal
    attention FLOP/s of the step, and of the attention kernel alone against the
    tensor roofline. Returns the JSON line as a dict (cpu_baseline only when
    cpu_budget is given)."""
    pw = workloads.prefill_config(pf_no)
    if layers is not None:
        pw.layers = max(1, min(layers, pw.layers))
    st = PrefillState(pw)
    st.capture()
    stream = torch.cuda.current_stream()
    # causal attention: per query head and attended pair, 2 D flops for q.k and 2 D for p.v
    flops_layer = 4.0 * pw.head_dim * pw.n_qo_heads * pw.attended_pairs()
    for _ in range(warmup):
        st.run()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(torch.cuda.current_device()) as clocks:
        e0.record(stream)
        for _ in range(steps):
            st.run()
        e1.record(stream)
        torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    events = []
    for _ in range(steps):
        st.run(events)
    torch.cuda.synchronize()
    attn_ms = float(np.mean([a.elapsed_time(b) for a, b in events]))
    if st.plan.status() != 0:
        raise RuntimeError("a prefill pipeline wait exceeded its bound: the timed results are invalid")
    peak, peak_kind = measured_tensor_peak()
    step_tflops = flops_layer * pw.layers / (ms * 1e-3) / 1e12
    attn_tflops = flops_layer / (attn_ms * 1e-3) / 1e12
    line = {
        "metric": "chunked-prefill attention over the token pool: useful causal TFLOP/s",
        "value": step_tflops, "unit": "TFLOP/s", "n_gpus": 1, "steps": steps,
        "warmup": warmup, "ms_per_step": ms, "higher_is_better": True, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": f"{pw.name}: {pw.description}", "layers": pw.layers,
                   "batch": pw.batch, "query_tokens": pw.total_q,
                   "context_tokens": pw.total_tokens, "attended_pairs": pw.attended_pairs(),
                   "flops_per_layer": flops_layer,
                   "launch": "cuda graph of the layer loop (append + attention per layer)"},
        "roofline": {"bound": "tensor", "achieved": attn_tflops, "peak": peak,
                     "unit": "TFLOP/s", "frac": attn_tflops / peak, "traffic": None,
                     "kernel": f"paged_prefill_attn, avg of {len(events)} event-timed eager "
                               f"calls {attn_ms * 1e3:.1f} us, tcgen05.mma with TMEM accumulators",
                     "peak_kind": peak_kind},
        "clocks": clocks.summary(),
    }
    if cpu_budget is not None:
        line["cpu_baseline"] = prefill_cpu_baseline(pw, cpu_budget)
    del st
    torch.cuda.empty_cache()
    return line


def run_curve(args):
    """Decode attention over a grid of batch sizes and context lengths (the Qwen3-4B
    attention shape, scattered slots, 2-8 layers per step, fused append, graph replay):
    where the path reaches the HBM roofline. One JSON line with every point."""
    import paged_kv_gqa_tokentokvpool_gb300 as pkv
    torch.cuda.set_device(0)
    peak, peak_kind = measured_hbm_peak()
    points = []
    for ctx in (512, 4096, 32768):
        for batch in (1, 4, 8, 16, 32, 64, 128):
            # pools a little larger than the listed slots, and as many layers (2-8) as
            # fit in about 48 GB, so the per-step plan and graph launch weigh little
            pool_slots = batch * ctx + batch * ctx // 20 + 1024
            layer_bytes = pool_slots * 8 * 128 * 2 * 2
            layers = int(max(2, min(8, 48e9 // layer_bytes)))
            wl = workloads.scattered_workload([ctx] * batch, layers=layers, pool_slots=pool_slots,
                                              seed=3000 + batch, name="curve", description="")
            st = StepState(wl)
            st.capture()
            nbytes = step_bytes(wl)
            stream = torch.cuda.current_stream()
            for _ in range(args.warmup):
                st.run()
            torch.cuda.synchronize()
            # steps that fit in L2 twice are timed one by one after an L2 flush; larger
            # ones back to back between two events
            flush = (torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=stream.device)
                     if nbytes["step"] < 2 * L2_BYTES else None)

            def time_steps():
                if flush is None:
                    t0 = torch.cuda.Event(enable_timing=True)
                    t1 = torch.cuda.Event(enable_timing=True)
                    t0.record(stream)
                    for _ in range(args.steps):
                        st.run()
                    t1.record(stream)
                    t1.synchronize()
                    return t0.elapsed_time(t1)
                total = 0.0
                for _ in range(args.steps):
                    flush.fill_(1)
                    t0 = torch.cuda.Event(enable_timing=True)
                    t1 = torch.cuda.Event(enable_timing=True)
                    t0.record(stream)
                    st.run()
                    t1.record(stream)
                    t1.synchronize()
                    total += t0.elapsed_time(t1)
                return total

            with ClockSampler(0) as clocks:
                total_ms = time_steps()
            if st.plan.status() != 0:
                raise RuntimeError("a decode pipeline wait exceeded its bound")
            us_layer = total_ms / args.steps / wl.layers * 1e3
            gbs = nbytes["step"] / wl.layers / (us_layer * 1e-6) / 1e9
            point = {"batch": batch, "context": ctx, "layers": layers, "us_per_layer": us_layer, "gbs": gbs,
                     "frac_of_measured": gbs / peak, "single_launch": st.plan.single_launch(),
                     "l2_flushed": flush is not None, "clocks": clocks.summary()}
            # the other mode where the plan can run it (PKV_PLAN_SINGLE_LAUNCH /
            # PKV_PLAN_PERSISTENT), timed the same way
            other = pkv.PKV_PLAN_PERSISTENT if point["single_launch"] else pkv.PKV_PLAN_SINGLE_LAUNCH
            try:
                st.plan.set_flags((pkv.PKV_PLAN_EARLY_GATHER if st.early else 0) | other)
            except pkv.PkvError:
                other = None
            if other is not None:
                st.graph = None  # the next step plans in the other mode: capture it anew
                st.capture()
                for _ in range(args.warmup):
                    st.run()
                total_ms = time_steps()
                if st.plan.status() != 0:
                    raise RuntimeError("a decode pipeline wait exceeded its bound")
                point["us_per_layer_other_mode"] = total_ms / args.steps / wl.layers * 1e3
            points.append(point)
            del st, flush
            torch.cuda.empty_cache()
    line = {"metric": "paged GQA decode attention, batch x context curve (us per layer, GB/s)",
            "unit": "GB/s", "data": "synthetic", "dtype": "bf16", "steps": args.steps,
            "warmup": args.warmup, "peak_gbs": peak, "peak_kind": peak_kind,
            "config": {"workload": "Qwen3-4B attention shape (32Q/8KV, head_dim 128), scattered "
                                   "slots, 2-8 layers per step (as fit in about 48 GB), fused "
                                   "append, CUDA graph of the layers, plan per step"},
            "points": points}
    print(json.dumps(line), flush=True)
    return 0


def run_prefill_bench(args):
    line = measure_prefill(args.prefill, args.steps, args.warmup, args.layers,
                           None if args.no_cpu_baseline else args.cpu_budget)
    print(json.dumps(line), flush=True)
    return 0


def prefill_cpu_baseline(pw: workloads.PrefillWorkload, budget_s: float):
    """The fp64 oracle on the host cores over a bounded sample of the same step:
    whole requests of layer 0, one at a time, until about budget_s seconds."""
    import oracle
    orc = oracle.default()
    q, kp, vp, kn, vn = workloads.prefill_tensors(pw, 0, device="cpu")
    kb = orc.append(workloads.bf16_bits(kp), pw.chunk_slots, workloads.bf16_bits(kn))
    vb = orc.append(workloads.bf16_bits(vp), pw.chunk_slots, workloads.bf16_bits(vn))
    qb = workloads.bf16_bits(q)
    flops = 0.0
    done = 0
    t0 = time.perf_counter()
    for b in np.argsort(pw.contexts):  # shortest first, so the sample is not empty
        C, L = int(pw.chunks[b]), int(pw.contexts[b])
        q0, k0 = int(pw.qo_indptr[b]), int(pw.kv_indptr[b])
        orc.prefill(qb[q0:q0 + C], kb, vb, np.array([0, C], np.int32),
                    np.array([0, L], np.int32), pw.kv_indices[k0:k0 + L], pw.n_qo_heads,
                    pw.n_kv_heads, pw.head_dim, pw.sm_scale)
        flops += 4.0 * pw.head_dim * pw.n_qo_heads * (C * (L - C) + C * (C + 1) // 2)
        done += 1
        if time.perf_counter() - t0 > budget_s:
            break
    el = time.perf_counter() - t0
    return {"value": flops / el / 1e12, "unit": "TFLOP/s", "cores": orc.max_threads(),
            "kind": "oracle",
            "sample": f"{done} of {pw.batch} requests of layer 0 (shortest first), fp64 C++ "
                      f"oracle, {el:.1f} s"}


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def run_reference(args, world, rank):
    """The oracle as the reference arm: each step is the oracle over one layer of
    the workload (all requests), on the host cores."""
    if rank != 0:
        return 0
    wl = workloads.config_workload(args.config)
    import oracle
    orc = oracle.default()
    bytes_layer = step_bytes(wl)["attn_per_layer"]
    t = workloads.layer_tensors(wl, 0, device="cpu")
    uniq, inv = np.unique(wl.kv_indices, return_inverse=True)
    k = workloads.bf16_bits(t.k_pool[torch.from_numpy(uniq.astype(np.int64))])
    v = workloads.bf16_bits(t.v_pool[torch.from_numpy(uniq.astype(np.int64))])
    q = workloads.bf16_bits(t.q)
    compact = inv.astype(np.int32)

    def one():
        orc.decode(q, k, v, wl.kv_indptr, compact, wl.n_qo_heads, wl.n_kv_heads,
                   wl.head_dim, wl.sm_scale)

    for _ in range(args.warmup):
        one()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one()
    el = time.perf_counter() - t0
    value = bytes_layer * args.steps / el / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": el / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{wl.name}: {wl.description}",
                       "sample": "one layer (all requests) per step"},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": orc.max_threads(),
                             "kind": "oracle",
                             "sample": f"layer 0 of {wl.layers} of {wl.name}, all "
                                       f"{wl.batch} requests, per step"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def measure_decode(config_no: int, args, world=1, pg=None, local=0, cpu_budget=None,
                   layers=None):
    """Time one decode workload: K graph-replayed steps (device time, max over
    ranks), an eager pass that times each attention call alone, and the end-to-end
    step through the public API with host buffers. Returns the JSON line as a dict
    (cpu_baseline only when cpu_budget is given)."""
    wl = workloads.config_workload(config_no)
    if layers is not None:
        wl.layers = max(1, min(layers, wl.layers))
        wl.description += f" [first {wl.layers} layers only]"
    st = StepState(wl, fused=not args.separate_append, share=not args.no_share,
                   early=not args.no_early)
    if not args.no_graph:
        st.capture()
    nbytes = step_bytes(wl)
    stream = torch.cuda.current_stream()

    def barrier():
        if pg is not None:
            pg.barrier()
        torch.cuda.synchronize()

    for _ in range(args.warmup):
        st.run()
    barrier()
    attn_events = []
    # A step that reads less than twice the L2 would be timed warm: then each step is
    # timed on its own, with a write of a buffer larger than L2 between steps.
    flush = (torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=stream.device)
             if nbytes["step"] < 2 * L2_BYTES else None)

    def timed(fn):
        if flush is None:
            t0 = torch.cuda.Event(enable_timing=True)
            t1 = torch.cuda.Event(enable_timing=True)
            t0.record(stream)
            for _ in range(args.steps):
                fn()
            t1.record(stream)
            torch.cuda.synchronize()
            return t0.elapsed_time(t1)
        pairs = []
        for _ in range(args.steps):
            flush.fill_(1)
            t0 = torch.cuda.Event(enable_timing=True)
            t1 = torch.cuda.Event(enable_timing=True)
            t0.record(stream)
            fn()
            t1.record(stream)
            pairs.append((t0, t1))
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in pairs)

    st.plan_host_s, st.plan_calls = 0.0, 0
    st.plan.reset_timing()
    with ClockSampler(local) as clocks:
        step_ms = timed(st.run)
    barrier()
    plan_timing = st.plan.timing()
    plan_wall_us = st.plan_host_s / max(st.plan_calls, 1) * 1e6
    elapsed_ms = max_over_ranks(step_ms, pg, "cuda")
    # The timed loop queues every step at once, so the host runs ahead of the GPU and
    # each plan call waits for a free staging buffer. Here the host instead waits for
    # the step two back before planning (it stays two steps ahead): the plan call's
    # own wait should then be about zero.
    done = []
    st.plan.reset_timing()
    for _ in range(args.steps):
        if len(done) >= 2:
            done[-2].synchronize()
        st.run()
        ev = torch.cuda.Event()
        ev.record(stream)
        done.append(ev)
    torch.cuda.synchronize()
    plan_two_ahead = st.plan.timing()
    # The attention calls alone, each bracketed by CUDA events on its stream
    # (eager launches: an event between two kernels also ends their overlap).
    for _ in range(args.steps):
        if flush is not None:
            flush.fill_(1)
        st.run(attn_events)
    torch.cuda.synchronize()
    attn_ms = [a.elapsed_time(b) for a, b in attn_events]
    if st.plan.status() != 0:
        raise RuntimeError("a decode pipeline wait exceeded its bound: the timed results are invalid")

    # end to end through the public API, host buffers in and out
    io = HostIO(st)
    for _ in range(args.warmup):
        io.run()
    barrier()
    e2e_ms = max_over_ranks(timed(io.run), pg, "cuda")

    ms_per_step = elapsed_ms / args.steps
    value = replica_gbs(world, nbytes["step"], args.steps, elapsed_ms)
    e2e_value = replica_gbs(world, nbytes["step"], args.steps, e2e_ms)
    peak, peak_kind = measured_hbm_peak()
    attn_avg_ms = statistics.mean(attn_ms)
    # The timed region is the step's attention calls back to back (the append is fused
    # into them when it can be), so one call's average duration there is the step time
    # over the layers; the eager pass above also times each call alone.
    n_layers = len(st.layer_ids)
    layer_ms = elapsed_ms / args.steps / n_layers
    achieved = nbytes["step"] / n_layers / (layer_ms * 1e-3) / 1e9
    eager_gbs = nbytes["attn_per_layer"] / (attn_avg_ms * 1e-3) / 1e9
    info = st.plan.info()
    attn_kernels = ("paged_decode_attn (single-launch cluster kernel, merge in distributed "
                    "shared memory): " if st.plan.single_launch() else
                    "paged_decode_attn (split-KV decode kernel + LSE merge kernel): ")
    traffic = _profiled_traffic(config_no) if layers is None else None
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {
            "workload": f"{wl.name}: {wl.description}", "layers": wl.layers,
            "batch": wl.batch, "n_qo_heads": wl.n_qo_heads, "n_kv_heads": wl.n_kv_heads,
            "head_dim": wl.head_dim, "pool_slots": wl.pool_slots,
            "total_context_tokens": wl.total_tokens, "us_per_step": ms_per_step * 1e3,
            "bytes_per_step": nbytes["step"],
            "hbm_frac_of_peak": value / world / peak, "peak_gbs": peak, "peak_kind": peak_kind,
            "effective_logical_gbs": world * nbytes["step_logical"] * args.steps
            / (elapsed_ms * 1e-3) / 1e9,
            "plan": {"units": info["n_units"], "merges": info["n_merges"],
                     "chunk_tokens": info["chunk_tokens"], "ctas": info["n_ctas"],
                     "host_us_per_step": plan_wall_us,
                     "compute_us_per_step": plan_timing["compute_us"],
                     "wait_us_per_step": plan_timing["wait_us"],
                     "wait_us_two_ahead": plan_two_ahead["wait_us"],
                     "compute_us_two_ahead": plan_two_ahead["compute_us"],
                     "host_note": "host time of the per-step plan call (wall), of its "
                                  "partition alone (compute) and of its wait for a free "
                                  "staging buffer (wait), averaged over the timed steps, "
                                  "where the host queues every step at once and runs "
                                  "ahead of the GPU; *_two_ahead: the same with the host "
                                  "kept two steps ahead of the GPU"},
            "l2": (f"inputs larger than L2: each step reads {nbytes['step'] / 1e9:.2f} GB "
                   f"across {wl.layers} layers' pools (L2 {L2_BYTES / 2**20:.0f} MiB)"
                   if flush is None else
                   f"L2 flushed between timed steps (a {2 * L2_BYTES / 2**20:.0f} MiB write); "
                   f"each step reads {nbytes['step'] / 1e6:.1f} MB"),
            "hbm_frac_of_nominal": value / world / NOMINAL_HBM_GBS,
            "parallelism": f"replicas x{world}",
            "launch": "eager" if args.no_graph else "cuda graph of the layer loop per step; plan on host",
            "append": "fused into the attention launch" if st.fused else "separate kernel",
            "shared_prefixes": "described to the planner" if st.sharing is not None else "none",
            "early_gather": st.early,
        },
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": attn_kernels +
                               f"{layer_ms * 1e3:.1f} us per call in the timed graph replay "
                               f"(step time over {n_layers} layers), "
                               f"{nbytes['step'] / n_layers / 1e6:.1f} MB algorithmic per call",
                     "eager_call": {"us": attn_avg_ms * 1e3, "gbs": eager_gbs,
                                    "note": f"avg of {len(attn_ms)} calls each timed alone with "
                                            "events (eager launches, no overlap between calls"
                                            + (", L2 flushed before each step)" if flush is not None
                                               else ")")},
                     "peak_kind": peak_kind},
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": io.h2d_bytes,
                "d2h_bytes_per_step": io.d2h_bytes, "ms_per_step": e2e_ms / args.steps},
        "gpu_launches": st.launches_per_step * args.steps,
        "clocks": clocks.summary(),
    }
    if cpu_budget is not None and world == 1:
        line["cpu_baseline"] = cpu_baseline(st, budget_s=cpu_budget)
    del io, st
    torch.cuda.empty_cache()
    return line


def sweep_entry(line: dict) -> dict:
    """The figures of one workload's bench line that the sweep records."""
    c, r = line["config"], line["roofline"]
    e = {"workload": c["workload"], "layers": c["layers"], "batch": c["batch"],
         "steps": line["steps"], "clocks": line["clocks"]}
    if line["unit"] == "GB/s":
        e.update({"us_per_step": c["us_per_step"], "gbs": line["value"],
                  "frac_of_measured": c["hbm_frac_of_peak"],
                  "frac_of_nominal": c["hbm_frac_of_nominal"], "peak_kind": c["peak_kind"],
                  "bytes_per_step": c["bytes_per_step"],
                  "attn_call_eager_us": r["eager_call"]["us"], "e2e_gbs": line["e2e"]["value"],
                  "e2e_us_per_step": line["e2e"]["ms_per_step"] * 1e3, "plan": c["plan"],
                  "l2": c["l2"], "shared_prefixes": c["shared_prefixes"]})
    else:
        e.update({"ms_per_step": line["ms_per_step"], "tflops": line["value"],
                  "attn_call_tflops": r["achieved"], "frac_of_measured_sustained": r["frac"],
                  "peak_kind": r["peak_kind"]})
    return e


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--config", type=int, default=DEFAULT_CONFIG, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--separate-append", action="store_true",
                    help="run kvpool_append as its own kernel before each attention call")
    ap.add_argument("--tier-bench", action="store_true",
                    help="measure the host KV tier (offload / prefetch) instead of the step")
    ap.add_argument("--prefill", type=int, default=None, choices=[1, 2, 3],
                    help="measure a chunked-prefill workload instead of the decode step")
    ap.add_argument("--no-share", action="store_true",
                    help="plan the prefix-sharing workload without describing its shared prefixes")
    ap.add_argument("--no-early", action="store_true",
                    help="do not let the attention kernel gather before the previous kernel "
                         "completes (PKV_PLAN_EARLY_GATHER off)")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch every layer eagerly instead of replaying a CUDA graph")
    ap.add_argument("--layers", type=int, default=None,
                    help="run only the first N layers of the workload (small profiling "
                         "captures); the JSON line records it")
    ap.add_argument("--sweep", dest="sweep", action="store_true", default=None,
                    help="also time the other decode workloads and the chunked-prefill "
                         "workloads and record them under config.sweep (default on one GPU "
                         "for the default workload)")
    ap.add_argument("--no-sweep", dest="sweep", action="store_false")
    ap.add_argument("--curve", action="store_true",
                    help="time decode attention over a grid of batch sizes and context lengths "
                         "instead of the step (one JSON line of points)")
    args = ap.parse_args(argv)
    if args.warmup < 3 and args.impl == "ours":
        ap.error("--warmup must be >= 3")
    world, rank, local = _dist()
    if args.impl == "reference":
        return run_reference(args, world, rank)
    if args.tier_bench:
        return run_tier_bench(args)
    if args.curve:
        return run_curve(args)
    if args.prefill is not None:
        return run_prefill_bench(args)

    torch.cuda.set_device(local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        pg = dist
    sweep = args.sweep
    if sweep is None:
        sweep = world == 1 and args.config == DEFAULT_CONFIG and args.layers is None

    line = measure_decode(args.config, args, world, pg, local,
                          None if args.no_cpu_baseline else args.cpu_budget, args.layers)
    if sweep:
        # The other decode workloads (batch 1, 32, 16 and 128) and the chunked-prefill
        # workloads, each timed like the default one, one after the other with the
        # previous one's memory released.
        entries = {}
        for no in (1, 3, 4, 5):
            if no != args.config:
                entries[f"cfg{no}"] = sweep_entry(measure_decode(no, args, world, pg, local))
        for no in (1, 2, 3):
            entries[f"pf{no}"] = sweep_entry(measure_prefill(no, args.steps, args.warmup))
        entries["tier"] = measure_tier(5, args.steps, args.warmup)
        entries[f"cfg{args.config}"] = sweep_entry(line)
        line["config"]["sweep"] = entries
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()
    return 0


def kernel_source_sha() -> str:
    """sha256 of the code that decides a decode call's DRAM traffic: the kernel
    (csrc/decode.cu, then csrc/ptx.cuh) and the planner that splits the contexts
    (csrc/plan_host.cpp: the split parts' partial results are part of the traffic).
    Line comments and blank lines are left out, so that an edit of comments alone keeps
    a recorded capture valid, while any change of code does not."""
    import hashlib
    import re
    h = hashlib.sha256()
    for name in ("decode.cu", "ptx.cuh", "plan_host.cpp"):
        with open(os.path.join(ROOT, "paged_kv_gqa_tokentokvpool_gb300", "csrc", name)) as f:
            for line in f:
                code = re.sub(r"//.*$", "", line).rstrip()
                if code:
                    h.update(code.encode() + b"\n")
    return h.hexdigest()


def _profiled_traffic(config_no: int):
    """DRAM bytes per attention call from the committed ncu summary of this workload
    (profiles/traffic.txt), if it was taken on the current decode sources (as
    hashed by kernel_source_sha); else None."""
    sha = kernel_source_sha()
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.txt")) as f:
            for line in f:
                parts = line.split()
                if len(parts) >= 3 and not line.startswith("#") and parts[0] == str(config_no) \
                        and sha.startswith(parts[1]):
                    return int(parts[2])
    except OSError:
        pass
    return None


if __name__ == "__main__":
    sys.exit(main())
