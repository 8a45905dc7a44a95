"""Seeded synthetic decode workloads shared by the tests and the benchmark.

This module only draws random numbers and lays out slot lists. It holds none of
the attention arithmetic: neither the oracle nor the CUDA path is imported here,
and both receive what this module produces as plain arrays.

The shapes follow the decode workloads of the pages this library is built from:
Qwen3-4B (36 layers, 32 query heads sharing 8 KV heads, head_dim 128) and the
full-attention layers of the Qwen3.5 hybrid (head_dim 256), per "Pegainfer:
纯Rust+CUDA构建的LLM推理引擎", sections "支持的模型架构" and "1. 注意力机制优化" /
"2. Qwen3.5的混合架构支持", over a token-granular KV pool with page size 1
("Agent-Infer", section "分页 KV 缓存").

Recipe (identical for every workload):
  * context lengths are integers, drawn uniformly (inclusive bounds) or
    log-uniformly (round(exp(U[ln a, ln b]))) with numpy's PCG64 seeded by
    ``seed``;
  * slot placement: one ``permutation(pool_slots)``; each request takes the next
    run of unused slots, so slots are distinct and scattered. A request of
    context L holds L - 1 history slots plus the slot of the token appended this
    step, which is the LAST entry of its CSR list;
  * prefix-sharing groups list the same prefix slot ids first, then private
    suffix slots;
  * q, K, V and the appended rows are N(0, 1) drawn in fp32 by a
    ``torch.Generator`` (Philox on CUDA, MT on CPU) and rounded to bf16
    (round-to-nearest-even); K is multiplied by ``k_scale`` before rounding.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

BF16_NAN_BITS = 0x7FC0


@dataclass
class Workload:
    name: str
    layers: int
    batch: int
    n_qo_heads: int
    n_kv_heads: int
    head_dim: int
    pool_slots: int
    sm_scale: float
    k_scale: float
    seed: int
    lengths: np.ndarray            # [batch] int64, context incl. the appended token
    kv_indptr: np.ndarray          # [batch + 1] int32
    kv_indices: np.ndarray         # [N] int32
    append_slots: np.ndarray       # [n_append] int32 (last slot of each non-empty request)
    append_rows: np.ndarray        # [n_append] int64, request index of each appended row
    description: str = ""
    meta: dict = field(default_factory=dict)

    @property
    def total_tokens(self) -> int:
        return int(self.kv_indptr[-1])

    @property
    def group(self) -> int:
        return self.n_qo_heads // self.n_kv_heads

    def kv_bytes_per_layer(self) -> int:
        """Algorithmic K+V bytes one layer's attention reads (each listed slot once)."""
        return self.total_tokens * 2 * self.n_kv_heads * self.head_dim * 2

    def unique_kv_bytes_per_layer(self) -> int:
        return int(np.unique(self.kv_indices).size) * 2 * self.n_kv_heads * self.head_dim * 2


def _sm_scale(head_dim: int) -> float:
    return float(np.float32(1.0 / math.sqrt(head_dim)))


def _finish(name, layers, hq, hkv, d, pool_slots, k_scale, seed, lengths, slot_lists,
            description="", meta=None) -> Workload:
    lengths = np.asarray(lengths, dtype=np.int64)
    indptr = np.zeros(len(lengths) + 1, dtype=np.int64)
    indptr[1:] = np.cumsum(lengths)
    if indptr[-1] >= 2**31:
        raise ValueError("total context exceeds int32 CSR range")
    indices = (np.concatenate(slot_lists) if slot_lists else np.zeros(0)).astype(np.int32)
    assert indices.size == indptr[-1]
    nonempty = np.nonzero(lengths > 0)[0]
    append_slots = indices[indptr[nonempty + 1] - 1].astype(np.int32)
    return Workload(name=name, layers=layers, batch=len(lengths), n_qo_heads=hq,
                    n_kv_heads=hkv, head_dim=d, pool_slots=pool_slots,
                    sm_scale=_sm_scale(d), k_scale=k_scale, seed=seed, lengths=lengths,
                    kv_indptr=indptr.astype(np.int32), kv_indices=indices,
                    append_slots=append_slots, append_rows=nonempty.astype(np.int64),
                    description=description, meta=meta or {})


def scattered_workload(lengths, *, n_qo_heads=32, n_kv_heads=8, head_dim=128,
                       pool_slots=None, layers=1, k_scale=1.0, seed=0,
                       name="custom", description="") -> Workload:
    """Requests with private, randomly scattered slot lists."""
    lengths = [int(x) for x in lengths]
    need = sum(lengths)
    if pool_slots is None:
        pool_slots = max(16, 2 * need)
    if need > pool_slots:
        raise ValueError("pool too small for the requested contexts")
    rng = np.random.default_rng(seed)
    perm = rng.permutation(pool_slots)
    lists, off = [], 0
    for L in lengths:
        lists.append(perm[off:off + L])
        off += L
    return _finish(name, layers, n_qo_heads, n_kv_heads, head_dim, pool_slots, k_scale,
                   seed, lengths, lists, description)


def prefix_shared_workload(prefix_lens, suffix_lens, group_size, *, n_qo_heads=32,
                           n_kv_heads=8, head_dim=128, pool_slots=None, layers=1,
                           k_scale=1.0, seed=0, name="prefix", description="") -> Workload:
    """Groups of ``group_size`` requests; each group lists the same prefix slots first."""
    n_groups = len(prefix_lens)
    assert len(suffix_lens) == n_groups * group_size
    need = sum(prefix_lens) + sum(suffix_lens)
    if pool_slots is None:
        pool_slots = max(16, 2 * need)
    rng = np.random.default_rng(seed)
    perm = rng.permutation(pool_slots)
    off = 0
    prefixes = []
    for P in prefix_lens:
        prefixes.append(perm[off:off + P])
        off += P
    lists, lengths = [], []
    for g in range(n_groups):
        for j in range(group_size):
            s = suffix_lens[g * group_size + j]
            lists.append(np.concatenate([prefixes[g], perm[off:off + s]]))
            off += s
            lengths.append(prefix_lens[g] + s)
    return _finish(name, layers, n_qo_heads, n_kv_heads, head_dim, pool_slots, k_scale,
                   seed, lengths, lists, description,
                   meta={"prefix_lens": list(map(int, prefix_lens)), "group_size": group_size})


CONFIG_DESCRIPTIONS = {
    1: "1 layer, batch 1, 32Q/8KV, head_dim 128, context 512, 4096-slot pool",
    2: "Qwen3-4B-shaped decode step: 36 layers, batch 8, 32Q/8KV, head_dim 128, "
       "contexts U[512,4096], 65536-slot pools",
    3: "prefix-sharing step: 36 layers, batch 32 = 4 groups x 8, prefixes U[2048,8192] "
       "shared, suffixes U[64,2048], 131072-slot pools",
    4: "hybrid full-attention layers: 8 layers, head_dim 256, 16Q/4KV, batch 16, "
       "contexts U[8192,32768], 2^20-slot pools, K x 0.5",
    5: "skewed long-context batch: 1 layer, batch 128, 127 contexts log-U[128,32768] "
       "plus one of 131072, 2^22-slot pool",
}


def config_workload(no: int) -> Workload:
    """The five decode workloads the benchmark and the parity tests use (seed 1000 + no)."""
    seed = 1000 + no
    rng = np.random.default_rng(seed)
    desc = CONFIG_DESCRIPTIONS[no]
    if no == 1:
        return scattered_workload([512], pool_slots=4096, seed=seed, name="cfg1",
                                  description=desc)
    if no == 2:
        lengths = rng.integers(512, 4096, size=8, endpoint=True)
        return scattered_workload(lengths, pool_slots=65536, layers=36, seed=seed,
                                  name="cfg2", description=desc)
    if no == 3:
        prefix = rng.integers(2048, 8192, size=4, endpoint=True)
        suffix = rng.integers(64, 2048, size=32, endpoint=True)
        return prefix_shared_workload(list(prefix), list(suffix), 8, pool_slots=131072,
                                      layers=36, seed=seed, name="cfg3", description=desc)
    if no == 4:
        lengths = rng.integers(8192, 32768, size=16, endpoint=True)
        return scattered_workload(lengths, n_qo_heads=16, n_kv_heads=4, head_dim=256,
                                  pool_slots=1 << 20, layers=8, k_scale=0.5, seed=seed,
                                  name="cfg4", description=desc)
    if no == 5:
        lengths = np.rint(np.exp(rng.uniform(math.log(128), math.log(32768), size=127)))
        lengths = np.clip(lengths, 128, 32768).astype(np.int64)
        pos = int(rng.integers(0, 128))
        lengths = np.insert(lengths, pos, 131072)
        return scattered_workload(lengths, pool_slots=1 << 22, seed=seed, name="cfg5",
                                  description=desc)
    raise ValueError(f"unknown config {no}")


# ---------------------------------------------------------------------------
# value generation
# ---------------------------------------------------------------------------

def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _fill_normal_bf16(out: torch.Tensor, gen: torch.Generator, scale: float = 1.0,
                      chunk_elems: int = 1 << 26) -> None:
    """Fill a bf16 tensor with N(0,1)*scale drawn in fp32, rounded RNE, chunk by chunk."""
    flat = out.view(-1)
    for s in range(0, flat.numel(), chunk_elems):
        e = min(flat.numel(), s + chunk_elems)
        x = torch.randn(e - s, generator=gen, device=out.device, dtype=torch.float32)
        if scale != 1.0:
            x.mul_(scale)
        flat[s:e].copy_(x.to(torch.bfloat16))


@dataclass
class LayerTensors:
    q: torch.Tensor        # [B, Hq, D] bf16
    k_pool: torch.Tensor   # [S, Hkv, D] bf16 (before append)
    v_pool: torch.Tensor   # [S, Hkv, D] bf16 (before append)
    k_new: torch.Tensor    # [n_append, Hkv, D] bf16
    v_new: torch.Tensor    # [n_append, Hkv, D] bf16


def layer_tensors(wl: Workload, layer: int, device="cpu", poison_unreferenced=False,
                  pools=True) -> LayerTensors:
    """Seeded tensors of one layer. With ``poison_unreferenced`` every pool slot that no
    request lists (and the appended slots, before the append) holds bf16 NaN, so any
    stray read turns an output into NaN."""
    device = torch.device(device)
    gen = _gen(device, wl.seed * 1000 + layer)
    B, Hq, Hkv, D, S = wl.batch, wl.n_qo_heads, wl.n_kv_heads, wl.head_dim, wl.pool_slots
    q = torch.empty(B, Hq, D, dtype=torch.bfloat16, device=device)
    _fill_normal_bf16(q, gen)
    n_app = len(wl.append_slots)
    k_new = torch.empty(n_app, Hkv, D, dtype=torch.bfloat16, device=device)
    v_new = torch.empty(n_app, Hkv, D, dtype=torch.bfloat16, device=device)
    _fill_normal_bf16(k_new, gen, wl.k_scale)
    _fill_normal_bf16(v_new, gen)
    if pools:
        k_pool = torch.empty(S, Hkv, D, dtype=torch.bfloat16, device=device)
        v_pool = torch.empty(S, Hkv, D, dtype=torch.bfloat16, device=device)
        _fill_normal_bf16(k_pool, gen, wl.k_scale)
        _fill_normal_bf16(v_pool, gen)
        if poison_unreferenced:
            keep = torch.zeros(S, dtype=torch.bool, device=device)
            keep[torch.as_tensor(wl.kv_indices, dtype=torch.int64, device=device)] = True
            keep[torch.as_tensor(wl.append_slots, dtype=torch.int64, device=device)] = False
            nan = torch.tensor(BF16_NAN_BITS, dtype=torch.int16, device=device)
            k_pool.view(torch.int16)[~keep] = nan
            v_pool.view(torch.int16)[~keep] = nan
    else:
        k_pool = v_pool = None
    return LayerTensors(q, k_pool, v_pool, k_new, v_new)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Raw bf16 bit patterns of a tensor as a host uint16 array (no arithmetic)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


# ---------------------------------------------------------------------------
# chunked prefill ("Agent-Infer", section "连续批处理": chunks of 512 tokens, 64
# while decodes are running)
# ---------------------------------------------------------------------------

@dataclass
class PrefillWorkload:
    name: str
    layers: int
    batch: int
    n_qo_heads: int
    n_kv_heads: int
    head_dim: int
    pool_slots: int
    sm_scale: float
    k_scale: float
    seed: int
    chunks: np.ndarray         # [batch] int64, query tokens of each chunk
    contexts: np.ndarray       # [batch] int64, listed slots incl. the chunk's own
    qo_indptr: np.ndarray      # [batch + 1] int32
    kv_indptr: np.ndarray      # [batch + 1] int32
    kv_indices: np.ndarray     # [N] int32
    chunk_slots: np.ndarray    # [qo_indptr[-1]] int32: the slot of every chunk token
    description: str = ""

    @property
    def total_q(self) -> int:
        return int(self.qo_indptr[-1])

    @property
    def total_tokens(self) -> int:
        return int(self.kv_indptr[-1])

    def attended_pairs(self) -> int:
        """Sum over chunk tokens of the list entries each attends (causal)."""
        c, l = self.chunks.astype(np.int64), self.contexts.astype(np.int64)
        return int(np.sum(c * (l - c) + c * (c + 1) // 2))


def prefill_workload(chunks, contexts, *, n_qo_heads=32, n_kv_heads=8, head_dim=128,
                     pool_slots=None, layers=1, k_scale=1.0, seed=0, name="prefill",
                     description="") -> PrefillWorkload:
    """Requests whose newest chunks[b] tokens are a prefill chunk: each lists
    contexts[b] >= chunks[b] scattered slots, the chunk's slots last."""
    chunks = np.asarray([int(x) for x in chunks], dtype=np.int64)
    contexts = np.asarray([int(x) for x in contexts], dtype=np.int64)
    assert chunks.size == contexts.size and np.all((0 <= chunks) & (chunks <= contexts))
    need = int(contexts.sum())
    if pool_slots is None:
        pool_slots = max(16, 2 * need)
    if need > pool_slots:
        raise ValueError("pool too small for the requested contexts")
    rng = np.random.default_rng(seed)
    perm = rng.permutation(pool_slots)
    lists, off = [], 0
    for L in contexts:
        lists.append(perm[off:off + L])
        off += int(L)
    kv_indptr = np.zeros(chunks.size + 1, dtype=np.int64)
    kv_indptr[1:] = np.cumsum(contexts)
    qo_indptr = np.zeros(chunks.size + 1, dtype=np.int64)
    qo_indptr[1:] = np.cumsum(chunks)
    if kv_indptr[-1] >= 2**31:
        raise ValueError("total context exceeds int32 CSR range")
    indices = (np.concatenate(lists) if lists else np.zeros(0)).astype(np.int32)
    chunk_slots = (np.concatenate([lst[len(lst) - c:] for lst, c in zip(lists, chunks)])
                   if lists else np.zeros(0)).astype(np.int32)
    return PrefillWorkload(name=name, layers=layers, batch=int(chunks.size),
                           n_qo_heads=n_qo_heads, n_kv_heads=n_kv_heads, head_dim=head_dim,
                           pool_slots=pool_slots, sm_scale=_sm_scale(head_dim), k_scale=k_scale,
                           seed=seed, chunks=chunks, contexts=contexts,
                           qo_indptr=qo_indptr.astype(np.int32),
                           kv_indptr=kv_indptr.astype(np.int32), kv_indices=indices,
                           chunk_slots=chunk_slots, description=description)


PREFILL_DESCRIPTIONS = {
    1: "chunked prefill, Qwen3-4B shape: 36 layers, 4 requests x 512-token chunks at "
       "contexts U[512,8192], 32Q/8KV, head_dim 128, 65536-slot pools",
    2: "chunked prefill beside decodes: 36 layers, 8 requests x 64-token chunks at contexts "
       "U[64,16384], 32Q/8KV, head_dim 128, 2^18-slot pools",
    3: "chunked prefill, hybrid full-attention layers: 8 layers, 4 requests x 512-token chunks "
       "at contexts U[512,32768], 16Q/4KV, head_dim 256, K scaled 0.5, 2^18-slot pools",
}


def prefill_config(no: int) -> PrefillWorkload:
    """The chunked-prefill workloads (seed 2000 + no)."""
    seed = 2000 + no
    rng = np.random.default_rng(seed)
    desc = PREFILL_DESCRIPTIONS[no]
    if no == 1:
        ctx = rng.integers(512, 8192, size=4, endpoint=True)
        return prefill_workload([512] * 4, ctx, pool_slots=65536, layers=36, seed=seed,
                                name="pf1", description=desc)
    if no == 2:
        ctx = rng.integers(64, 16384, size=8, endpoint=True)
        return prefill_workload([64] * 8, ctx, pool_slots=1 << 18, layers=36, seed=seed,
                                name="pf2", description=desc)
    if no == 3:
        ctx = rng.integers(512, 32768, size=4, endpoint=True)
        return prefill_workload([512] * 4, ctx, n_qo_heads=16, n_kv_heads=4, head_dim=256,
                                pool_slots=1 << 18, layers=8, k_scale=0.5, seed=seed,
                                name="pf3", description=desc)
    raise ValueError(f"unknown prefill config {no}")


def prefill_tensors(pw: PrefillWorkload, layer: int, device="cpu", poison_unreferenced=False):
    """Seeded tensors of one layer: (q [NQ, Hq, D], k_pool, v_pool before the chunk's
    append, k_new, v_new [NQ, Hkv, D] the chunk's rows). With ``poison_unreferenced``
    unlisted slots and the chunk's own slots (before the append) hold bf16 NaN."""
    device = torch.device(device)
    gen = _gen(device, pw.seed * 1000 + layer)
    NQ, Hq, Hkv, D, S = pw.total_q, pw.n_qo_heads, pw.n_kv_heads, pw.head_dim, pw.pool_slots
    q = torch.empty(NQ, Hq, D, dtype=torch.bfloat16, device=device)
    _fill_normal_bf16(q, gen)
    k_new = torch.empty(NQ, Hkv, D, dtype=torch.bfloat16, device=device)
    v_new = torch.empty(NQ, Hkv, D, dtype=torch.bfloat16, device=device)
    _fill_normal_bf16(k_new, gen, pw.k_scale)
    _fill_normal_bf16(v_new, gen)
    k_pool = torch.empty(S, Hkv, D, dtype=torch.bfloat16, device=device)
    v_pool = torch.empty(S, Hkv, D, dtype=torch.bfloat16, device=device)
    _fill_normal_bf16(k_pool, gen, pw.k_scale)
    _fill_normal_bf16(v_pool, gen)
    if poison_unreferenced:
        keep = torch.zeros(S, dtype=torch.bool, device=device)
        keep[torch.as_tensor(pw.kv_indices, dtype=torch.int64, device=device)] = True
        keep[torch.as_tensor(pw.chunk_slots, dtype=torch.int64, device=device)] = False
        nan = torch.tensor(BF16_NAN_BITS, dtype=torch.int16, device=device)
        k_pool.view(torch.int16)[~keep] = nan
        v_pool.view(torch.int16)[~keep] = nan
    return q, k_pool, v_pool, k_new, v_new
