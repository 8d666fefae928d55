"""Prompt-phase batches built twice from the same seeded inputs: through the
library (native allocator, copy_blocks, kv_reshape_and_cache and
paged_attention_prefill on the GPU) and through the oracle (reference
allocator, oracle copy, cache write and prompt-phase attention on the CPU).

Both pools start filled with NaN, so that slots no token was written to hold
values that would poison any result that read them.  A workload with
prefix_len > 0 shares one cached prefix between all requests (each forks the
prefix sequence, so the prefix's partly filled last block is copied on the
first write); with prefix_len = 0 each sequence first caches its own
context_lens[s] - query_lens[s] tokens.
"""
from __future__ import annotations

from typing import Optional

import numpy as np
import torch

import oracle
import paged_kv_cache_139_gb300 as pkv
import workloads
from paged_kv_cache_139_gb300.engine import PagedKVCache

ATOL, RTOL = 2e-3, 1e-2


def custom(S_ctx, S_new, H=4, Hkv=2, d=128, B=16, dtype="f16", seed=500, prefix_len=0, extra_blocks=7):
    ctx = np.asarray(S_ctx, np.int64)
    n = np.asarray(S_new, np.int64)
    mb = max(1, -(-int(ctx.max()) // B))
    if prefix_len:
        nb = -(-prefix_len // B) + int(sum(-(-int(c) // B) - prefix_len // B for c in ctx)) + extra_blocks
    else:
        nb = int(sum(-(-int(c) // B) for c in ctx)) + extra_blocks
    return workloads.Workload(f"prefill custom ctx={list(ctx)} new={list(n)}", len(ctx), H, Hkv, d, B, dtype,
                              ctx, mb, nb, seed, query_lens=n, prefix_len=prefix_len)


def _ops(w):
    """(cached-token count per sequence creation, fork or not)."""
    if w.prefix_len:
        return [("prefix", w.prefix_len)] + [("fork", 0)] * w.num_seqs
    return [("new", int(c - n)) for c, n in zip(w.context_lens, w.query_lens)]


def _slots_of(table, B, t0, t1):
    return np.array([table[t // B] * B + t % B for t in range(t0, t1)], np.int64)


class PrefillCase:
    def __init__(self, w: workloads.Workload, device="cuda", nan_pool=True, order=None):
        self.w = w
        self.device = torch.device(device)
        t = workloads.prefill_tensors(w, "cpu")
        self.t = t
        self.order = workloads.free_order(w.num_blocks, w.seed) if order is None else np.asarray(order, np.int32)
        self.nan_pool = nan_pool
        self._run_reference_allocator()
        self._run_gpu()

    # -- reference allocator: ids, cached-token slots, then the new tokens' plan
    def _setup(self, alloc):
        w, B = self.w, self.w.block_size
        seqs, cached_slots = [], []
        if w.prefix_len:
            p = alloc.seq_new(w.prefix_len)
            cached_slots.append(_slots_of(alloc.block_table(p), B, 0, w.prefix_len))
            seqs = [alloc.fork(p) for _ in range(w.num_seqs)]
        else:
            for op, c in _ops(w):
                s = alloc.seq_new(c)
                seqs.append(s)
                cached_slots.append(_slots_of(alloc.block_table(s), B, 0, c))
        slots = np.concatenate(cached_slots) if cached_slots else np.empty(0, np.int64)
        return seqs, slots

    def _run_reference_allocator(self):
        w = self.w
        ref = oracle.RefAllocator(w.num_blocks, w.block_size, self.order)
        seqs, self.ref_cached_slots = self._setup(ref)
        order = np.repeat(np.asarray(seqs, np.int32), w.query_lens)
        self.ref_slots, self.ref_pairs = ref.append_batch(order) if order.size else ([], [])
        self.ref_tables = np.full((w.num_seqs, w.max_blocks_per_seq), -1, np.int32)
        for i, s in enumerate(seqs):
            bt = ref.block_table(s)
            self.ref_tables[i, :len(bt)] = bt
        self.ref_ctx = np.array([ref.seq_len(s) for s in seqs], np.int32)
        self.query_start = np.concatenate([[0], np.cumsum(w.query_lens)]).astype(np.int32)

    def _run_gpu(self):
        w, d = self.w, self.device
        eng = PagedKVCache(w.num_blocks, w.num_kv_heads, w.head_dim, w.block_size, w.torch_dtype, d,
                           w.max_blocks_per_seq, self.order)
        fill = float("nan") if self.nan_pool else 0.0
        eng.key_cache.fill_(fill)
        eng.value_cache.fill_(fill)
        self.fill_bits = int(oracle.bits16(eng.key_cache[:1, :1, :1, :1])[0, 0, 0, 0])
        seqs, cached_slots = self._setup(eng.alloc)
        self.cached_slots = cached_slots
        if cached_slots.size:
            eng.write(self.t["prefix_key"].to(d), self.t["prefix_value"].to(d),
                      torch.from_numpy(cached_slots).to(d))
        self.plan = eng.plan_prefill(seqs, w.query_lens)
        self.dev = eng.upload_prefill(self.plan)
        self.q_dev = self.t["query"].to(d)
        self.out = eng.prefill(self.q_dev, self.t["key"].to(d), self.t["value"].to(d), self.dev)
        self.eng = eng
        pkv.check()

    def rerun(self, out=None, max_query_len=None):
        o = torch.empty_like(self.q_dev) if out is None else out
        pkv.paged_attention_prefill(o, self.q_dev, self.eng.key_cache, self.eng.value_cache, self.dev.tables,
                                    self.dev.context_lens, self.dev.query_start,
                                    max_query_len=self.dev.max_query_len if max_query_len is None
                                    else max_query_len)
        pkv.check()
        return o

    # -- oracle side ---------------------------------------------------------------
    def check_allocator(self):
        assert np.array_equal(self.plan.tables, self.ref_tables)
        assert np.array_equal(self.plan.context_lens, self.ref_ctx)
        assert np.array_equal(self.cached_slots, self.ref_cached_slots)
        assert self.plan.slots.tolist() == list(self.ref_slots)
        assert [tuple(p) for p in self.plan.pairs.tolist()] == list(self.ref_pairs)
        assert np.array_equal(self.plan.query_start, self.query_start)

    def oracle_caches(self):
        if getattr(self, "_oc", None) is not None:
            return self._oc
        w = self.w
        shape = (w.num_blocks, w.num_kv_heads, w.block_size, w.head_dim)
        kc = np.full(shape, self.fill_bits, np.uint16)
        vc = np.full(shape, self.fill_bits, np.uint16)
        if len(self.ref_cached_slots):
            oracle.cache_write(self.t["prefix_key"], self.t["prefix_value"], kc, vc, self.ref_cached_slots)
        if len(self.ref_pairs):
            oracle.copy_blocks(kc, self.ref_pairs)
            oracle.copy_blocks(vc, self.ref_pairs)
        if len(self.ref_slots):
            oracle.cache_write(self.t["key"], self.t["value"], kc, vc, np.asarray(self.ref_slots, np.int64))
        self._oc = (kc, vc)
        return self._oc

    def gpu_caches(self):
        return oracle.bits16(self.eng.key_cache), oracle.bits16(self.eng.value_cache)

    def oracle_out(self, which=None):
        kc, vc = self.oracle_caches()
        return oracle.paged_prefill(self.t["query"], kc, vc, self.ref_tables, self.ref_ctx, self.query_start,
                                    self.w.dtype, which=which)

    def sample_rows(self, n_per_seq=3, heads=None, seed=0):
        """(token, head) pairs: each sequence's first, last and some middle new
        tokens, over a spread of heads."""
        rng = np.random.default_rng(seed)
        H = self.w.num_heads
        heads = list(range(H)) if heads is None else heads
        which = []
        for s in range(self.w.num_seqs):
            a, b = int(self.query_start[s]), int(self.query_start[s + 1])
            if b == a:
                continue
            toks = {a, b - 1} | {int(x) for x in rng.integers(a, b, size=n_per_seq)}
            for t in sorted(toks):
                which.append((t, int(heads[rng.integers(len(heads))])))
        return which


def assert_rows_close(got: np.ndarray, want: np.ndarray, which, what: str):
    g = np.array([got[t, h] for t, h in which], np.float64)
    e = np.array([want[t, h] for t, h in which], np.float64)
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    err = np.abs(g - e)
    bad = err > ATOL + RTOL * np.abs(e)
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} elements outside tolerance; "
                           f"max abs err {err.max():.3g}")
