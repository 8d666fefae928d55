"""Decode batches built twice from the same seeded inputs: once through the
library (native allocator + kernels, on the GPU) and once through the oracle
(reference allocator, oracle cache write / copy / attention, on the CPU).

For large workloads the oracle side works on a subset of the sequences, of
the kv heads, or both: the physical blocks those sequences reference are
gathered (from the pre-write input pool) into a compact pool with renumbered
tables and slots, keeping only the chosen kv heads (and the query heads that
read them).  A written block always belongs to its writer alone
(copy-on-write), so the subset's blocks are not touched by the other
sequences' writes; heads never mix in attention, so a head subset computes
exactly the rows it keeps.
"""
from __future__ import annotations

from typing import Optional

import numpy as np
import torch

import oracle
import paged_kv_cache_139_gb300 as pkv
import workloads
from paged_kv_cache_139_gb300.engine import PagedKVCache

ATOL, RTOL = 2e-3, 1e-2          # allclose form of max-abs 2e-3 / relative 1e-2


def _layout(w: workloads.Workload):
    """Sequence creation script: returns a list of ops on an allocator-like
    object and the decode order.  Ops: ("new", len) | ("fork", idx)."""
    ops = []
    if w.prompt_lens is not None:
        n = w.samples_per_prompt
        for p, plen in enumerate(w.prompt_lens):
            ops.append(("new", int(plen)))
            base = len(ops) - 1
            for _ in range(n - 1):
                ops.append(("fork", base))
    else:
        for c in w.context_lens:
            ops.append(("new", int(c) - 1))
    return ops


def _run_ops(alloc, ops):
    ids = []
    for op, arg in ops:
        ids.append(alloc.seq_new(arg) if op == "new" else alloc.fork(ids[arg]))
    return ids


def _suffix_order(w, ids):
    if w.suffix_lens is None:
        return []
    order = []
    for i, sid in enumerate(ids):
        order += [sid] * int(w.suffix_lens[i])
    return order


class Case:
    """One workload: the library side runs on construction (run_gpu), the
    oracle side on demand (oracle_out)."""

    def __init__(self, w: workloads.Workload, device="cuda", gen_device="cpu",
                 subset: Optional[list] = None, partition_size: Optional[int] = None, fused: bool = False,
                 kv_heads: Optional[list] = None):
        self.fused = fused
        self.w = w
        G = w.num_heads // w.num_kv_heads
        self.kv_heads = None if kv_heads is None else sorted(int(g) for g in kv_heads)
        # query heads the oracle computes (those reading the kept kv heads)
        self.q_heads = (np.arange(w.num_heads) if self.kv_heads is None else
                        np.array([g * G + j for g in self.kv_heads for j in range(G)], np.int64))
        self.device = torch.device(device)
        self.partition_size = w.partition_size if partition_size is None else partition_size
        t = workloads.tensors(w, device=gen_device)
        self.query = t["query"]
        self.key, self.value = t["key"], t["value"]
        self.suffix = workloads.suffix_tensors(w, device=gen_device)
        self.order = workloads.free_order(w.num_blocks, w.seed)
        self.ops = _layout(w)
        self._pool_k, self._pool_v = t["key_cache"], t["value_cache"]
        self.subset = subset
        # the oracle's allocator replay comes first: it tells which blocks the
        # subset needs, gathered from the input pool before the kernels run
        self._replay_reference()
        self._gather_oracle_pool()
        self.run_gpu()

    # -- reference allocator ----------------------------------------------------
    def _replay_reference(self):
        w = self.w
        ref = oracle.RefAllocator(w.num_blocks, w.block_size, self.order)
        ids = _run_ops(ref, self.ops)
        self.ref_ids = ids
        sfx = _suffix_order(w, ids)
        self.ref_sfx_slots, self.ref_sfx_pairs = ref.append_batch(sfx) if sfx else ([], [])
        self.ref_slots, self.ref_pairs = ref.append_batch(ids)
        mb = w.max_blocks_per_seq
        self.ref_tables = np.full((len(ids), mb), -1, np.int32)
        for i, sid in enumerate(ids):
            bt = ref.block_table(sid)
            self.ref_tables[i, :len(bt)] = bt
        self.ref_ctx = np.array([ref.seq_len(s) for s in ids], np.int32)
        self.ref = ref

    def _gather_oracle_pool(self):
        """Blocks the oracle needs: all of them, or the subset's (plus the
        sources of their copies)."""
        w = self.w
        if self.subset is None:
            self.sel = np.arange(w.num_seqs)
            self.blocks = np.arange(w.num_blocks)
        else:
            self.sel = np.asarray(sorted(self.subset))
            need = set()
            for i in self.sel:
                need.update(int(b) for b in self.ref_tables[i] if b >= 0)
            for src, dst in list(self.ref_sfx_pairs) + list(self.ref_pairs):
                if dst in need:
                    need.add(int(src))
            self.blocks = np.array(sorted(need), dtype=np.int64)
        idx = torch.from_numpy(self.blocks).to(self._pool_k.device)
        pk, pv = self._pool_k.index_select(0, idx), self._pool_v.index_select(0, idx)
        if self.kv_heads is not None:
            hidx = torch.tensor(self.kv_heads, device=pk.device)
            pk, pv = pk.index_select(1, hidx), pv.index_select(1, hidx)
        self.o_kc = oracle.bits16(pk)
        self.o_vc = oracle.bits16(pv)
        self.remap = {int(b): i for i, b in enumerate(self.blocks)}

    def _kv_rows(self, x):
        """New-token keys or values [T][Hkv][d] restricted to the kept kv heads."""
        return x if self.kv_heads is None else x[:, self.kv_heads]

    # -- library side -------------------------------------------------------------
    def run_gpu(self):
        w, d = self.w, self.device
        # the oracle's blocks were copied out already, so the engine may own the input pool
        kc = self._pool_k.to(d)
        vc = self._pool_v.to(d)
        self._pool_k = self._pool_v = None
        eng = PagedKVCache(w.num_blocks, w.num_kv_heads, w.head_dim, w.block_size, w.torch_dtype, d,
                           w.max_blocks_per_seq, self.order, key_cache=kc, value_cache=vc)
        ids = _run_ops(eng.alloc, self.ops)
        self.ids = ids
        sfx = _suffix_order(w, ids)
        if sfx:
            plan = eng.plan_step(sfx)
            self.sfx_slots, self.sfx_pairs = plan.slots, plan.pairs
            dev = eng.upload(plan)
            eng.copy_on_write(dev.pairs)
            eng.write(self.suffix["key"].to(d), self.suffix["value"].to(d), dev.slots)
        else:
            self.sfx_slots, self.sfx_pairs = np.empty(0, np.int64), np.empty((0, 2), np.int32)
        self.plan = eng.plan_step(ids)
        self.dev = eng.upload(self.plan)
        self.q_dev = self.query.to(d)
        self.k_dev, self.v_dev = self.key.to(d), self.value.to(d)
        if self.fused:
            # the new tokens' write inside the attention launch (paged_attention_decode_write)
            self.out = torch.empty_like(self.q_dev)
            prep = eng.prepare(self.q_dev, self.k_dev, self.v_dev, self.dev, self.out,
                               partition_size=self.partition_size, fused=True)
            assert prep._fused
            prep()
        else:
            self.out = eng.decode(self.q_dev, self.k_dev, self.v_dev, self.dev, partition_size=self.partition_size)
        self.eng = eng
        pkv.check()                     # raises (and clears) any error the device latched

    def rerun_attention(self, partition_size=None, out=None):
        ps = self.partition_size if partition_size is None else partition_size
        o = self.eng.attend(self.q_dev, self.dev, out=out, partition_size=ps)
        pkv.check()
        return o

    # -- oracle side -----------------------------------------------------------------
    def check_allocator(self):
        assert np.array_equal(self.plan.tables, self.ref_tables)
        assert np.array_equal(self.plan.context_lens, self.ref_ctx)
        assert self.plan.slots.tolist() == list(self.ref_slots)
        assert [tuple(p) for p in self.plan.pairs.tolist()] == list(self.ref_pairs)
        assert self.sfx_slots.tolist() == list(self.ref_sfx_slots)
        assert [tuple(p) for p in self.sfx_pairs.tolist()] == list(self.ref_sfx_pairs)

    def _remap_slots(self, slots):
        B = self.w.block_size
        out = []
        for s in slots:
            b = int(s) // B
            out.append(self.remap[b] * B + int(s) % B if b in self.remap else -1)
        return np.array(out, np.int64)

    def _remap_pairs(self, pairs):
        return [(self.remap[s], self.remap[d]) for s, d in pairs if d in self.remap]

    def oracle_caches(self):
        """The oracle's K/V pools (compact numbering) after the suffix and the
        decode step's copies and writes."""
        if getattr(self, "_o_done", False):
            return self.o_kc, self.o_vc
        kc, vc = self.o_kc, self.o_vc
        if self.suffix["key"].shape[0]:
            pr = self._remap_pairs(self.ref_sfx_pairs)
            if pr:
                oracle.copy_blocks(kc, pr)
                oracle.copy_blocks(vc, pr)
            oracle.cache_write(self._kv_rows(self.suffix["key"]), self._kv_rows(self.suffix["value"]), kc, vc,
                               self._remap_slots(self.ref_sfx_slots))
        pr = self._remap_pairs(self.ref_pairs)
        if pr:
            oracle.copy_blocks(kc, pr)
            oracle.copy_blocks(vc, pr)
        oracle.cache_write(self._kv_rows(self.key), self._kv_rows(self.value), kc, vc,
                           self._remap_slots(self.ref_slots))
        self._o_done = True
        return kc, vc

    def oracle_tables(self):
        t = self.ref_tables[self.sel].copy()
        for i in range(t.shape[0]):
            for j in range(t.shape[1]):
                if t[i, j] >= 0:
                    t[i, j] = self.remap[int(t[i, j])]
        return t

    def oracle_out(self, heads=None):
        """fp64 [len(sel)][len(q_heads)][d]; `heads`: optional list of (row in
        sel, index in q_heads)."""
        kc, vc = self.oracle_caches()
        q = self.query[torch.from_numpy(self.sel).to(self.query.device)]
        q = q[:, torch.from_numpy(self.q_heads).to(q.device)]
        return oracle.paged_attention(q, kc, vc, self.oracle_tables(), self.ref_ctx[self.sel],
                                      self.w.dtype, which=heads)

    def gpu_out(self, out=None):
        """The library's output [len(sel)][len(q_heads)][d] as fp64."""
        o = self.out if out is None else out
        o = o.index_select(0, torch.from_numpy(self.sel).to(o.device))
        return o.index_select(1, torch.from_numpy(self.q_heads).to(o.device)).double().cpu().numpy()

    def gpu_cache_blocks(self):
        """The library's K/V pools after the step, restricted to the oracle's
        blocks (and kv heads)."""
        idx = torch.from_numpy(self.blocks).to(self.device)
        k, v = self.eng.key_cache.index_select(0, idx), self.eng.value_cache.index_select(0, idx)
        if self.kv_heads is not None:
            hidx = torch.tensor(self.kv_heads, device=self.device)
            k, v = k.index_select(1, hidx), v.index_select(1, hidx)
        return oracle.bits16(k), oracle.bits16(v)


def assert_close(got: np.ndarray, want: np.ndarray, what: str = ""):
    err = np.abs(got - want)
    bound = ATOL + RTOL * np.abs(want)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside allclose(atol={ATOL}, rtol={RTOL}); "
                             f"worst at {i}: got {got[i]!r} want {want[i]!r}; max abs err {err.max():.3g}")
    return float(err.max()), float((err / np.maximum(np.abs(want), 1e-30)).max())
