"""A one-layer paged KV cache engine: the device K/V pools, the native block
allocator, and the decode step that ties the three device calls together.

One decode iteration ("vLLM & PagedAttention: Efficient Memory Management
for LLM Serving", §V): allocate physical blocks for the batch's new tokens
(copy-on-write where a sequence writes into a shared block, §VII), copy the
shared blocks, write the new keys and values at their slots, then run the
paged attention kernel over the block tables.  Host bookkeeping happens in
the native allocator; the four device steps run in libpkv's kernels.
"""
from __future__ import annotations

import dataclasses
from typing import Optional, Sequence

import numpy as np
import torch

import ctypes
import math

from . import (BlockAllocator, PkvError, copy_blocks, kv_reshape_and_cache, make_workspace,
               paged_attention_decode, paged_attention_prefill, paged_attention_workspace_size, swap_blocks)
from ._lib import load


@dataclasses.dataclass
class StepPlan:
    """Host-side result of allocating one decode step."""

    seqs: np.ndarray          # int32 [n]
    slots: np.ndarray         # int64 [n]
    pairs: np.ndarray         # int32 [m][2] copy-on-write (src, dst)
    tables: np.ndarray        # int32 [n][max_blocks]
    context_lens: np.ndarray  # int32 [n]


@dataclasses.dataclass
class DeviceStep:
    """The same plan on the device."""

    slots: torch.Tensor
    pairs: torch.Tensor
    tables: torch.Tensor
    context_lens: torch.Tensor
    max_context_len: int


@dataclasses.dataclass
class PrefillPlan:
    """Host-side result of allocating the new tokens of a prompt-phase step."""

    seqs: np.ndarray          # int32 [n]
    slots: np.ndarray         # int64 [T], sequence-major
    pairs: np.ndarray         # int32 [m][2] copy-on-write (src, dst)
    tables: np.ndarray        # int32 [n][max_blocks]
    context_lens: np.ndarray  # int32 [n]
    query_start: np.ndarray   # int32 [n + 1]


@dataclasses.dataclass
class DevicePrefill:
    slots: torch.Tensor
    pairs: torch.Tensor
    tables: torch.Tensor
    context_lens: torch.Tensor
    query_start: torch.Tensor
    max_query_len: int


class StagedInputs:
    """A step's host inputs in one pinned buffer and their device copies in one
    device buffer, laid out alike (each tensor 256-byte aligned): a step then
    moves all its inputs with a single host-to-device copy instead of one per
    tensor.  Write the step's inputs into `host[name]`, call `upload()`, and
    pass `dev[name]` to the device calls."""

    def __init__(self, specs, device):
        """specs: {name: (shape, dtype)}."""
        self.device = torch.device(device)
        offs, off = {}, 0
        for name, (shape, dtype) in specs.items():
            n = int(np.prod(shape)) * torch.tensor([], dtype=dtype).element_size()
            offs[name] = (off, n, tuple(shape), dtype)
            off += (n + 255) // 256 * 256
        self.nbytes = off
        self._hbuf = torch.empty(max(off, 1), dtype=torch.uint8).pin_memory()
        self._dbuf = torch.empty(max(off, 1), dtype=torch.uint8, device=self.device)
        view = lambda buf, o, n, shape, dt: buf[o:o + n].view(dt).view(shape)
        self.host = {k: view(self._hbuf, *v) for k, v in offs.items()}
        self.dev = {k: view(self._dbuf, *v) for k, v in offs.items()}

    def upload(self, stream: Optional[torch.cuda.Stream] = None) -> None:
        """One asynchronous copy of every input (on `stream`, default current)."""
        s = stream or torch.cuda.current_stream(self.device)
        with torch.cuda.stream(s):
            self._dbuf.copy_(self._hbuf, non_blocking=True)


class GraphStep:
    """A whole step -- one staged upload of its inputs, its device calls, the
    read-back of its output -- captured once in a CUDA graph and replayed:
    the GPU runs the copies and kernels back to back with no host round trip
    between them.  `prepare(stream)` must build the device calls (for example
    PagedKVCache.prepare / prepare_prefill) on the stream it is given, with
    the staged inputs' device views as arguments; the buffers must stay fixed
    (their contents may change between replays)."""

    def __init__(self, staged: StagedInputs, prepare, out: torch.Tensor, host_out: torch.Tensor, warmup: int = 2):
        dev = staged.device
        self._stream = torch.cuda.Stream(dev)
        self._prep = prepare(self._stream)
        self._staged, self._out, self._host_out = staged, out, host_out
        self._stream.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(self._stream):
            for _ in range(warmup):                  # first launches configure the kernels
                self._body()
        self._stream.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=self._stream):
            self._body()
        self.device = dev

    def _body(self):
        self._staged.upload(self._stream)
        self._prep()
        self._host_out.copy_(self._out, non_blocking=True)

    def replay(self) -> None:
        self.graph.replay()


class HostKVPool:
    """The CPU side of swapping ("vLLM & PagedAttention" §VIII, Fig. 4): K and
    V pools in pinned host memory, which the GPU addresses directly, and the
    CPU block allocator that owns them."""

    def __init__(self, num_blocks: int, num_kv_heads: int, head_dim: int, block_size: int, dtype: torch.dtype,
                 free_order: Optional[Sequence[int]] = None):
        shape = (num_blocks, num_kv_heads, block_size, head_dim)
        self.key_cache = torch.empty(shape, dtype=dtype, pin_memory=True)
        self.value_cache = torch.empty(shape, dtype=dtype, pin_memory=True)
        self.alloc = BlockAllocator(num_blocks, block_size, free_order)
        self.num_blocks, self.block_size = num_blocks, block_size


class PagedKVCache:
    def __init__(self, num_blocks: int, num_kv_heads: int, head_dim: int, block_size: int,
                 dtype: torch.dtype, device, max_blocks_per_seq: int,
                 free_order: Optional[Sequence[int]] = None,
                 key_cache: Optional[torch.Tensor] = None, value_cache: Optional[torch.Tensor] = None):
        shape = (num_blocks, num_kv_heads, block_size, head_dim)
        self.device = torch.device(device)
        self.key_cache = key_cache if key_cache is not None else torch.empty(shape, dtype=dtype, device=self.device)
        self.value_cache = value_cache if value_cache is not None else torch.empty(shape, dtype=dtype,
                                                                                    device=self.device)
        assert tuple(self.key_cache.shape) == shape and tuple(self.value_cache.shape) == shape
        self.alloc = BlockAllocator(num_blocks, block_size, free_order)
        self.num_blocks, self.num_kv_heads, self.head_dim, self.block_size = shape[0], shape[1], shape[3], shape[2]
        self.max_blocks_per_seq = max_blocks_per_seq
        self._ws: Optional[torch.Tensor] = None
        self._ws_retired: list = []

    # -- host bookkeeping ------------------------------------------------------
    def new_sequence(self, length: int) -> int:
        return self.alloc.seq_new(length)

    def fork(self, seq: int) -> int:
        return self.alloc.fork(seq)

    def free(self, seq: int) -> None:
        self.alloc.free(seq)

    def plan_step(self, seqs: Sequence[int]) -> StepPlan:
        """Append one token to each sequence (all or nothing) and build the
        tables the attention kernel reads."""
        s = np.asarray(seqs, dtype=np.int32)
        slots, pairs = self.alloc.append_batch(s)
        tables, ctx = self.alloc.build_block_tables(s, self.max_blocks_per_seq)
        return StepPlan(s, slots, pairs, tables, ctx)

    def plan_beam_step(self, beams: Sequence[int], parents: Sequence[int]) -> StepPlan:
        """One beam-search step on the host: new candidate i continues
        beams[parents[i]] (fork where a parent has several children, prune
        the rest), each appends its token; the plan holds the new beams."""
        new, slots, pairs = self.alloc.beam_step(beams, parents)
        s = np.asarray(new, dtype=np.int32)
        tables, ctx = self.alloc.build_block_tables(s, self.max_blocks_per_seq)
        return StepPlan(s, slots, pairs, tables, ctx)

    def plan_tables(self, seqs: Sequence[int]) -> StepPlan:
        """Tables of the sequences as they stand (no new token)."""
        s = np.asarray(seqs, dtype=np.int32)
        tables, ctx = self.alloc.build_block_tables(s, self.max_blocks_per_seq)
        return StepPlan(s, np.empty(0, np.int64), np.empty((0, 2), np.int32), tables, ctx)

    def plan_prefill(self, seqs: Sequence[int], new_tokens: Sequence[int]) -> PrefillPlan:
        """Append new_tokens[i] tokens to seqs[i] (all or nothing): the prompt
        phase of a request, or its own input after a forked shared prefix."""
        s = np.asarray(seqs, dtype=np.int32)
        n = np.asarray(new_tokens, dtype=np.int64)
        slots, pairs = self.alloc.append_batch(np.repeat(s, n).astype(np.int32))
        tables, ctx = self.alloc.build_block_tables(s, self.max_blocks_per_seq)
        qs = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
        return PrefillPlan(s, slots, pairs, tables, ctx, qs)

    def upload_prefill(self, plan: PrefillPlan, non_blocking: bool = False) -> DevicePrefill:
        d = self.device
        n = np.diff(plan.query_start)
        return DevicePrefill(
            slots=torch.from_numpy(plan.slots).to(d, non_blocking=non_blocking),
            pairs=torch.from_numpy(np.ascontiguousarray(plan.pairs)).to(d, non_blocking=non_blocking),
            tables=torch.from_numpy(plan.tables).to(d, non_blocking=non_blocking),
            context_lens=torch.from_numpy(plan.context_lens).to(d, non_blocking=non_blocking),
            query_start=torch.from_numpy(plan.query_start).to(d, non_blocking=non_blocking),
            max_query_len=int(n.max()) if n.size else 0)

    def upload(self, plan: StepPlan, non_blocking: bool = False) -> DeviceStep:
        d = self.device
        return DeviceStep(
            slots=torch.from_numpy(plan.slots).to(d, non_blocking=non_blocking),
            pairs=torch.from_numpy(np.ascontiguousarray(plan.pairs)).to(d, non_blocking=non_blocking),
            tables=torch.from_numpy(plan.tables).to(d, non_blocking=non_blocking),
            context_lens=torch.from_numpy(plan.context_lens).to(d, non_blocking=non_blocking),
            max_context_len=int(plan.context_lens.max()) if plan.context_lens.size else 0)

    # -- device steps ------------------------------------------------------------
    def workspace(self, num_seqs: int, num_heads: int, max_context_len: int, partition_size: int = 0):
        need = paged_attention_workspace_size(num_seqs, num_heads, self.num_kv_heads, self.head_dim,
                                              max_context_len, partition_size)
        if self._ws is None or self._ws.numel() < need:
            if self._ws is not None:
                self._ws_retired.append(self._ws)   # calls in flight on other streams may hold it
            self._ws = make_workspace(self.device, need)
        return self._ws

    def copy_on_write(self, pairs: torch.Tensor) -> None:
        if pairs.numel():
            copy_blocks(self.key_cache, pairs)
            copy_blocks(self.value_cache, pairs)

    def write(self, key: torch.Tensor, value: torch.Tensor, slots: torch.Tensor) -> None:
        kv_reshape_and_cache(key, value, self.key_cache, self.value_cache, slots)

    def attend(self, query: torch.Tensor, step: DeviceStep, out: Optional[torch.Tensor] = None,
               scale: Optional[float] = None, partition_size: int = 0,
               max_context_len: Optional[int] = None) -> torch.Tensor:
        if out is None:
            out = torch.empty_like(query)
        mcl = step.max_context_len if max_context_len is None else max_context_len
        ws = self.workspace(query.shape[0], query.shape[1], mcl, partition_size)
        return paged_attention_decode(out, query, self.key_cache, self.value_cache, step.tables,
                                      step.context_lens, scale=scale, max_context_len=mcl,
                                      partition_size=partition_size, workspace=ws)

    def decode(self, query: torch.Tensor, key: torch.Tensor, value: torch.Tensor, step: DeviceStep,
               out: Optional[torch.Tensor] = None, scale: Optional[float] = None,
               partition_size: int = 0) -> torch.Tensor:
        """The device half of one decode iteration: copy-on-write copies, the
        new tokens' cache write, then attention (which reads the new tokens)."""
        self.copy_on_write(step.pairs)
        self.write(key, value, step.slots)
        return self.attend(query, step, out, scale, partition_size)

    def prefill_workspace(self) -> torch.Tensor:
        """The prompt-phase attention's work counter (256 bytes, prepared
        once); the cache's prefill calls share it, one at a time."""
        if getattr(self, "_pf_ws", None) is None:
            self._pf_ws = make_workspace(self.device, 256)
        return self._pf_ws

    def prefill(self, query: torch.Tensor, key: torch.Tensor, value: torch.Tensor, step: DevicePrefill,
                out: Optional[torch.Tensor] = None, scale: Optional[float] = None) -> torch.Tensor:
        """The device half of a prompt-phase step: copy-on-write copies (a
        shared prefix's partly filled last block), the new tokens' cache write,
        then causal attention of the new tokens over the paged cache."""
        if out is None:
            out = torch.empty_like(query)
        self.copy_on_write(step.pairs)
        self.write(key, value, step.slots)
        return paged_attention_prefill(out, query, self.key_cache, self.value_cache, step.tables,
                                       step.context_lens, step.query_start, scale=scale,
                                       max_query_len=step.max_query_len, workspace=self.prefill_workspace())

    # -- swapping ----------------------------------------------------------------
    def swap_out(self, seqs: Sequence[int], host: HostKVPool, stream=None):
        """Evict a sequence group to the host pool, all or nothing: its blocks
        move to host blocks (one swap_blocks launch for keys, one for values)
        and the GPU blocks are freed.  Returns the group's ids in the host
        pool and the (GPU block, host block) pairs."""
        ids, pairs = self.alloc.move_group(host.alloc, seqs)
        if len(pairs):
            p = torch.from_numpy(pairs).pin_memory()
            swap_blocks(host.key_cache, self.key_cache, p, stream)
            swap_blocks(host.value_cache, self.value_cache, p, stream)
            self._keep_pairs = p            # alive until the copies are done (next sync)
        return ids, pairs

    def swap_in(self, host_seqs: Sequence[int], host: HostKVPool, stream=None):
        """Bring a swapped-out group back: the reverse move and copies.
        Returns the group's GPU ids and the (host block, GPU block) pairs."""
        ids, pairs = host.alloc.move_group(self.alloc, host_seqs)
        if len(pairs):
            p = torch.from_numpy(pairs).pin_memory()
            swap_blocks(self.key_cache, host.key_cache, p, stream)
            swap_blocks(self.value_cache, host.value_cache, p, stream)
            self._keep_pairs = p
        return ids, pairs

    def prepare_prefill(self, query: torch.Tensor, key: torch.Tensor, value: torch.Tensor, step: DevicePrefill,
                        out: torch.Tensor, scale: Optional[float] = None,
                        stream: Optional[torch.cuda.Stream] = None) -> "PreparedPrefill":
        """The device calls of a prompt-phase step on fixed buffers, with their
        C-ABI arguments built once."""
        return PreparedPrefill(self, query, key, value, step, out, scale, stream)

    def prepare(self, query: torch.Tensor, key: torch.Tensor, value: torch.Tensor, step: DeviceStep,
                out: torch.Tensor, scale: Optional[float] = None, partition_size: int = 0,
                stream: Optional[torch.cuda.Stream] = None, fused: bool = True) -> "PreparedStep":
        """The device calls of a decode step on fixed buffers, with their C-ABI
        arguments built once.  fused: the cache write rides in the attention
        launch (paged_attention_decode_write) when the step has one new token
        per sequence."""
        return PreparedStep(self, query, key, value, step, out, scale, partition_size, stream, fused)


class PreparedStep:
    """copy_blocks, kv_reshape_and_cache and paged_attention_decode for one
    set of buffers, their arguments checked and marshalled once: issuing the
    step then costs three or four plain C calls.  For decode loops that run
    the same buffers every iteration (the buffers' contents may change)."""

    def __init__(self, eng: PagedKVCache, query, key, value, step: DeviceStep, out, scale, partition_size, stream,
                 fused=True):
        self._L = load()
        S, H, d = query.shape
        assert out.shape == query.shape and out.dtype == query.dtype == eng.key_cache.dtype
        assert key.shape == value.shape == (step.slots.shape[0], eng.num_kv_heads, d)
        for t in (query, key, value, out, step.slots, step.tables, step.context_lens, step.pairs):
            assert t.is_cuda and t.is_contiguous()
        code = 1 if query.dtype == torch.bfloat16 else 0
        st = ctypes.c_void_p((stream or torch.cuda.current_stream(eng.device)).cuda_stream)
        ws = eng.workspace(S, H, step.max_context_len, partition_size)
        self._keep = (query, key, value, step, out, ws)
        NB, B = eng.num_blocks, eng.block_size
        block_bytes = eng.num_kv_heads * B * d * eng.key_cache.element_size()
        n = step.pairs.shape[0] if step.pairs.dim() == 2 else 0
        self._copy = [(c.data_ptr(), step.pairs.data_ptr(), n, block_bytes, NB, st)
                      for c in (eng.key_cache, eng.value_cache)] if n else []
        T = step.slots.shape[0]
        self._write = (key.data_ptr(), value.data_ptr(), eng.key_cache.data_ptr(), eng.value_cache.data_ptr(),
                       step.slots.data_ptr(), T, eng.num_kv_heads, d, B, NB, code, st)
        self._attend = (out.data_ptr(), query.data_ptr(), eng.key_cache.data_ptr(), eng.value_cache.data_ptr(),
                        step.tables.data_ptr(), step.context_lens.data_ptr(), S, step.tables.shape[1],
                        step.max_context_len, B, NB, H, eng.num_kv_heads, d,
                        float(1.0 / math.sqrt(d) if scale is None else scale), partition_size, ws.data_ptr(),
                        ws.numel(), code, st)
        # one new token per sequence, in sequence order: the write can ride in the attention launch
        self._fused = fused and T == S
        self._write_attend = (out.data_ptr(), query.data_ptr(), key.data_ptr(), value.data_ptr(),
                              eng.key_cache.data_ptr(), eng.value_cache.data_ptr(), step.slots.data_ptr(),
                              step.tables.data_ptr(), step.context_lens.data_ptr(), S, step.tables.shape[1],
                              step.max_context_len, B, NB, H, eng.num_kv_heads, d,
                              float(1.0 / math.sqrt(d) if scale is None else scale), partition_size, ws.data_ptr(),
                              ws.numel(), code, st)

    def copy(self) -> None:
        for args in self._copy:
            rc = self._L.copy_blocks(*args)
            if rc:
                raise PkvError(rc, "copy_blocks")

    def write(self) -> None:
        if self._write[5]:
            rc = self._L.kv_reshape_and_cache(*self._write)
            if rc:
                raise PkvError(rc, "kv_reshape_and_cache")

    def attend(self) -> None:
        rc = self._L.paged_attention_decode(*self._attend)
        if rc:
            raise PkvError(rc, "paged_attention_decode")

    def write_attend(self) -> None:
        """The cache write and the attention in one launch (paged_attention_decode_write)."""
        rc = self._L.paged_attention_decode_write(*self._write_attend)
        if rc:
            raise PkvError(rc, "paged_attention_decode_write")

    def front(self) -> None:
        """What runs before the attention launch: the copies (and the write when not fused)."""
        self.copy()
        if not self._fused:
            self.write()

    def back(self) -> None:
        """The attention launch (with the write when fused)."""
        if self._fused:
            self.write_attend()
        else:
            self.attend()

    def __call__(self) -> None:
        self.front()
        self.back()


class PreparedPrefill:
    """copy_blocks, kv_reshape_and_cache and paged_attention_prefill for one
    set of buffers, their arguments checked and marshalled once."""

    def __init__(self, eng: PagedKVCache, query, key, value, step: DevicePrefill, out, scale, stream):
        self._L = load()
        T, H, d = query.shape
        assert out.shape == query.shape and out.dtype == query.dtype == eng.key_cache.dtype
        assert key.shape == value.shape == (step.slots.shape[0], eng.num_kv_heads, d)
        for t in (query, key, value, out, step.slots, step.tables, step.context_lens, step.query_start, step.pairs):
            assert t.is_cuda and t.is_contiguous()
        code = 1 if query.dtype == torch.bfloat16 else 0
        st = ctypes.c_void_p((stream or torch.cuda.current_stream(eng.device)).cuda_stream)
        ws = eng.prefill_workspace()
        self._keep = (query, key, value, step, out, ws)
        NB, B = eng.num_blocks, eng.block_size
        block_bytes = eng.num_kv_heads * B * d * eng.key_cache.element_size()
        n = step.pairs.shape[0] if step.pairs.dim() == 2 else 0
        self._copy = [(c.data_ptr(), step.pairs.data_ptr(), n, block_bytes, NB, st)
                      for c in (eng.key_cache, eng.value_cache)] if n else []
        Tw = step.slots.shape[0]
        self._write = (key.data_ptr(), value.data_ptr(), eng.key_cache.data_ptr(), eng.value_cache.data_ptr(),
                       step.slots.data_ptr(), Tw, eng.num_kv_heads, d, B, NB, code, st)
        S = step.context_lens.shape[0]
        self._attend = (out.data_ptr(), query.data_ptr(), eng.key_cache.data_ptr(), eng.value_cache.data_ptr(),
                        step.tables.data_ptr(), step.context_lens.data_ptr(), step.query_start.data_ptr(), S, T,
                        step.max_query_len, step.tables.shape[1], B, NB, H, eng.num_kv_heads, d,
                        float(1.0 / math.sqrt(d) if scale is None else scale), ws.data_ptr(), ws.numel(), code,
                        st)

    def copy(self) -> None:
        for args in self._copy:
            rc = self._L.copy_blocks(*args)
            if rc:
                raise PkvError(rc, "copy_blocks")

    def write(self) -> None:
        if self._write[5]:
            rc = self._L.kv_reshape_and_cache(*self._write)
            if rc:
                raise PkvError(rc, "kv_reshape_and_cache")

    def attend(self) -> None:
        rc = self._L.paged_attention_prefill(*self._attend)
        if rc:
            raise PkvError(rc, "paged_attention_prefill")

    def __call__(self) -> None:
        self.copy()
        self.write()
        self.attend()
