"""paged_kv_cache_139_gb300 -- the decode hot path of PagedAttention on GB300.

A thin Python binding of libpkv.so (declared in include/pkv.h).  Every
function here only checks and marshals its arguments -- torch tensors to
device pointers, the current CUDA stream -- and calls the C entry point of
the same name; all the work runs in the library's sm_103a kernels.  PyTorch
provides device memory and streams.  There is no fallback: if the library is
missing, the first call raises.

    kv_reshape_and_cache     slot-mapped K/V write into the paged cache
    paged_attention_decode   block-table gather + decode attention
    copy_blocks              copy-on-write block copy
    BlockAllocator           the native ref-counted block allocator
"""
from __future__ import annotations

import ctypes
import math
from typing import Optional, Sequence

import numpy as np
import torch

from ._lib import STATUS, load

__all__ = ["PkvError", "PkvOOM", "kv_reshape_and_cache", "paged_attention_decode",
           "paged_attention_decode_noalloc", "paged_attention_decode_write", "paged_attention_prefill", "paged_attention_workspace_size",
           "make_workspace",
           "paged_attention_partition_size", "copy_blocks",
           "validate_copy_pairs", "swap_blocks", "check", "launch_count", "version", "BlockAllocator", "library_path"]

PKV_F16, PKV_BF16 = 0, 1


class PkvError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        self.status_name = STATUS.get(status, str(status))
        super().__init__(f"{what}: {self.status_name}: {load().pkv_last_error_string().decode()}")


class PkvOOM(PkvError):
    """The allocator has too few free blocks; its state is unchanged."""


def _ck(rc: int, what: str) -> None:
    if rc != 0:
        raise (PkvOOM if rc == 2 else PkvError)(rc, what)


def library_path() -> str:
    from ._lib import LIB_PATH
    return str(LIB_PATH)


def version() -> int:
    return load().pkv_version()


def launch_count() -> int:
    """Kernels launched by the library in this process."""
    return int(load().pkv_launch_count())


# -- marshalling -----------------------------------------------------------------

def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float16:
        return PKV_F16
    if t.dtype == torch.bfloat16:
        return PKV_BF16
    raise TypeError(f"expected float16 or bfloat16, got {t.dtype}")


def _dev(t: torch.Tensor, name: str, dtype=None, ndim=None) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dimensions, got shape {tuple(t.shape)}")
    return t.data_ptr()


def _stream(stream: Optional[torch.cuda.Stream], device) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return ctypes.c_void_p(s.cuda_stream)


# -- the three device calls -------------------------------------------------------

def kv_reshape_and_cache(key: torch.Tensor, value: torch.Tensor, key_cache: torch.Tensor,
                         value_cache: torch.Tensor, slot_mapping: torch.Tensor,
                         stream: Optional[torch.cuda.Stream] = None) -> None:
    """key/value [T][Hkv][d]; caches [NB][Hkv][B][d]; slot_mapping int64 [T]."""
    NB, Hkv, B, d = key_cache.shape
    T = key.shape[0]
    if tuple(key.shape) != (T, Hkv, d) or key.shape != value.shape or value_cache.shape != key_cache.shape:
        raise ValueError("kv_reshape_and_cache: shape mismatch")
    if key.dtype != key_cache.dtype or value.dtype != key_cache.dtype or value_cache.dtype != key_cache.dtype:
        raise TypeError("kv_reshape_and_cache: dtype mismatch")
    if slot_mapping.shape != (T,):
        raise ValueError("kv_reshape_and_cache: slot_mapping must be [num_tokens]")
    args = (_dev(key, "key"), _dev(value, "value"), _dev(key_cache, "key_cache"),
            _dev(value_cache, "value_cache"), _dev(slot_mapping, "slot_mapping", torch.int64))
    rc = load().kv_reshape_and_cache(*args, T, Hkv, d, B, NB, _dtype_code(key_cache),
                                     _stream(stream, key_cache.device))
    _ck(rc, "kv_reshape_and_cache")


def paged_attention_workspace_size(num_seqs: int, num_heads: int, num_kv_heads: int, head_dim: int,
                                   max_context_len: int, partition_size: int = 0) -> int:
    return int(load().paged_attention_workspace_size(num_seqs, num_heads, num_kv_heads, head_dim,
                                                     max_context_len, partition_size))


def paged_attention_partition_size(num_seqs: int, num_heads: int, num_kv_heads: int, head_dim: int,
                                   max_context_len: int, partition_size: int = 0) -> int:
    return int(load().paged_attention_partition_size(num_seqs, num_heads, num_kv_heads, head_dim,
                                                     max_context_len, partition_size))


def make_workspace(device, nbytes: int, stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """A device buffer of at least nbytes, prepared for paged_attention_decode
    and paged_attention_prefill (paged_attention_workspace_init).  Returns
    once the preparation has finished, so any stream may use the buffer."""
    dev = torch.device(device)
    buf = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev)
    st = _stream(stream, dev)
    _ck(load().paged_attention_workspace_init(buf.data_ptr(), buf.numel(), st), "paged_attention_workspace_init")
    (stream or torch.cuda.current_stream(dev)).synchronize()
    return buf


_ws_cache: dict = {}
_ws_retired: list = []


def _workspace(device, nbytes: int) -> torch.Tensor:
    """The binding's own workspace: at least nbytes, kept per device.  A
    buffer replaced by a larger one is kept alive, since calls on other
    streams may still be using it (the sizes only grow, so few are kept)."""
    key = torch.device(device)
    buf = _ws_cache.get(key)
    if buf is None or buf.numel() < nbytes:
        if buf is not None:
            _ws_retired.append(buf)
        buf = make_workspace(key, nbytes)
        _ws_cache[key] = buf
    return buf


def paged_attention_decode(out: torch.Tensor, query: torch.Tensor, key_cache: torch.Tensor,
                           value_cache: torch.Tensor, block_tables: torch.Tensor,
                           context_lens: torch.Tensor, scale: Optional[float] = None,
                           max_context_len: int = 0, partition_size: int = 0,
                           workspace: Optional[torch.Tensor] = None,
                           stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """out/query [S][H][d]; caches [NB][Hkv][B][d]; block_tables int32 [S][MB];
    context_lens int32 [S].  scale defaults to 1/sqrt(d).  A workspace passed
    in must come from make_workspace (or paged_attention_workspace_init) and
    serve one call at a time; None takes the binding's own per-device buffer,
    which every decode and prefill call without a workspace shares, so calls
    through it must not overlap on the GPU (give calls on concurrent streams
    a workspace each).  Returns out."""
    S, H, d = query.shape
    NB, Hkv, B, d2 = key_cache.shape
    if d2 != d or out.shape != query.shape or value_cache.shape != key_cache.shape:
        raise ValueError("paged_attention_decode: shape mismatch")
    if block_tables.dim() != 2 or block_tables.shape[0] != S or context_lens.shape != (S,):
        raise ValueError("paged_attention_decode: block_tables must be [S][max_blocks], context_lens [S]")
    if not (query.dtype == out.dtype == key_cache.dtype == value_cache.dtype):
        raise TypeError("paged_attention_decode: dtype mismatch")
    mb = block_tables.shape[1]
    mcl = max_context_len if max_context_len > 0 else mb * B
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if workspace is None:
        workspace = _workspace(query.device, paged_attention_workspace_size(S, H, Hkv, d, mcl, partition_size))
    ws_ptr = _dev(workspace, "workspace")
    ws_bytes = workspace.numel() * workspace.element_size()
    rc = load().paged_attention_decode(
        _dev(out, "out"), _dev(query, "query"), _dev(key_cache, "key_cache"), _dev(value_cache, "value_cache"),
        _dev(block_tables, "block_tables", torch.int32), _dev(context_lens, "context_lens", torch.int32),
        S, mb, max_context_len, B, NB, H, Hkv, d, float(scale), partition_size, ws_ptr, ws_bytes,
        _dtype_code(query), _stream(stream, query.device))
    _ck(rc, "paged_attention_decode")
    return out


def paged_attention_decode_write(out: torch.Tensor, query: torch.Tensor, key: torch.Tensor, value: torch.Tensor,
                                 key_cache: torch.Tensor, value_cache: torch.Tensor, slot_mapping: torch.Tensor,
                                 block_tables: torch.Tensor, context_lens: torch.Tensor,
                                 scale: Optional[float] = None, max_context_len: int = 0, partition_size: int = 0,
                                 workspace: Optional[torch.Tensor] = None,
                                 stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """kv_reshape_and_cache of each sequence's new token (key/value [S][Hkv][d],
    slot_mapping int64 [S], the slot of position context_lens[s] - 1) and
    paged_attention_decode in one launch.  workspace as for
    paged_attention_decode: None shares the binding's per-device buffer, so
    calls through it must not overlap on the GPU.  Returns out."""
    S, H, d = query.shape
    NB, Hkv, B, d2 = key_cache.shape
    if d2 != d or out.shape != query.shape or value_cache.shape != key_cache.shape:
        raise ValueError("paged_attention_decode_write: shape mismatch")
    if key.shape != (S, Hkv, d) or value.shape != key.shape or slot_mapping.shape != (S,):
        raise ValueError("paged_attention_decode_write: key/value must be [S][Hkv][d], slot_mapping [S]")
    if block_tables.dim() != 2 or block_tables.shape[0] != S or context_lens.shape != (S,):
        raise ValueError("paged_attention_decode_write: block_tables must be [S][max_blocks], context_lens [S]")
    mb = block_tables.shape[1]
    mcl = max_context_len if max_context_len > 0 else mb * B
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if workspace is None:
        workspace = _workspace(query.device, paged_attention_workspace_size(S, H, Hkv, d, mcl, partition_size))
    rc = load().paged_attention_decode_write(
        _dev(out, "out"), _dev(query, "query"), _dev(key, "key"), _dev(value, "value"),
        _dev(key_cache, "key_cache"), _dev(value_cache, "value_cache"),
        _dev(slot_mapping, "slot_mapping", torch.int64), _dev(block_tables, "block_tables", torch.int32),
        _dev(context_lens, "context_lens", torch.int32), S, mb, max_context_len, B, NB, H, Hkv, d, float(scale),
        partition_size, _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _dtype_code(query), _stream(stream, query.device))
    _ck(rc, "paged_attention_decode_write")
    return out


def paged_attention_prefill(out: torch.Tensor, query: torch.Tensor, key_cache: torch.Tensor,
                            value_cache: torch.Tensor, block_tables: torch.Tensor,
                            context_lens: torch.Tensor, query_start: torch.Tensor,
                            scale: Optional[float] = None, max_query_len: int = 0,
                            workspace: Optional[torch.Tensor] = None,
                            stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Prompt-phase attention: out/query [T][H][d] hold the new tokens of all
    sequences back to back, query_start int32 [S+1] their offsets; the new
    tokens of sequence s are the last n_s of its context_lens[s] and each
    attends every token up to its own position.  Their keys and values must
    already be in the cache.  workspace: a buffer from make_workspace (its
    counter balances the work over the SMs), serving one call at a time; None
    takes the binding's own per-device buffer, which paged_attention_decode
    calls share (calls through it must not overlap on the GPU).  Returns out."""
    T, H, d = query.shape
    NB, Hkv, B, d2 = key_cache.shape
    S = context_lens.shape[0]
    if d2 != d or out.shape != query.shape or value_cache.shape != key_cache.shape:
        raise ValueError("paged_attention_prefill: shape mismatch")
    if block_tables.dim() != 2 or block_tables.shape[0] != S or query_start.shape != (S + 1,):
        raise ValueError("paged_attention_prefill: block_tables must be [S][max_blocks], query_start [S+1]")
    if not (query.dtype == out.dtype == key_cache.dtype == value_cache.dtype):
        raise TypeError("paged_attention_prefill: dtype mismatch")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    ws = _workspace(query.device, 256) if workspace is None else workspace
    rc = load().paged_attention_prefill(
        _dev(out, "out"), _dev(query, "query"), _dev(key_cache, "key_cache"), _dev(value_cache, "value_cache"),
        _dev(block_tables, "block_tables", torch.int32), _dev(context_lens, "context_lens", torch.int32),
        _dev(query_start, "query_start", torch.int32), S, T, max_query_len, block_tables.shape[1], B, NB, H, Hkv,
        d, float(scale), _dev(ws, "workspace", torch.uint8), ws.numel(), _dtype_code(query),
        _stream(stream, query.device))
    _ck(rc, "paged_attention_prefill")
    return out


def paged_attention_decode_noalloc(out: torch.Tensor, query: torch.Tensor, key_cache: torch.Tensor,
                                   value_cache: torch.Tensor, block_tables: torch.Tensor,
                                   context_lens: torch.Tensor, scale: Optional[float] = None,
                                   max_context_len: int = 0, partition_size: int = 0,
                                   stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """paged_attention_decode without a workspace: for callers that may not
    allocate device memory when they run attention.  The partition partials
    use the library's built-in 16 MiB device array, shared by every call on a
    device (one call at a time); larger sizes raise PkvError (PKV_EINVAL).
    The first call on a device, and the first after check() reported a
    device-wait timeout, prepares the array and waits for it, so it must not
    run during stream capture (PkvError, PKV_EINVAL)."""
    S, H, d = query.shape
    NB, Hkv, B, d2 = key_cache.shape
    if d2 != d or out.shape != query.shape or value_cache.shape != key_cache.shape:
        raise ValueError("paged_attention_decode_noalloc: shape mismatch")
    if block_tables.dim() != 2 or block_tables.shape[0] != S or context_lens.shape != (S,):
        raise ValueError("paged_attention_decode_noalloc: block_tables must be [S][max_blocks], context_lens [S]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    rc = load().paged_attention_decode_noalloc(
        _dev(out, "out"), _dev(query, "query"), _dev(key_cache, "key_cache"), _dev(value_cache, "value_cache"),
        _dev(block_tables, "block_tables", torch.int32), _dev(context_lens, "context_lens", torch.int32),
        S, block_tables.shape[1], max_context_len, B, NB, H, Hkv, d, float(scale), partition_size,
        _dtype_code(query), _stream(stream, query.device))
    _ck(rc, "paged_attention_decode_noalloc")
    return out


def copy_blocks(cache: torch.Tensor, src_dst_pairs: torch.Tensor,
                stream: Optional[torch.cuda.Stream] = None) -> None:
    """cache [NB][...] (one block per leading index); src_dst_pairs int32 [n][2] on the device."""
    n = src_dst_pairs.shape[0] if src_dst_pairs.dim() == 2 else 0
    if src_dst_pairs.numel() and (src_dst_pairs.dim() != 2 or src_dst_pairs.shape[1] != 2):
        raise ValueError("copy_blocks: src_dst_pairs must be [n][2]")
    NB = cache.shape[0]
    block_bytes = (cache.numel() // NB if NB else 0) * cache.element_size()
    pairs_ptr = _dev(src_dst_pairs, "src_dst_pairs", torch.int32) if n else None
    rc = load().copy_blocks(_dev(cache, "cache"), pairs_ptr, n, block_bytes, NB, _stream(stream, cache.device))
    _ck(rc, "copy_blocks")


def validate_copy_pairs(pairs, num_blocks: int) -> None:
    """Host-side check: ids in range, distinct destinations, no destination
    that is also a source.  Raises PkvError (PKV_EINVAL) otherwise."""
    a = np.ascontiguousarray(np.asarray(pairs, dtype=np.int32).reshape(-1, 2))
    rc = load().pkv_validate_copy_pairs(a.ctypes.data_as(ctypes.c_void_p) if a.size else None,
                                        a.shape[0], num_blocks)
    _ck(rc, "validate_copy_pairs")


def swap_blocks(dst_pool: torch.Tensor, src_pool: torch.Tensor, pairs: torch.Tensor,
                stream: Optional[torch.cuda.Stream] = None) -> None:
    """Block pairs[p][1] of dst_pool takes block pairs[p][0] of src_pool (one
    launch for all pairs).  Pools [NB][...] of one layout: CUDA tensors or
    pinned host tensors; pairs int32 [n][2] on the GPU or pinned."""
    def addr(t, name):
        if not isinstance(t, torch.Tensor) or not (t.is_cuda or t.is_pinned()):
            raise TypeError(f"{name} must be a CUDA tensor or pinned host memory")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        return t.data_ptr()
    if dst_pool.shape[1:] != src_pool.shape[1:] or dst_pool.dtype != src_pool.dtype:
        raise ValueError("swap_blocks: pools of different layouts")
    n = pairs.shape[0] if pairs.dim() == 2 else 0
    if n == 0:
        return
    if pairs.dtype != torch.int32 or pairs.shape[1] != 2:
        raise TypeError("swap_blocks: pairs must be int32 [n][2]")
    block_bytes = dst_pool[0].numel() * dst_pool.element_size()
    dev = dst_pool.device if dst_pool.is_cuda else src_pool.device
    rc = load().swap_blocks(addr(dst_pool, "dst_pool"), addr(src_pool, "src_pool"), addr(pairs, "pairs"), n,
                            block_bytes, src_pool.shape[0], dst_pool.shape[0], _stream(stream, dev))
    _ck(rc, "swap_blocks")


def check(stream: Optional[torch.cuda.Stream] = None, device=None) -> None:
    """Synchronise the stream and raise if the device latched an index error
    or a wait timeout since the last check."""
    s = stream if stream is not None else torch.cuda.current_stream(device)
    _ck(load().pkv_check(ctypes.c_void_p(s.cuda_stream)), "pkv_check")


# -- host block allocator ---------------------------------------------------------

class BlockAllocator:
    """The native ref-counted block allocator (fork / append / free)."""

    def __init__(self, num_blocks: int, block_size: int, free_order: Optional[Sequence[int]] = None):
        self._L = load()
        h = ctypes.c_void_p()
        if free_order is not None:
            fo = np.ascontiguousarray(np.asarray(free_order, dtype=np.int32))
            if fo.shape != (num_blocks,):
                raise ValueError("free_order must list every block once")
            fp = fo.ctypes.data_as(ctypes.c_void_p)
        else:
            fp = None
        _ck(self._L.pkv_alloc_create(num_blocks, block_size, fp, ctypes.byref(h)), "pkv_alloc_create")
        self._h = h
        self.num_blocks = num_blocks
        self.block_size = block_size

    def close(self) -> None:
        if getattr(self, "_h", None):
            self._L.pkv_alloc_destroy(self._h)
            self._h = None

    def __del__(self):
        self.close()

    def seq_new(self, length: int) -> int:
        sid = ctypes.c_int32()
        _ck(self._L.pkv_seq_new(self._h, length, ctypes.byref(sid)), "pkv_seq_new")
        return sid.value

    def fork(self, seq: int) -> int:
        child = ctypes.c_int32()
        _ck(self._L.pkv_seq_fork(self._h, seq, ctypes.byref(child)), "pkv_seq_fork")
        return child.value

    def append(self, seq: int):
        """Returns (slot, cow) with cow = (src, dst) or None."""
        slot, src, dst = ctypes.c_int64(), ctypes.c_int32(), ctypes.c_int32()
        _ck(self._L.pkv_seq_append(self._h, seq, ctypes.byref(slot), ctypes.byref(src), ctypes.byref(dst)),
            "pkv_seq_append")
        return slot.value, (None if src.value < 0 else (src.value, dst.value))

    def append_batch(self, seqs: Sequence[int]):
        """One token per sequence, all or nothing.  Returns (slots int64[n], pairs int32[m][2])."""
        s = np.ascontiguousarray(np.asarray(seqs, dtype=np.int32))
        n = s.shape[0]
        slots = np.empty(n, np.int64)
        pairs = np.empty((max(n, 1), 2), np.int32)
        npairs = ctypes.c_int()
        _ck(self._L.pkv_seq_append_batch(self._h, s.ctypes.data_as(ctypes.c_void_p), n,
                                         slots.ctypes.data_as(ctypes.c_void_p),
                                         pairs.ctypes.data_as(ctypes.c_void_p), ctypes.byref(npairs)),
            "pkv_seq_append_batch")
        return slots, pairs[:npairs.value].copy()

    def free(self, seq: int) -> None:
        _ck(self._L.pkv_seq_free(self._h, seq), "pkv_seq_free")

    def seq_len(self, seq: int) -> int:
        n = ctypes.c_int64()
        _ck(self._L.pkv_seq_len(self._h, seq, ctypes.byref(n)), "pkv_seq_len")
        return n.value

    def block_table(self, seq: int) -> list:
        n = ctypes.c_int()
        self._L.pkv_seq_block_table(self._h, seq, None, 0, ctypes.byref(n))
        out = np.empty(max(n.value, 1), np.int32)
        _ck(self._L.pkv_seq_block_table(self._h, seq, out.ctypes.data_as(ctypes.c_void_p), out.shape[0],
                                        ctypes.byref(n)), "pkv_seq_block_table")
        return out[:n.value].tolist()

    def beam_step(self, beams: Sequence[int], parents: Sequence[int]):
        """One beam-search step: new candidate i continues beams[parents[i]]
        (the first child continues the sequence, later ones fork it; all
        append a token; unchosen beams are freed).  Returns (new beam ids,
        slots int64 [kn], copy-on-write pairs int32 [m][2]); PkvOOM leaves
        everything unchanged."""
        b = np.ascontiguousarray(np.asarray(beams, dtype=np.int32))
        p = np.ascontiguousarray(np.asarray(parents, dtype=np.int32))
        kn = p.shape[0]
        new = np.empty(max(kn, 1), np.int32)
        slots = np.empty(max(kn, 1), np.int64)
        pairs = np.empty((max(kn, 1), 2), np.int32)
        npairs = ctypes.c_int()
        _ck(self._L.pkv_beam_step(self._h, b.ctypes.data_as(ctypes.c_void_p) if b.size else None, b.shape[0],
                                  p.ctypes.data_as(ctypes.c_void_p) if kn else None, kn,
                                  new.ctypes.data_as(ctypes.c_void_p), slots.ctypes.data_as(ctypes.c_void_p),
                                  pairs.ctypes.data_as(ctypes.c_void_p), ctypes.byref(npairs)), "pkv_beam_step")
        return new[:kn].tolist(), slots[:kn].copy(), pairs[:npairs.value].copy()

    def blocks_in_use(self) -> int:
        return self._L.pkv_blocks_in_use(self._h)

    def move_group(self, dst: "BlockAllocator", seqs: Sequence[int]):
        """Move the sequence group `seqs` (holding every reference to its
        blocks) to allocator `dst`, all or nothing: returns (new ids in dst,
        pairs int32 [m][2] of (block here, block in dst)) for swap_blocks.
        PkvOOM if dst has too few free blocks."""
        s = np.ascontiguousarray(np.asarray(seqs, dtype=np.int32))
        n = s.shape[0]
        ids = np.empty(max(n, 1), np.int32)
        cap = max(1, sum(len(self.block_table(int(x))) for x in s))
        pairs = np.empty((cap, 2), np.int32)
        npairs = ctypes.c_int()
        _ck(self._L.pkv_move_group(self._h, dst._h, s.ctypes.data_as(ctypes.c_void_p) if n else None, n,
                                   ids.ctypes.data_as(ctypes.c_void_p), pairs.ctypes.data_as(ctypes.c_void_p), cap,
                                   ctypes.byref(npairs)), "pkv_move_group")
        return ids[:n].tolist(), pairs[:npairs.value].copy()

    def build_block_tables(self, seqs: Sequence[int], max_blocks: int):
        """(tables int32 [n][max_blocks] padded with -1, context_lens int32 [n])."""
        s = np.ascontiguousarray(np.asarray(seqs, dtype=np.int32))
        n = s.shape[0]
        tables = np.empty((n, max_blocks), np.int32)
        ctx = np.empty(n, np.int32)
        _ck(self._L.pkv_build_block_tables(self._h, s.ctypes.data_as(ctypes.c_void_p), n,
                                           tables.ctypes.data_as(ctypes.c_void_p), max_blocks,
                                           ctx.ctypes.data_as(ctypes.c_void_p)), "pkv_build_block_tables")
        return tables, ctx

    def block_ref(self, block: int) -> int:
        return self._L.pkv_block_ref(self._h, block)

    def num_free(self) -> int:
        return self._L.pkv_num_free(self._h)

    def free_list(self) -> list:
        n = ctypes.c_int()
        out = np.empty(max(self.num_blocks, 1), np.int32)
        _ck(self._L.pkv_free_list(self._h, out.ctypes.data_as(ctypes.c_void_p), out.shape[0], ctypes.byref(n)),
            "pkv_free_list")
        return out[:n.value].tolist()
