"""Oracle for the paged decode path -- TEST INFRASTRUCTURE ONLY.

Plain, slow, fp64 CPU code that states what the path computes.  Only the
tests, the smoke check and the benchmark's CPU-baseline leg use it; the
library (paged_kv_cache_139_gb300) never imports it, and it imports nothing
from the library.

Contents:
  pkv_oracle.c   fp64 attention over the paged cache (decode: one query
                 token per sequence; prompt phase: many, causal), the
                 slot-mapped cache write, the block copy, per-partition statistics and their
                 log-sum-exp merge (built by build.py with gcc).
  allocator.py   the reference ref-counted block allocator (with the move of
                 a sequence group to a second pool, for swapping).

Parity status: every function here is pinned by tests/test_oracle_pins.py
and tests/test_oracle_allocator.py (worked examples from the pages, closed
forms, invariants and library routines).  No function is unpinned.
"""
from __future__ import annotations

import ctypes
import math

import numpy as np
import torch

from .allocator import AllocatorOOM, RefAllocator, blocks_needed
from .build import LIB, build

__all__ = ["AllocatorOOM", "RefAllocator", "blocks_needed", "kv_bytes_per_token",
           "cache_write", "copy_blocks", "copy_blocks_between", "paged_attention", "partition_stats",
           "merge_partitions", "paged_prefill", "locate_tokens", "decode16", "bits16", "lib"]

_lib = None

_p = ctypes.c_void_p
_i = ctypes.c_int
_i64 = ctypes.c_int64
_d = ctypes.c_double


def load(path) -> ctypes.CDLL:
    """Open a build of pkv_oracle.c and declare its functions."""
    L = ctypes.CDLL(str(path))
    L.oracle_decode16.argtypes = [_p, _i64, _i, _p]
    L.oracle_decode16.restype = None
    L.oracle_locate_tokens.argtypes = [_p, _i, _i64, _p, _p]
    L.oracle_cache_write.argtypes = [_p, _p, _p, _p, _p, _i, _i, _i, _i, _i]
    L.oracle_copy_blocks.argtypes = [_p, _p, _i, _i64, _i]
    L.oracle_copy_blocks_between.argtypes = [_p, _p, _p, _i, _i64, _i, _i]
    L.oracle_paged_attention.argtypes = [_p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i,
                                         _d, _i, _i, _p, _i]
    L.oracle_paged_prefill.argtypes = [_p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i,
                                       _d, _i, _i, _p, _i]
    L.oracle_partition_stats.argtypes = [_p, _p, _p, _p, _p, _i, _i, _i, _i, _i, _i, _d,
                                         _i, _i, _i, _i, _i, _p, _p, _p]
    L.oracle_merge_partitions.argtypes = [_p, _p, _p, _i, _i, _p]
    L.oracle_merge_partitions.restype = None
    return L


def lib():
    global _lib
    if _lib is None:
        _lib = load(build())
    return _lib


def kv_bytes_per_token(hidden: int, layers: int, bytes_per_number: int) -> int:
    """One key and one value, each as wide as the model, for every layer
    ("PagedAttention and vLLM, annotated" §1; "vLLM & PagedAttention" §I)."""
    return 2 * hidden * layers * bytes_per_number


# -- array plumbing -----------------------------------------------------------

def bits16(x) -> np.ndarray:
    """The raw 16-bit patterns of an fp16/bf16 tensor (or a uint16 array), as a
    C-contiguous numpy uint16 array that shares nothing with the input."""
    if isinstance(x, torch.Tensor):
        assert x.dtype in (torch.float16, torch.bfloat16), x.dtype
        return x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16).copy()
    a = np.ascontiguousarray(x)
    assert a.dtype == np.uint16
    return a.copy()


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _is_bf16(dtype) -> int:
    if dtype in ("bf16", torch.bfloat16):
        return 1
    if dtype in ("f16", torch.float16):
        return 0
    raise ValueError(dtype)


def _check(rc: int, what: str):
    if rc < 0:
        raise ValueError(f"oracle {what}: error {rc} ({'bad size' if rc == -1 else 'index out of range'})")
    return rc


# -- the path -----------------------------------------------------------------

def decode16(bits: np.ndarray, dtype) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(b.shape, dtype=np.float64)
    lib().oracle_decode16(_ptr(b), b.size, _is_bf16(dtype), _ptr(out))
    return out


def locate_tokens(table_row, block_size: int, ctx: int):
    """(physical block, offset) of each of the first ctx tokens."""
    row = np.ascontiguousarray(table_row, dtype=np.int32)
    phys = np.empty(ctx, np.int32)
    off = np.empty(ctx, np.int32)
    _check(lib().oracle_locate_tokens(_ptr(row), block_size, ctx, _ptr(phys), _ptr(off)),
           "locate_tokens")
    return phys, off


def cache_write(key, value, key_cache: np.ndarray, value_cache: np.ndarray, slots) -> None:
    """In place on the uint16 cache arrays [NB][Hkv][B][d]."""
    k, v = bits16(key), bits16(value)
    s = np.ascontiguousarray(slots, dtype=np.int64)
    NB, Hkv, B, d = key_cache.shape
    T = s.shape[0]
    assert k.shape == (T, Hkv, d) and v.shape == (T, Hkv, d)
    assert key_cache.flags.c_contiguous and value_cache.flags.c_contiguous
    _check(lib().oracle_cache_write(_ptr(k), _ptr(v), _ptr(key_cache), _ptr(value_cache),
                                    _ptr(s), T, Hkv, d, B, NB), "cache_write")


def copy_blocks(cache: np.ndarray, pairs) -> None:
    """In place on a uint16 cache array [NB][...]."""
    pr = np.ascontiguousarray(np.asarray(pairs, dtype=np.int32).reshape(-1, 2))
    NB = cache.shape[0]
    assert cache.flags.c_contiguous
    _check(lib().oracle_copy_blocks(_ptr(cache), _ptr(pr), pr.shape[0],
                                    int(np.prod(cache.shape[1:])), NB), "copy_blocks")


def copy_blocks_between(dst_pool: np.ndarray, src_pool: np.ndarray, pairs) -> None:
    """In place on the uint16 array dst_pool [NBd][...]: block pairs[i][1] of
    dst_pool takes block pairs[i][0] of src_pool."""
    pr = np.ascontiguousarray(np.asarray(pairs, dtype=np.int32).reshape(-1, 2))
    assert dst_pool.flags.c_contiguous and src_pool.flags.c_contiguous
    assert dst_pool.shape[1:] == src_pool.shape[1:]
    _check(lib().oracle_copy_blocks_between(_ptr(dst_pool), _ptr(np.ascontiguousarray(src_pool)), _ptr(pr),
                                            pr.shape[0], int(np.prod(dst_pool.shape[1:])), src_pool.shape[0],
                                            dst_pool.shape[0]), "copy_blocks_between")


def default_scale(head_dim: int) -> float:
    """1/sqrt(d), the scaling of the attention equations ("vLLM & PagedAttention" §I, §III)."""
    return 1.0 / math.sqrt(head_dim)


def paged_attention(query, key_cache, value_cache, block_tables, context_lens, dtype,
                    scale=None, which=None) -> np.ndarray:
    """fp64 out[S][H][d].  `which`: optional list of (s, h) to compute (others stay NaN)."""
    q = bits16(query)
    kc = key_cache if isinstance(key_cache, np.ndarray) else bits16(key_cache)
    vc = value_cache if isinstance(value_cache, np.ndarray) else bits16(value_cache)
    kc = np.ascontiguousarray(kc)
    vc = np.ascontiguousarray(vc)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    S, H, d = q.shape
    NB, Hkv, B, d2 = kc.shape
    assert d2 == d and vc.shape == kc.shape and bt.shape[0] == S and cl.shape == (S,)
    if scale is None:
        scale = default_scale(d)
    out = np.full((S, H, d), np.nan, dtype=np.float64)
    if which is None:
        w, nw = None, 0
    else:
        wa = np.ascontiguousarray(np.asarray(which, dtype=np.int32).reshape(-1, 2))
        w, nw = _ptr(wa), wa.shape[0]
    _check(lib().oracle_paged_attention(_ptr(out), _ptr(q), _ptr(kc), _ptr(vc), _ptr(bt), _ptr(cl),
                                        S, bt.shape[1], B, H, Hkv, d, float(scale), _is_bf16(dtype),
                                        NB, w, nw), "paged_attention")
    return out


def paged_prefill(query, key_cache, value_cache, block_tables, context_lens, query_start, dtype,
                  scale=None, which=None) -> np.ndarray:
    """fp64 out[T][H][d] of the prompt phase: new token j of sequence s (the
    last n_s = query_start[s+1] - query_start[s] tokens of its context)
    attends every token up to its own position.  `which`: optional list of
    (token, h) to compute (other rows stay NaN)."""
    q = bits16(query)
    kc = np.ascontiguousarray(key_cache if isinstance(key_cache, np.ndarray) else bits16(key_cache))
    vc = np.ascontiguousarray(value_cache if isinstance(value_cache, np.ndarray) else bits16(value_cache))
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    qs = np.ascontiguousarray(query_start, dtype=np.int32)
    T, H, d = q.shape
    NB, Hkv, B, d2 = kc.shape
    S = cl.shape[0]
    assert d2 == d and vc.shape == kc.shape and bt.shape[0] == S and qs.shape == (S + 1,)
    assert int(qs[-1]) == T
    if scale is None:
        scale = default_scale(d)
    out = np.full((T, H, d), np.nan, dtype=np.float64)
    if which is None:
        w, nw = None, 0
    else:
        wa = np.ascontiguousarray(np.asarray(which, dtype=np.int32).reshape(-1, 2))
        w, nw = _ptr(wa), wa.shape[0]
    _check(lib().oracle_paged_prefill(_ptr(out), _ptr(q), _ptr(kc), _ptr(vc), _ptr(bt), _ptr(cl), _ptr(qs),
                                      S, bt.shape[1], B, H, Hkv, d, float(scale), _is_bf16(dtype), NB, w, nw),
           "paged_prefill")
    return out


def partition_stats(query, key_cache, value_cache, block_tables, context_lens, dtype,
                    s: int, h: int, partition_size: int, scale=None):
    """Per-partition (m, l, o) of one (s, h): partition p covers tokens
    [p*P, min((p+1)*P, ctx))."""
    q = bits16(query)
    kc = np.ascontiguousarray(key_cache if isinstance(key_cache, np.ndarray) else bits16(key_cache))
    vc = np.ascontiguousarray(value_cache if isinstance(value_cache, np.ndarray) else bits16(value_cache))
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    cl = np.ascontiguousarray(context_lens, dtype=np.int32)
    S, H, d = q.shape
    NB, Hkv, B, _ = kc.shape
    if scale is None:
        scale = default_scale(d)
    nmax = max(1, -(-int(cl[s]) // partition_size))
    m = np.empty(nmax, np.float64)
    l = np.empty(nmax, np.float64)
    o = np.empty((nmax, d), np.float64)
    n = _check(lib().oracle_partition_stats(_ptr(q), _ptr(kc), _ptr(vc), _ptr(bt), _ptr(cl), S,
                                            bt.shape[1], B, H, Hkv, d, float(scale), _is_bf16(dtype),
                                            NB, s, h, partition_size, _ptr(m), _ptr(l), _ptr(o)),
               "partition_stats")
    return m[:n].copy(), l[:n].copy(), o[:n].copy()


def merge_partitions(m, l, o) -> np.ndarray:
    m = np.ascontiguousarray(m, np.float64)
    l = np.ascontiguousarray(l, np.float64)
    o = np.ascontiguousarray(o, np.float64)
    n = m.shape[0]
    d = o.shape[1] if o.ndim == 2 else 0
    out = np.empty(d, np.float64)
    lib().oracle_merge_partitions(_ptr(m), _ptr(l), _ptr(o), n, d, _ptr(out))
    return out
