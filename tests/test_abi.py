"""The C-ABI library loads and exports every symbol include/*.h declares;
host-side argument checks reject bad calls before any launch (CPU only)."""
import ctypes
import glob
import os
import re

import numpy as np
import pytest

import paged_kv_cache_139_gb300 as pkv
from paged_kv_cache_139_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", text, re.M):
            names.append(m.group(1))
    return sorted(set(n for n in names if n not in ("if", "while", "for", "return", "sizeof")))


def test_library_is_in_tree():
    assert os.path.realpath(pkv.library_path()).startswith(os.path.realpath(ROOT))


def test_every_declared_symbol_is_exported():
    L = _lib.load()
    names = _declared()
    assert len(names) >= 20
    missing = [n for n in names if not hasattr(L, n)]
    assert not missing, missing
    # and the binding declares a signature for each
    assert set(names) <= set(_lib.SIGNATURES), set(names) - set(_lib.SIGNATURES)


def test_version():
    assert pkv.version() >= 100


def _call_attention(**over):
    args = dict(out=16, query=16, kc=16, vc=16, bt=16, cl=16, S=2, mb=4, mcl=0, B=16, NB=8, H=4, Hkv=2,
                d=128, scale=0.1, P=0, ws=None, wsb=0, dt=0, st=None)
    args.update(over)
    L = _lib.load()
    return L.paged_attention_decode(args["out"], args["query"], args["kc"], args["vc"], args["bt"], args["cl"],
                                    args["S"], args["mb"], args["mcl"], args["B"], args["NB"], args["H"],
                                    args["Hkv"], args["d"], args["scale"], args["P"], args["ws"], args["wsb"],
                                    args["dt"], args["st"])


@pytest.mark.parametrize("over", [
    dict(d=96), dict(d=0), dict(B=12), dict(B=2), dict(B=256), dict(H=5, Hkv=2), dict(Hkv=0),
    dict(P=48), dict(P=-32), dict(mcl=65), dict(dt=7), dict(S=-1), dict(out=None), dict(bt=None),
    dict(query=18),
])
def test_attention_rejects_bad_arguments(over):
    assert _call_attention(**over) == 1                  # PKV_EINVAL, before any launch
    assert _lib.load().pkv_last_error_string()


def _call_prefill(**over):
    args = dict(out=16, query=16, kc=16, vc=16, bt=16, cl=16, qs=16, S=2, T=10, mql=0, mb=4, B=16, NB=8, H=4,
                Hkv=2, d=128, scale=0.1, ws=None, wsb=0, dt=0, st=None)
    args.update(over)
    return _lib.load().paged_attention_prefill(
        args["out"], args["query"], args["kc"], args["vc"], args["bt"], args["cl"], args["qs"], args["S"],
        args["T"], args["mql"], args["mb"], args["B"], args["NB"], args["H"], args["Hkv"], args["d"],
        args["scale"], args["ws"], args["wsb"], args["dt"], args["st"])


@pytest.mark.parametrize("over", [
    dict(d=96), dict(d=0), dict(B=12), dict(B=2), dict(B=256), dict(H=5, Hkv=2), dict(Hkv=0), dict(dt=7),
    dict(S=-1), dict(T=-3), dict(mql=-1), dict(S=70000), dict(out=None), dict(qs=None), dict(query=18),
    dict(NB=0), dict(scale=float("inf")), dict(scale=float("nan")), dict(scale=0.0), dict(scale=-0.1),
    dict(ws=16, wsb=128), dict(ws=24, wsb=256), dict(S=65535, H=65535, Hkv=1, T=1 << 20, mql=1 << 20),
])
def test_prefill_rejects_bad_arguments(over):
    assert _call_prefill(**over) == 1                    # PKV_EINVAL, before any launch
    assert _lib.load().pkv_last_error_string()


def test_prefill_with_nothing_to_do_launches_nothing():
    assert _call_prefill(T=0) == 0 and _call_prefill(S=0) == 0


def test_attention_workspace_needed():
    # 4 blocks of 16 = 64 tokens and partitions of 32: two partitions -> workspace required
    assert pkv.paged_attention_workspace_size(2, 4, 2, 128, 64, 32) > 0
    assert _call_attention(P=32) == 1
    assert pkv.paged_attention_workspace_size(2, 4, 2, 128, 64, 64) == 256     # the counters only


def test_workspace_size_formula():
    # m and l: S*H*P floats each, o: S*H*P*d floats, each rounded up to 256 bytes
    S, H, d, ctx, P = 8, 32, 128, 32768, 512
    n = S * H * (ctx // P)
    r = lambda x: (x + 255) // 256 * 256
    # + one partition counter per (sequence, head)
    assert pkv.paged_attention_workspace_size(S, H, 8, d, ctx, P) == 256 + r(4 * n) * 2 + r(4 * n * d) + r(4 * S * H)


def test_workspace_init_rejects_bad_arguments():
    L = _lib.load()
    assert L.paged_attention_workspace_init(None, 4096, None) == 1
    assert L.paged_attention_workspace_init(16, 128, None) == 1        # smaller than the counters
    assert L.paged_attention_workspace_init(24, 4096, None) == 1       # misaligned


def test_cache_write_rejects_bad_arguments():
    L = _lib.load()
    assert L.kv_reshape_and_cache(16, 16, 16, 16, 16, 4, 2, 60, 16, 8, 0, None) == 1   # d % 8
    assert L.kv_reshape_and_cache(16, 16, 16, 16, 16, 4, 2, 64, 12, 8, 0, None) == 1   # block not 2^k
    assert L.kv_reshape_and_cache(16, 16, 16, 16, None, 4, 2, 64, 16, 8, 0, None) == 1
    assert L.kv_reshape_and_cache(16, 16, 16, 24, 16, 4, 2, 64, 16, 8, 0, None) == 1   # misaligned
    assert L.kv_reshape_and_cache(None, None, None, None, None, 0, 2, 64, 16, 8, 0, None) == 0  # empty


def test_copy_blocks_rejects_bad_arguments():
    L = _lib.load()
    assert L.copy_blocks(16, 16, 3, 100, 8, None) == 1          # not a multiple of 16
    assert L.copy_blocks(16, 16, -1, 128, 8, None) == 1
    assert L.copy_blocks(None, 16, 3, 128, 8, None) == 1
    assert L.copy_blocks(None, None, 0, 128, 8, None) == 0       # nothing to do


@pytest.mark.parametrize("pairs,ok", [
    ([(1, 2), (3, 4)], True),
    ([], True),
    ([(1, 2), (3, 2)], False),            # destination twice
    ([(1, 2), (2, 4)], False),            # destination is also a source
    ([(1, 9)], False),                    # out of range
    ([(-1, 2)], False),
    ([(5, 6), (5, 7)], True),             # one source, two copies
])
def test_validate_copy_pairs(pairs, ok):
    if ok:
        pkv.validate_copy_pairs(pairs, 8)
    else:
        with pytest.raises(pkv.PkvError):
            pkv.validate_copy_pairs(pairs, 8)


def test_default_partition_size_follows_head_dim():
    """512 tokens at head_dim 128; 2048 at head_dim 64 (the same bytes per
    work item) unless that leaves fewer than 2048 items; an explicit size
    always wins."""
    f = _lib.load().paged_attention_partition_size
    assert f(256, 32, 32, 128, 4096, 0) == 512
    assert f(256, 32, 32, 64, 4096, 0) == 2048
    assert f(16, 32, 32, 64, 4096, 0) == 1024      # 16 x 32 x 4 = 2048 items at 1024
    assert f(1, 8, 8, 64, 32768, 0) == 512         # too few items at 1024 and 2048
    assert f(256, 32, 32, 64, 4096, 256) == 256
