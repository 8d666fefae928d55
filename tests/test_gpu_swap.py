"""Swapping: pkv_move_group + swap_blocks through the engine, against the
oracle's group move and cross-pool copy.  Blocks move between the GPU pool and
a pinned host pool the kernel reads and writes directly; a round trip leaves
every sequence's attention output bit-identical."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_139_gb300 as pkv
import workloads
from paged_kv_cache_139_gb300.engine import HostKVPool, PagedKVCache

pytestmark = pytest.mark.gpu


def _groups(eng, rng, n, prompt=(5, 200), forks=(1, 4), suffix=(0, 40)):
    groups = []
    for _ in range(n):
        root = eng.new_sequence(int(rng.integers(*prompt)))
        g = [root] + [eng.fork(root) for _ in range(int(rng.integers(*forks)) - 1)]
        for sid in g:
            for _ in range(int(rng.integers(*suffix))):
                eng.alloc.append(sid)
        groups.append(g)
    return groups


def _attend(eng, seqs, q):
    plan = eng.plan_tables(seqs)
    dev = eng.upload(plan)
    out = eng.attend(q, dev)
    pkv.check()
    return out


@pytest.mark.parametrize("B,dtype", [(16, torch.float16), (4, torch.bfloat16), (128, torch.float16)])
def test_swap_round_trip(cuda_device, B, dtype):
    rng = np.random.default_rng(B)
    Hkv, d, H = 4, 128, 8
    NB, NC = 600 * 16 // B + 40, 500 * 16 // B + 40
    kc = workloads.normal((NB, Hkv, B, d), "bf16" if dtype == torch.bfloat16 else "f16", 7 + B, cuda_device)
    vc = workloads.normal((NB, Hkv, B, d), "bf16" if dtype == torch.bfloat16 else "f16", 8 + B, cuda_device)
    eng = PagedKVCache(NB, Hkv, d, B, dtype, cuda_device, 64 * 16 // B + 8, rng.permutation(NB),
                       key_cache=kc, value_cache=vc)
    host = HostKVPool(NC, Hkv, d, B, dtype, rng.permutation(NC))
    groups = _groups(eng, rng, 6)
    seqs = [s for g in groups for s in g]
    q = workloads.normal((len(seqs), H, d), "bf16" if dtype == torch.bfloat16 else "f16", 9, cuda_device)
    before = _attend(eng, seqs, q)
    gpu_k, gpu_v = oracle.bits16(eng.key_cache), oracle.bits16(eng.value_cache)
    host_k0, host_v0 = oracle.bits16(host.key_cache), oracle.bits16(host.value_cache)
    out_ids, out_pairs = [], []
    for g in groups[::2]:                       # every other group leaves
        ids, pairs = eng.swap_out(g, host)
        out_ids.append(ids)
        out_pairs.append(pairs)
    pkv.check()
    # the host pool now holds exactly the oracle's copies
    for pairs in out_pairs:
        oracle.copy_blocks_between(host_k0, gpu_k, pairs)
        oracle.copy_blocks_between(host_v0, gpu_v, pairs)
    assert np.array_equal(oracle.bits16(host.key_cache), host_k0)
    assert np.array_equal(oracle.bits16(host.value_cache), host_v0)
    # the freed GPU blocks are clobbered by new sequences before the group comes back
    filler = eng.new_sequence(min(eng.alloc.num_free(), 40) * B)
    t = eng.alloc.block_table(filler)
    eng.key_cache[t] = float("nan")
    eng.value_cache[t] = float("nan")
    eng.free(filler)
    back = []
    for ids in out_ids:
        new_ids, _ = eng.swap_in(ids, host)
        back.append(new_ids)
    pkv.check()
    assert host.alloc.num_free() == NC
    now = [s for g in groups[1::2] for s in g] + [s for g in back for s in g]
    order = [s for g in groups[1::2] for s in g] + [s for g in groups[::2] for s in g]
    after = _attend(eng, now, q[[seqs.index(s) for s in order]])
    assert torch.equal(after, before[[seqs.index(s) for s in order]])


def test_swap_many_small_blocks(cuda_device):
    """More pairs than one grid row holds (65535): the kernel loops over them."""
    n, NB = 70000, 70010
    src = torch.randint(-30000, 30000, (NB, 1, 4, 64), dtype=torch.int16, device=cuda_device).view(torch.float16)
    dst = torch.zeros((NB, 1, 4, 64), dtype=torch.float16).pin_memory()
    perm = torch.randperm(NB)[:n].to(torch.int32)
    pairs = torch.stack([perm, torch.arange(n, dtype=torch.int32)], 1).contiguous()
    pkv.swap_blocks(dst, src, pairs.to(cuda_device))
    pkv.check()
    assert torch.equal(dst[:n].view(torch.int16), src[perm.long().to(cuda_device)].cpu().view(torch.int16))
    assert (dst[n:].view(torch.int16) == 0).all()


def test_swap_bad_pair_is_latched(cuda_device):
    src = torch.ones((8, 2, 16, 64), dtype=torch.float16, device=cuda_device)
    dst = torch.zeros((4, 2, 16, 64), dtype=torch.float16).pin_memory()
    pairs = torch.tensor([[1, 0], [2, 9]], dtype=torch.int32).pin_memory()
    pkv.swap_blocks(dst, src, pairs)
    with pytest.raises(pkv.PkvError) as e:
        pkv.check()
    assert e.value.status == 3
    assert (dst[0] == 1).all() and (dst[1:] == 0).all()


def test_swap_between_device_pools(cuda_device):
    a = workloads.normal((10, 2, 8, 64), "f16", 3, cuda_device)
    b = torch.zeros((6, 2, 8, 64), dtype=torch.float16, device=cuda_device)
    pairs = torch.tensor([[9, 0], [0, 5], [4, 2]], dtype=torch.int32, device=cuda_device)
    pkv.swap_blocks(b, a, pairs)
    pkv.check()
    want = oracle.bits16(torch.zeros_like(b))
    oracle.copy_blocks_between(want, oracle.bits16(a), pairs.cpu().numpy())
    assert np.array_equal(oracle.bits16(b), want)


def test_swap_bench_workload(cuda_device):
    """The benchmark's swap workload (32 Llama-2-7B-layer sequences, 1.1 GB of K+V) swapped out and
    back through the engine: the host pool holds the oracle's copies, and the GPU pool after the
    round trip holds every sequence's blocks unchanged."""
    w = workloads.swap()
    t = workloads.tensors(w, device=cuda_device)
    eng = PagedKVCache(w.num_blocks, w.num_kv_heads, w.head_dim, w.block_size, w.torch_dtype, cuda_device,
                       w.max_blocks_per_seq, workloads.free_order(w.num_blocks, w.seed),
                       key_cache=t["key_cache"], value_cache=t["value_cache"])
    host = HostKVPool(w.num_blocks, w.num_kv_heads, w.head_dim, w.block_size, w.torch_dtype)
    ids = [eng.new_sequence(int(c)) for c in w.context_lens]
    tables0 = [eng.alloc.block_table(s) for s in ids]
    gk, gv = oracle.bits16(eng.key_cache), oracle.bits16(eng.value_cache)
    hids, out_pairs = eng.swap_out(ids, host)
    pkv.check()
    want_k = np.zeros_like(gk)
    oracle.copy_blocks_between(want_k, gk, out_pairs)
    hk = oracle.bits16(host.key_cache)
    assert np.array_equal(hk[out_pairs[:, 1]], want_k[out_pairs[:, 1]])
    eng.key_cache.zero_()
    eng.value_cache.zero_()
    gids, in_pairs = eng.swap_in(hids, host)
    pkv.check()
    nk, nv = oracle.bits16(eng.key_cache), oracle.bits16(eng.value_cache)
    for s0, s1 in zip(ids, gids):
        t0, t1 = tables0[ids.index(s0)], eng.alloc.block_table(s1)
        assert np.array_equal(nk[t1], gk[t0]) and np.array_equal(nv[t1], gv[t0])
