"""The library's native allocator against the reference allocator, step by
step and bit for bit: block tables, reference counts, slots, copy-on-write
pairs and free lists (CPU only)."""
import random

import numpy as np
import pytest

import paged_kv_cache_139_gb300 as pkv
from oracle import AllocatorOOM, RefAllocator
from pins import golden


def _same_state(nat: pkv.BlockAllocator, ref: RefAllocator, live):
    assert nat.num_free() == ref.num_free()
    assert nat.free_list() == ref.free_list()
    assert [nat.block_ref(b) for b in range(ref.num_blocks)] == ref.ref
    for s in live:
        assert nat.block_table(s) == ref.block_table(s)
        assert nat.seq_len(s) == ref.seq_len(s)


def test_request_flow_fig6():
    g = golden("request_flow_fig6.json")
    order = g["free_order_head"] + [b for b in range(8) if b not in g["free_order_head"]]
    a = pkv.BlockAllocator(8, g["block_size"], order)
    sid = a.seq_new(g["prompt_tokens"])
    assert a.block_table(sid) == g["after_prefill"]["blocks"]
    assert a.append(sid) == (7, None)
    assert a.block_table(sid) == g["after_decode_1"]["blocks"]
    assert a.append(sid) == (12, None)
    assert a.block_table(sid) == g["after_decode_2"]["blocks"]


def test_cow_and_fork():
    a = pkv.BlockAllocator(8, 4)
    s1 = a.seq_new(7)
    s2 = a.fork(s1)
    shared = a.block_table(s1)
    assert [a.block_ref(b) for b in shared] == [2, 2]
    slot, cow = a.append(s1)
    assert cow == (shared[1], a.block_table(s1)[1]) and a.block_ref(shared[1]) == 1
    slot2, cow2 = a.append(s2)
    assert cow2 is None and slot2 == shared[1] * 4 + 3


def test_oom_is_all_or_nothing():
    a = pkv.BlockAllocator(3, 4)
    s = a.seq_new(8)
    with pytest.raises(pkv.PkvOOM):
        a.seq_new(5)
    f = a.fork(s)
    a.append(s)
    before = (a.free_list(), a.block_table(s), a.block_table(f), [a.block_ref(b) for b in range(3)])
    with pytest.raises(pkv.PkvOOM):
        a.append_batch([f, f])
    assert (a.free_list(), a.block_table(s), a.block_table(f), [a.block_ref(b) for b in range(3)]) == before


def test_unknown_sequence_is_einval():
    a = pkv.BlockAllocator(4, 4)
    with pytest.raises(pkv.PkvError) as e:
        a.append(3)
    assert e.value.status_name == "PKV_EINVAL"
    s = a.seq_new(1)
    a.free(s)
    with pytest.raises(pkv.PkvError):
        a.free(s)
    with pytest.raises(pkv.PkvError):
        pkv.BlockAllocator(4, 4, [0, 1, 1, 2])           # not a permutation


def test_build_block_tables():
    a = pkv.BlockAllocator(16, 4, list(range(15, -1, -1)))
    s0 = a.seq_new(5)
    s1 = a.seq_new(0)
    s2 = a.seq_new(12)
    t, c = a.build_block_tables([s2, s0, s1], 4)
    assert c.tolist() == [12, 5, 0]
    assert t[0].tolist() == a.block_table(s2) + [-1]
    assert t[1].tolist() == a.block_table(s0) + [-1, -1]
    assert t[2].tolist() == [-1] * 4
    with pytest.raises(pkv.PkvError):
        a.build_block_tables([s2], 2)                       # too narrow


@pytest.mark.parametrize("seed", range(12))
def test_random_sequences_match_reference(seed):
    rnd = random.Random(1000 + seed)
    B = rnd.choice([1, 2, 4, 8, 16])
    NB = rnd.randint(4, 96)
    order = rnd.sample(range(NB), NB)
    nat = pkv.BlockAllocator(NB, B, order)
    ref = RefAllocator(NB, B, order)
    live = []
    for step in range(400):
        op = rnd.random()
        if op < 0.15 or not live:
            n = rnd.randint(0, 4 * B)
            try:
                r = ref.seq_new(n)
            except AllocatorOOM:
                with pytest.raises(pkv.PkvOOM):
                    nat.seq_new(n)
            else:
                assert nat.seq_new(n) == r
                live.append(r)
        elif op < 0.3:
            p = rnd.choice(live)
            c = ref.fork(p)
            assert nat.fork(p) == c
            live.append(c)
        elif op < 0.5:
            s = rnd.choice(live)
            try:
                want = ref.append(s)
            except AllocatorOOM:
                with pytest.raises(pkv.PkvOOM):
                    nat.append(s)
            else:
                assert nat.append(s) == want
        elif op < 0.85:
            seqs = [rnd.choice(live) for _ in range(rnd.randint(1, 2 * len(live)))]
            try:
                slots, pairs = ref.append_batch(seqs)
            except AllocatorOOM:
                with pytest.raises(pkv.PkvOOM):
                    nat.append_batch(seqs)
            else:
                ns, npairs = nat.append_batch(seqs)
                assert ns.tolist() == slots
                assert [tuple(p) for p in npairs.tolist()] == pairs
                pkv.validate_copy_pairs(npairs, NB)
        else:
            s = rnd.choice(live)
            ref.free(s)
            nat.free(s)
            live.remove(s)
        _same_state(nat, ref, live)
