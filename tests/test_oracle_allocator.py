"""The reference allocator against the pages' worked examples and against
invariants that hold after any sequence of operations (CPU only)."""
import random

import pytest

import oracle
from oracle import AllocatorOOM, RefAllocator
from pins import golden


def _filled_last(a, sid):
    n = a.seq_len(sid)
    return n - (len(a.block_table(sid)) - 1) * a.B if n else 0


def test_request_flow_fig6():
    g = golden("request_flow_fig6.json")
    B = g["block_size"]
    order = g["free_order_head"] + [b for b in range(8) if b not in g["free_order_head"]]
    a = RefAllocator(8, B, order)
    sid = a.seq_new(g["prompt_tokens"])
    assert a.block_table(sid) == g["after_prefill"]["blocks"]
    assert _filled_last(a, sid) == g["after_prefill"]["filled_last"]
    slot, cow = a.append(sid)
    assert cow is None and a.block_table(sid) == g["after_decode_1"]["blocks"]
    assert _filled_last(a, sid) == g["after_decode_1"]["filled_last"]
    assert slot == 1 * B + 3
    slot, cow = a.append(sid)
    assert cow is None and a.block_table(sid) == g["after_decode_2"]["blocks"]
    assert _filled_last(a, sid) == g["after_decode_2"]["filled_last"]
    assert slot == 3 * B + 0
    ra = g["request_A"]
    assert a.seq_len(sid) == ra["tokens"] and a.block_table(sid) == ra["blocks"]
    assert len(a.block_table(sid)) * B - a.seq_len(sid) == ra["empty_slots"]


def test_cow_stages_fig8():
    g = golden("cow_stages_fig8.json")
    B = g["block_size"]
    a = RefAllocator(8, B)
    s1 = a.seq_new(g["prompt_tokens"])
    s2 = a.fork(s1)
    shared = a.block_table(s1)
    assert shared == a.block_table(s2) and len(shared) == g["stage2"]["shared_blocks"]
    assert all(a.block_ref(b) == g["stage2"]["ref_count"] for b in shared)
    # stage 3: the first writer copies the shared, partly filled last block
    slot, cow = a.append(s1)
    assert cow is not None and cow[0] == shared[-1]
    assert a.block_table(s1) == [shared[0], cow[1]]
    assert a.block_ref(shared[-1]) == g["stage3"]["original_ref_after"]
    assert a.block_ref(shared[0]) == 2                  # the full first block is never copied
    assert slot == cow[1] * B + g["prompt_tokens"] % B
    # the second writer finds count 1 and writes in place
    slot2, cow2 = a.append(s2)
    assert cow2 is None and a.block_table(s2) == shared
    assert slot2 == shared[-1] * B + g["prompt_tokens"] % B
    # stage 4: both grow into their own new blocks
    _, c1 = a.append(s1)
    _, c2 = a.append(s2)
    assert c1 is None and c2 is None
    t1, t2 = a.block_table(s1), a.block_table(s2)
    assert len(t1) == len(t2) == 3 and t1[2] != t2[2]
    assert a.block_ref(t1[2]) == a.block_ref(t2[2]) == 1


def test_full_shared_block_never_copied():
    a = RefAllocator(8, 4)
    s1 = a.seq_new(8)                                  # two full blocks
    s2 = a.fork(s1)
    _, c1 = a.append(s1)
    _, c2 = a.append(s2)
    assert c1 is None and c2 is None
    assert a.block_table(s1)[:2] == a.block_table(s2)[:2]


def _build_fig9_tree():
    """Candidates A=[0,1,3,6], B=[0,1,3,7], C=[0,2,4,8], D=[0,1,5] (B = 2,
    every block full), built with fork/append in block-id order."""
    a = RefAllocator(16, 2)
    C = a.seq_new(2)                                    # [0]
    A = a.fork(C)
    a.append(A); a.append(A)                            # A: [0,1]
    a.append(C); a.append(C)                            # C: [0,2]
    D = a.fork(A)                                       # D: [0,1]
    a.append(A); a.append(A)                            # A: [0,1,3]
    Bc = a.fork(A)                                      # B: [0,1,3]
    a.append(C); a.append(C)                            # C: [0,2,4]
    a.append(D); a.append(D)                            # D: [0,1,5]
    a.append(A); a.append(A)                            # A: [0,1,3,6]
    a.append(Bc); a.append(Bc)                          # B: [0,1,3,7]
    a.append(C); a.append(C)                            # C: [0,2,4,8]
    return a, A, Bc, C, D


def test_beam_prune_fig9_tree():
    g = golden("beam_prune_fig9.json")
    a, A, Bc, C, D = _build_fig9_tree()
    assert a.block_table(A) == [0, 1, 3, 6] and a.block_table(Bc) == [0, 1, 3, 7]
    assert a.block_table(C) == [0, 2, 4, 8] and a.block_table(D) == [0, 1, 5]
    assert a.block_ref(g["shared_by_all"]) == 4
    # survivors A and B each branch in two and grow into new blocks
    new = []
    for parent in (A, Bc):
        child = a.fork(parent)
        for s in (parent, child):
            slot, cow = a.append(s)
            assert cow is None
            new.append(a.block_table(s)[-1])
    assert new == g["new_for_survivors"]
    a.free(C)
    a.free(D)
    freed = sorted(b for b in range(9) if a.block_ref(b) == 0)
    assert freed == g["freed_on_prune"]
    assert sorted(a.free_list()[:4]) == g["freed_on_prune"]
    assert a.block_ref(0) == 4 and a.block_ref(1) == 4


def test_oom_changes_nothing():
    a = RefAllocator(3, 4)
    s = a.seq_new(8)
    before = (list(a.ref), a.free_list(), a.block_table(s), a.seq_len(s))
    with pytest.raises(AllocatorOOM):
        a.seq_new(5)
    f = a.fork(s)
    a.append(s)                                         # takes the last block
    before = (list(a.ref), a.free_list(), a.block_table(s), a.block_table(f))
    with pytest.raises(AllocatorOOM):
        a.append_batch([f, f])                          # needs one more block
    assert (list(a.ref), a.free_list(), a.block_table(s), a.block_table(f)) == before


def _check_invariants(a: RefAllocator, live: dict):
    count = [0] * a.num_blocks
    for sid in live:
        t = a.block_table(sid)
        assert len(t) == oracle.blocks_needed(a.seq_len(sid), a.B)
        for b in t:
            count[b] += 1
    assert count == a.ref
    free = a.free_list()
    assert len(set(free)) == len(free)
    assert sorted(free) == [b for b in range(a.num_blocks) if a.ref[b] == 0]


def test_random_operation_invariants():
    rnd = random.Random(139)
    for trial in range(20):
        B = rnd.choice([1, 2, 4, 16])
        NB = rnd.randint(4, 64)
        a = RefAllocator(NB, B, rnd.sample(range(NB), NB))
        live = {}
        for _ in range(300):
            op = rnd.random()
            try:
                if op < 0.2 or not live:
                    sid = a.seq_new(rnd.randint(0, 3 * B))
                    live[sid] = True
                elif op < 0.35:
                    sid = a.fork(rnd.choice(list(live)))
                    live[sid] = True
                elif op < 0.85:
                    seqs = rnd.sample(list(live), rnd.randint(1, len(live)))
                    lens = {s: a.seq_len(s) for s in seqs}
                    slots, pairs = a.append_batch(seqs)
                    for s, slot in zip(seqs, slots):
                        t = a.block_table(s)
                        assert slot == t[lens[s] // B] * B + lens[s] % B
                        # copy-on-write: the written block belongs to the writer alone
                        assert a.block_ref(slot // B) == 1
                    for src, dst in pairs:
                        assert a.block_ref(dst) >= 1 and src != dst
                else:
                    sid = rnd.choice(list(live))
                    a.free(sid)
                    del live[sid]
            except AllocatorOOM:
                pass
            _check_invariants(a, live)
