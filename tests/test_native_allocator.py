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


def _groups(ref, rng, n):
    """n sequence groups (a prompt and its forks, some with suffixes) on the
    reference allocator, returned with the op script that rebuilds them."""
    script, groups = [], []
    for _ in range(n):
        plen, k = int(rng.integers(1, 12)), int(rng.integers(1, 4))
        sfx = [int(rng.integers(0, 6)) for _ in range(k)]
        script.append((plen, k, sfx))
    return script


def _build(alloc, script):
    groups = []
    for plen, k, sfx in script:
        root = alloc.seq_new(plen)
        g = [root] + [alloc.fork(root) for _ in range(k - 1)]
        for sid, n in zip(g, sfx):
            for _ in range(n):
                alloc.append(sid)
        groups.append(g)
    return groups


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_swap_moves_match_reference(seed):
    """Random groups swapped out to a CPU pool and back in random order: both
    pools' tables, counts, free lists and the copy pairs match the reference
    allocator exactly; too-small pools and half groups are refused without a
    change."""
    rng = np.random.default_rng(seed)
    NG, NC, B = 64, 40, 4
    og = rng.permutation(NG).astype(np.int32)
    oc = rng.permutation(NC).astype(np.int32)
    ng, nc = pkv.BlockAllocator(NG, B, og), pkv.BlockAllocator(NC, B, oc)
    rg, rc = RefAllocator(NG, B, og), RefAllocator(NC, B, oc)
    script = _groups(rg, rng, 6)
    gn, gr = _build(ng, script), _build(rg, script)
    assert gn == gr
    where = ["gpu"] * len(gn)
    for step in range(30):
        i = int(rng.integers(len(gn)))
        src_n, dst_n, src_r, dst_r = (ng, nc, rg, rc) if where[i] == "gpu" else (nc, ng, rc, rg)
        seqs = gn[i]
        shares = any(src_r.block_ref(b) > 1 for b in src_r.block_table(seqs[0]))
        if len(seqs) > 1 and shares and rng.random() < 0.3:
            # half a sharing group: refused, nothing changes
            with pytest.raises(pkv.PkvError):
                src_n.move_group(dst_n, seqs[:1])
            with pytest.raises(ValueError):
                src_r.move_group(dst_r, seqs[:1])
            continue
        try:
            ids_r, pairs_r = src_r.move_group(dst_r, seqs)
        except AllocatorOOM:
            with pytest.raises(pkv.PkvOOM):
                src_n.move_group(dst_n, seqs)
            continue
        ids_n, pairs_n = src_n.move_group(dst_n, seqs)
        assert ids_n == ids_r
        assert [tuple(p) for p in pairs_n.tolist()] == pairs_r
        gn[i] = ids_n
        where[i] = "cpu" if where[i] == "gpu" else "gpu"
        for a_n, a_r, side in ((ng, rg, "gpu"), (nc, rc, "cpu")):
            live = [s for g, w in zip(gn, where) if w == side for s in g]
            _same_state(a_n, a_r, live)


def test_swap_rejects_mismatched_pools():
    a, b = pkv.BlockAllocator(8, 4), pkv.BlockAllocator(8, 8)
    s = a.seq_new(5)
    with pytest.raises(pkv.PkvError):
        a.move_group(b, [s])
    with pytest.raises(pkv.PkvError):
        a.move_group(a, [s])
    with pytest.raises(pkv.PkvError):
        a.move_group(pkv.BlockAllocator(8, 4), [s, s])


def test_beam_step_fig9():
    """The pages' Figure 9 step, natively: blocks 9-12 for the survivors, 2,
    4, 5, 8 back in the pool."""
    g = golden("beam_prune_fig9.json")
    a = pkv.BlockAllocator(16, 2)
    C = a.seq_new(2)
    A = a.fork(C)
    a.append(A); a.append(A)
    a.append(C); a.append(C)
    D = a.fork(A)
    a.append(A); a.append(A)
    Bc = a.fork(A)
    a.append(C); a.append(C)
    a.append(D); a.append(D)
    a.append(A); a.append(A)
    a.append(Bc); a.append(Bc)
    a.append(C); a.append(C)
    new, slots, pairs = a.beam_step([A, Bc, C, D], [0, 0, 1, 1])
    assert [a.block_table(s)[-1] for s in new] == g["new_for_survivors"] and len(pairs) == 0
    assert sorted(a.free_list()[:4]) == g["freed_on_prune"]


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_beam_search_matches_reference(seed):
    """Random beam searches (width 2-6, random parent choices, pools small
    enough to run out): every step's ids, slots, copy pairs, tables, counts and
    free lists match the reference allocator, and an out-of-blocks step
    changes nothing on either side."""
    rng = np.random.default_rng(seed)
    NB, B = 48, 4
    order = rng.permutation(NB).astype(np.int32)
    nat, ref = pkv.BlockAllocator(NB, B, order), RefAllocator(NB, B, order)
    width = int(rng.integers(2, 7))
    plen = int(rng.integers(1, 20))
    beams_n = [nat.seq_new(plen)]
    beams_r = [ref.seq_new(plen)]
    ooms = 0
    for step in range(60):
        kn = width if step else width
        parents = rng.integers(0, len(beams_r), size=kn)
        parents = np.minimum(parents, rng.integers(0, len(beams_r), size=kn))   # favour low ranks
        try:
            new_r, slots_r, pairs_r = ref.beam_step(beams_r, parents)
        except AllocatorOOM:
            with pytest.raises(pkv.PkvOOM):
                nat.beam_step(beams_n, parents)
            ooms += 1
            _same_state(nat, ref, beams_r)
            # make room: drop the last beam on both sides
            nat.free(beams_n.pop())
            ref.free(beams_r.pop())
            if not beams_r:
                break
            continue
        new_n, slots_n, pairs_n = nat.beam_step(beams_n, parents)
        assert new_n == new_r and slots_n.tolist() == slots_r
        assert [tuple(p) for p in pairs_n.tolist()] == pairs_r
        beams_n, beams_r = new_n, new_r
        _same_state(nat, ref, beams_r)
        assert nat.blocks_in_use() == ref.blocks_in_use()
