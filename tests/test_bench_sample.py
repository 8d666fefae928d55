"""The CPU baseline's compact sample (bench.py): the sampled sequences'
blocks gathered into a compact pool with renumbered tables and slots must
give the oracle exactly the outputs it gives on the whole pool."""
import numpy as np

import bench
import oracle
import workloads


def _full_and_compact(w):
    tables, ctx, slots = bench.reference_plan(w)
    t = workloads.tensors(w, "cpu")
    kc, vc = oracle.bits16(t["key_cache"]), oracle.bits16(t["value_cache"])
    oracle.cache_write(t["key"], t["value"], kc, vc, slots)
    sel = bench.sample_sequences(w, ctx, max_bytes=int(ctx.astype(np.int64).sum()) * w.kv_bytes_per_token // 2)
    blocks, t2, c2, sl2 = bench.compact_tables(w, sel, tables, ctx, slots)
    return t, tables, ctx, slots, kc, vc, sel, blocks, t2, c2, sl2


def test_compact_sample_matches_the_whole_pool():
    w = workloads.opt13b(num_seqs=6)
    t, tables, ctx, slots, kc, vc, sel, blocks, t2, c2, sl2 = _full_and_compact(w)
    assert 1 <= len(sel) < w.num_seqs
    want = oracle.paged_attention(t["query"], kc, vc, tables, ctx, w.dtype)[sel]
    # the compact pool: the sampled sequences' blocks before the decode tokens' write, then their write
    t0 = workloads.tensors(w, "cpu")
    ck = oracle.bits16(t0["key_cache"][blocks])
    cv = oracle.bits16(t0["value_cache"][blocks])
    oracle.cache_write(t0["key"][sel], t0["value"][sel], ck, cv, sl2)
    got = oracle.paged_attention(t0["query"][sel], ck, cv, t2, c2, w.dtype)
    assert np.array_equal(got, want)


def test_compact_sample_keeps_shared_blocks_once():
    """Parallel sampling: sequences that share prompt blocks keep sharing them
    in the compact pool (each distinct block once), and every new-token slot
    lands in a block of its own sequence's table."""
    w = workloads.sampling(num_prompts=3, max_suffix=40)
    tables, ctx, slots = bench.reference_plan(w)
    sel = list(range(w.num_seqs))
    blocks, t2, c2, sl2 = bench.compact_tables(w, sel, tables, ctx, slots)
    used = {int(b) for i in sel for b in tables[i][: -(-int(ctx[i]) // w.block_size)]}
    assert len(blocks) == len(used | {int(s) // w.block_size for s in slots})
    for i in range(len(sel)):
        nb = -(-int(c2[i]) // w.block_size)
        assert int(sl2[i]) // w.block_size in set(t2[i][:nb].tolist())


def test_profiles_carry_traffic_for_the_current_library():
    """Every workload whose bench line reports roofline.traffic finds a DRAM
    traffic line under profiles/ for the library version that is built, so a
    version bump without new (or carried-over) ncu figures is caught here."""
    import paged_kv_cache_139_gb300 as pkv
    v = pkv.version()
    for name in ("llama7b_B16_d128", "opt13b", "sampling", "longgqa", "prefix", "swap"):
        t = bench.profile_traffic(name, v)
        assert t is not None and t > 0, f"no traffic_bytes_per_launch[{name}@{v}] under profiles/"
