"""Beam search through the engine against the oracle: every step's host plan
(the native beam step) replays on the reference allocator, the device copies
and cache writes replay on the oracle's pools, and the last step's attention
over all beams matches the oracle."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_139_gb300 as pkv
import workloads
from cases import assert_close
from paged_kv_cache_139_gb300.engine import PagedKVCache

pytestmark = pytest.mark.gpu


def _beam_search(cuda_device, width, B, dtype, H, Hkv, prompts, steps, seed):
    rng = np.random.default_rng(seed)
    d = 128
    NB = sum(width * (-(-(p + steps + 1) // B)) for p in prompts) + 16
    mb = -(-(max(prompts) + steps + 1) // B)
    order = workloads.free_order(NB, 31 + B)
    kc = workloads.normal((NB, Hkv, B, d), dtype, 41, cuda_device)
    vc = workloads.normal((NB, Hkv, B, d), dtype, 42, cuda_device)
    ok, ov = oracle.bits16(kc), oracle.bits16(vc)
    eng = PagedKVCache(NB, Hkv, d, B, workloads.DTYPES[dtype], cuda_device, mb, order, key_cache=kc, value_cache=vc)
    ref = oracle.RefAllocator(NB, B, order)
    beams = [[eng.new_sequence(p)] for p in prompts]
    rbeams = [[ref.seq_new(p)] for p in prompts]
    nq = len(prompts) * width
    q = None
    for step in range(steps):
        plans = []
        for r in range(len(prompts)):
            par = workloads.beam_parents(rng, len(beams[r]), width)
            plans.append(par)
        new_all, slots, pairs, rslots, rpairs = [], [], [], [], []
        for r, par in enumerate(plans):
            n_, s_, p_ = eng.alloc.beam_step(beams[r], par)
            rn, rs, rp = ref.beam_step(rbeams[r], par)
            assert n_ == rn and s_.tolist() == rs and [tuple(x) for x in p_.tolist()] == rp
            beams[r], rbeams[r] = n_, rn
            new_all += n_
            slots.append(s_)
            pairs.append(p_)
        seqs = np.asarray(new_all, np.int32)
        tables, ctx = eng.alloc.build_block_tables(seqs, mb)
        from paged_kv_cache_139_gb300.engine import StepPlan
        plan = StepPlan(seqs, np.concatenate(slots), np.concatenate(pairs).reshape(-1, 2).astype(np.int32), tables, ctx)
        dev = eng.upload(plan)
        key = workloads.normal((nq, Hkv, d), dtype, 1000 + step, cuda_device)
        value = workloads.normal((nq, Hkv, d), dtype, 2000 + step, cuda_device)
        q = workloads.normal((nq, H, d), dtype, 3000 + step, cuda_device)
        out = eng.decode(q, key, value, dev)
        pkv.check()
        if len(plan.pairs):
            oracle.copy_blocks(ok, plan.pairs)
            oracle.copy_blocks(ov, plan.pairs)
        oracle.cache_write(key, value, ok, ov, plan.slots)
    assert np.array_equal(oracle.bits16(eng.key_cache), ok) and np.array_equal(oracle.bits16(eng.value_cache), ov)
    want = oracle.paged_attention(q, ok, ov, plan.tables, plan.context_lens, dtype)
    assert_close(out.double().cpu().numpy(), want, f"beam width {width} B={B}")
    # sharing is real: fewer blocks than every beam's own copy
    used = eng.alloc.blocks_in_use()
    unshared = sum(-(-eng.alloc.seq_len(int(b)) // B) for b in seqs)
    assert used < unshared


@pytest.mark.parametrize("width,B,dtype", [(4, 16, "f16"), (6, 4, "bf16"), (2, 32, "f16")])
def test_beam_search_steps(cuda_device, width, B, dtype):
    _beam_search(cuda_device, width, B, dtype, 8, 4, [37, 5, 130], 24, width * 100 + B)


def test_beam_search_bench_shapes(cuda_device):
    """The benchmark's beam workload shapes (OPT-13B layer, 40 x 128 MHA, f16, B=16, width 4,
    16 requests with its lognormal prompts), 32 steps."""
    w = workloads.beam(width=4)
    _beam_search(cuda_device, 4, 16, "f16", 40, 40, [int(p) for p in w.context_lens], 32, 7)
