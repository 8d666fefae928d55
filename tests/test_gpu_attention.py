"""paged_attention_decode against the oracle on the GPU through the C ABI:
every workload (small sizes in full, full sizes on sampled sequences and
heads), the split-context path, GQA groupings, block sizes, head sizes, and
the degenerate cases."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_139_gb300 as pkv
import workloads
from cases import Case, assert_close

pytestmark = pytest.mark.gpu


def _check(c: Case, heads=None, what=""):
    c.check_allocator()
    want = c.oracle_out(heads)
    got = c.gpu_out()
    if heads is not None:
        rows = tuple(np.array(heads).T)
        got, want = got[rows], want[rows]
    return assert_close(got, want, what)


def _custom(name="custom", S=3, H=4, Hkv=2, d=128, B=16, dtype="f16", ctx=(1, 40, 333), max_ctx=None,
            seed=77, partition=0):
    ctx = np.asarray(ctx, np.int64)
    mc = int(max_ctx or max(int(ctx.max()), 1))
    mb = -(-mc // B)
    nb = int(sum(-(-int(c) // B) for c in ctx)) + 5
    return workloads.Workload(name, S, H, Hkv, d, B, dtype, ctx, mb, nb, seed, partition)


def _head_sample(w, k):
    """A seeded choice of k kv heads of the workload (the parity sample of a
    full-size batch)."""
    return sorted(np.random.default_rng(w.seed).choice(w.num_kv_heads, k, replace=False).tolist())


def test_tiny_workload(cuda_device):
    c = Case(workloads.tiny(), cuda_device)
    _check(c, what="tiny")
    k, v = c.gpu_cache_blocks()
    ok, ov = c.oracle_caches()
    assert np.array_equal(k, ok) and np.array_equal(v, ov)


def test_opt13b_small(cuda_device):
    _check(Case(workloads.opt13b(num_seqs=8), cuda_device), what="opt13b x8")


def test_opt13b_full(cuda_device):
    """The 64-sequence OPT-13B layer batch in full, in the default launch."""
    _check(Case(workloads.opt13b(), cuda_device), what="opt13b")


@pytest.mark.parametrize("B", [8, 16, 32])
def test_llama7b_small(cuda_device, B):
    _check(Case(workloads.llama7b(block_size=B, num_seqs=12, max_ctx=1500), cuda_device), what=f"llama7b B={B}")


@pytest.mark.parametrize("S,P", [(16, 1024), (4, 512)])
def test_default_partition_d64_halves(cuda_device, S, P):
    """At head_dim 64 the default partition starts at 2048 and halves while
    fewer than 2048 work items would remain: 16 sequences x 32 heads take
    1024, 4 take 512; both match the oracle."""
    w = workloads.llama7b(block_size=16, head_dim=64, num_seqs=S)
    mcl = int(w.context_lens.max())
    assert pkv.paged_attention_partition_size(S, 32, 32, 64, mcl, 0) == P
    c = Case(w, cuda_device, gen_device="cuda", subset=list(range(min(S, 4))))
    _check(c, what=f"llama7b d=64 S={S}")


@pytest.mark.parametrize("B,d", [(8, 128), (16, 128), (32, 128),
                                 # the block-size study: small and large blocks, small heads
                                 (4, 128), (128, 128), (4, 64), (16, 64), (64, 64), (128, 64)])
def test_llama7b_full_sampled(cuda_device, B, d):
    """The full 256 x uniform[1,4096] batch in the default launch: every
    sequence, on a seeded sample of 4 of the 32 heads."""
    w = workloads.llama7b(block_size=B, head_dim=d)
    c = Case(w, cuda_device, gen_device="cuda", kv_heads=_head_sample(w, 4))
    _check(c, what=f"llama7b full B={B} d={d}")


def test_sampling_small(cuda_device):
    _check(Case(workloads.sampling(num_prompts=6, max_suffix=60), cuda_device), what="sampling x6")


def test_sampling_full_sampled(cuda_device):
    """The full 64 prompts x 4 samples batch (copy-on-write of the shared last
    blocks, suffixes, decode step): every sequence, 4 sampled heads."""
    w = workloads.sampling()
    c = Case(w, cuda_device, kv_heads=_head_sample(w, 4))
    _check(c, what="sampling full")


def test_longgqa_small(cuda_device):
    _check(Case(workloads.longgqa(num_seqs=2, ctx_len=4096), cuda_device), what="longgqa small")


def test_longgqa_full_sampled(cuda_device):
    """8 x 32768 tokens, bf16, GQA 32/8, partitions of 512: every sequence, on
    the 8 query heads of 2 sampled kv heads."""
    w = workloads.longgqa()
    c = Case(w, cuda_device, gen_device="cuda", kv_heads=_head_sample(w, 2))
    _check(c, what="longgqa full")


@pytest.mark.parametrize("H,Hkv", [(4, 4), (4, 2), (8, 2), (12, 4), (16, 2), (10, 2), (6, 6), (7, 1)])
def test_head_groupings(cuda_device, H, Hkv):
    w = _custom(H=H, Hkv=Hkv, ctx=(1, 17, 200, 513, 1030), S=5, dtype="bf16")
    c = Case(w, cuda_device, partition_size=256)
    _check(c, what=f"H={H} Hkv={Hkv}")


@pytest.mark.parametrize("B", [4, 8, 16, 32, 64, 128])
@pytest.mark.parametrize("d", [64, 128])
def test_block_and_head_sizes(cuda_device, B, d):
    w = _custom(d=d, B=B, ctx=(1, 3, 31, 32, 33, 64, 127, 500, 1027), S=9, dtype="f16" if B % 8 else "bf16")
    for P in (0, 32, 128):
        c = Case(w, cuda_device, partition_size=P)
        _check(c, what=f"B={B} d={d} P={P}")


@pytest.mark.parametrize("P", [32, 64, 96, 512, 4096])
def test_partition_sizes_agree(cuda_device, P):
    """Split and unsplit runs of the same batch both match the oracle."""
    w = _custom(H=8, Hkv=2, ctx=(5, 511, 512, 513, 2048, 3001), S=6, max_ctx=4096)
    c = Case(w, cuda_device, partition_size=P)
    _check(c, what=f"P={P}")


@pytest.mark.parametrize("H,Hkv,d,dtype", [(8, 2, 128, "f16"), (32, 8, 128, "bf16"), (4, 4, 64, "f16"),
                                         (16, 2, 64, "bf16")])
def test_merge_kernel_chunks(cuda_device, H, Hkv, d, dtype):
    """Splits into 1, 16, 17, 24, 25, 64, 65, 255 and 256 partitions of 32
    tokens, merged by partition_reduce_kernel in chunks of 64 (head_dim 128)
    or 128 (head_dim 64) partitions, against the oracle; a second call is
    bit-identical."""
    w = _custom(H=H, Hkv=Hkv, d=d, dtype=dtype, ctx=(1, 512, 520, 768, 790, 2048, 2050, 8150, 8192), S=9)
    c = Case(w, cuda_device, partition_size=32)
    before = pkv.launch_count()
    again = c.rerun_attention().clone()
    assert pkv.launch_count() - before == 2
    assert torch.equal(again, c.out)
    _check(c, what=f"merge kernel H={H} Hkv={Hkv} d={d}")


def test_context_zero_and_one(cuda_device):
    w = _custom(ctx=(1, 2, 1, 40), S=4)
    c = Case(w, cuda_device)
    _check(c, what="short")
    # ctx = 1 returns the single value exactly up to output rounding
    v = c.eng.value_cache[int(c.plan.tables[0, 0]), 0, 0].double().cpu().numpy()
    assert np.array_equal(c.gpu_out()[0, 0], v)
    # ctx = 0: zeros
    ctx0 = torch.zeros_like(c.dev.context_lens)
    step = dataclasses.replace(c.dev, context_lens=ctx0)
    out = c.eng.attend(c.q_dev, step, max_context_len=32)
    pkv.check()
    assert int(out.abs().sum().item()) == 0


def test_permutation_invariance_bit_exact(cuda_device):
    """Moving the blocks to other physical ids changes no output bit."""
    w = _custom(H=8, Hkv=2, ctx=(100, 700, 1500), S=3, dtype="bf16")
    c = Case(w, cuda_device, partition_size=256)
    out1 = c.out.clone()
    perm = torch.randperm(w.num_blocks, generator=torch.Generator().manual_seed(5)).to(cuda_device)
    kc2 = torch.empty_like(c.eng.key_cache)
    vc2 = torch.empty_like(c.eng.value_cache)
    kc2[perm] = c.eng.key_cache
    vc2[perm] = c.eng.value_cache
    t = c.dev.tables.long()
    t2 = torch.where(t >= 0, perm[t.clamp(min=0)], t).to(torch.int32)
    out2 = torch.empty_like(out1)
    pkv.paged_attention_decode(out2, c.q_dev, kc2, vc2, t2, c.dev.context_lens, partition_size=256)
    pkv.check()
    assert torch.equal(out1, out2)


def test_identity_table_equals_contiguous_oracle(cuda_device):
    """With the identity table (each sequence's blocks adjacent) the kernel
    equals the oracle, which here is plain contiguous attention."""
    S, H, d, B, mb = 4, 4, 128, 16, 40
    q = workloads.normal((S, H, d), "f16", 1).to(cuda_device)
    kc = workloads.normal((S * mb, H, B, d), "f16", 2).to(cuda_device)
    vc = workloads.normal((S * mb, H, B, d), "f16", 3).to(cuda_device)
    tables = torch.arange(S * mb, dtype=torch.int32, device=cuda_device).view(S, mb)
    ctx = torch.tensor([640, 1, 77, 500], dtype=torch.int32, device=cuda_device)
    out = torch.empty_like(q)
    pkv.paged_attention_decode(out, q, kc, vc, tables, ctx)
    pkv.check()
    want = oracle.paged_attention(q.cpu(), kc.cpu(), vc.cpu(), tables.cpu().numpy(), ctx.cpu().numpy(), "f16")
    assert_close(out.double().cpu().numpy(), want, "identity table")


def test_bad_block_id_latches_eindex(cuda_device):
    w = _custom(ctx=(50, 90), S=2)
    c = Case(w, cuda_device)
    pkv.check()
    t = c.dev.tables.clone()
    t[1, 2] = w.num_blocks + 3
    pkv.paged_attention_decode(torch.empty_like(c.q_dev), c.q_dev, c.eng.key_cache, c.eng.value_cache, t,
                               c.dev.context_lens)
    with pytest.raises(pkv.PkvError) as e:
        pkv.check()
    assert e.value.status_name == "PKV_EINDEX" and "block" in str(e.value)
    pkv.check()                                          # cleared


def test_context_beyond_bound_latches_eindex(cuda_device):
    w = _custom(ctx=(50, 90), S=2)
    c = Case(w, cuda_device)
    pkv.paged_attention_decode(torch.empty_like(c.q_dev), c.q_dev, c.eng.key_cache, c.eng.value_cache,
                               c.dev.tables, c.dev.context_lens, max_context_len=64)
    with pytest.raises(pkv.PkvError) as e:
        pkv.check()
    assert e.value.status_name == "PKV_EINDEX" and "context" in str(e.value)


def test_uninitialised_workspace_is_reported(cuda_device):
    w = _custom(ctx=(50, 90), S=2)
    c = Case(w, cuda_device)
    ws = torch.zeros(4096, dtype=torch.uint8, device=cuda_device)          # never initialised
    out = torch.full_like(c.q_dev, 3.0)
    pkv.paged_attention_decode(out, c.q_dev, c.eng.key_cache, c.eng.value_cache, c.dev.tables,
                               c.dev.context_lens, workspace=ws)
    with pytest.raises(pkv.PkvError) as e:
        pkv.check()
    assert e.value.status_name == "PKV_EINVAL" and "workspace" in str(e.value)
    assert bool((out == 3.0).all())                                          # nothing was written


@pytest.mark.parametrize("P", [128, 32])
def test_repeated_calls_reuse_the_workspace(cuda_device, P):
    """The ticket and partition counters reset themselves: many calls on one
    workspace give identical results (fused merge at P=128, merge kernel at
    P=32)."""
    w = _custom(H=8, Hkv=2, ctx=(5, 900, 1500, 31), S=4)
    c = Case(w, cuda_device, partition_size=P)
    outs = [c.rerun_attention().clone() for _ in range(5)]
    assert all(torch.equal(outs[0], o) for o in outs[1:]) and torch.equal(outs[0], c.out)
    _check(c, what=f"repeat P={P}")


def test_bounded_wait_times_out_and_context_survives(cuda_device):
    L = pkv._lib.load()
    import ctypes
    s = torch.cuda.current_stream()
    assert L.pkv_selftest_wait_timeout(1 << 20, ctypes.c_void_p(s.cuda_stream)) == 0
    with pytest.raises(pkv.PkvError) as e:
        pkv.check()
    assert e.value.status_name == "PKV_ETIMEOUT"
    # the context is still usable
    test_tiny_workload(cuda_device)


def test_output_guard_bytes(cuda_device):
    """Nothing outside out[S][H][d] is written."""
    w = _custom(H=8, Hkv=2, ctx=(33, 1000), S=2)
    c = Case(w, cuda_device, partition_size=128)
    n = c.q_dev.numel()
    buf = torch.full((n + 2048,), 7.0, dtype=c.q_dev.dtype, device=cuda_device)
    out = buf[1024:1024 + n].view_as(c.q_dev)
    c.rerun_attention(out=out)
    pkv.check()
    assert bool((buf[:1024] == 7).all()) and bool((buf[1024 + n:] == 7).all())
    assert torch.equal(out, c.out)


def test_launch_count_and_native_library(cuda_device):
    c = Case(_custom(ctx=(600, 700), S=2, H=4, Hkv=4), cuda_device, partition_size=256)
    before = pkv.launch_count()
    c.eng.decode(c.q_dev, c.k_dev, c.v_dev, c.dev, partition_size=256)
    pkv.check()
    # cache write + attention; three partitions per sequence merge inside the
    # attention kernel (the workspace exists already)
    assert pkv.launch_count() - before == 2
    # a split into more than 16 partitions adds the merge kernel (the first
    # such call also grows and prepares the workspace)
    c.eng.attend(c.q_dev, c.dev, partition_size=32)
    before = pkv.launch_count()
    c.eng.decode(c.q_dev, c.k_dev, c.v_dev, c.dev, partition_size=32)
    pkv.check()
    assert pkv.launch_count() - before == 3
    import os
    maps = open("/proc/self/maps").read()
    assert os.path.realpath(pkv.library_path()) in maps


def test_prepared_step_matches_decode(cuda_device):
    """The prepared decode step (arguments marshalled once) launches the same
    calls as the engine's decode."""
    w = _custom(H=8, Hkv=4, ctx=(300, 1, 1200), S=3)
    c = Case(w, cuda_device, partition_size=256)
    out = torch.empty_like(c.q_dev)
    # the write rides in the attention launch (one launch, the merge fused too) ...
    prep = c.eng.prepare(c.q_dev, c.k_dev, c.v_dev, c.dev, out, partition_size=256)
    before = pkv.launch_count()
    prep()
    pkv.check()
    assert pkv.launch_count() - before == 1
    assert torch.equal(out, c.out)
    # ... or takes its own launch
    out2 = torch.empty_like(c.q_dev)
    prep2 = c.eng.prepare(c.q_dev, c.k_dev, c.v_dev, c.dev, out2, partition_size=256, fused=False)
    before = pkv.launch_count()
    prep2()
    pkv.check()
    assert pkv.launch_count() - before == 2
    assert torch.equal(out2, c.out)


def test_staged_inputs_single_upload(cuda_device):
    """A decode step whose inputs arrive through one pinned staging buffer (one
    host-to-device copy) gives the same output as separately uploaded ones."""
    from paged_kv_cache_139_gb300.engine import StagedInputs
    w = _custom(H=8, Hkv=2, ctx=(5, 300, 1000, 77), S=4)
    c = Case(w, cuda_device)
    plan, eng = c.plan, c.eng
    src = {"q": c.query, "key": c.key, "value": c.value, "slots": torch.from_numpy(plan.slots),
           "tables": torch.from_numpy(plan.tables), "ctx": torch.from_numpy(plan.context_lens)}
    stg = StagedInputs({n: (tuple(x.shape), x.dtype) for n, x in src.items()}, cuda_device)
    assert all(stg.dev[n].data_ptr() % 256 == 0 for n in src)
    for n, x in src.items():
        stg.host[n].copy_(x)
    stg.upload()
    torch.cuda.synchronize()
    for n, x in src.items():
        assert torch.equal(stg.dev[n].cpu(), x.cpu())
    d = stg.dev
    step = type(c.dev)(d["slots"], c.dev.pairs, d["tables"], d["ctx"], c.dev.max_context_len)
    out = eng.attend(d["q"], step)
    pkv.check()
    assert torch.equal(out, c.out)


def test_graph_step_replays_the_step(cuda_device):
    """The staged upload, decode calls and read-back captured in one CUDA graph:
    replays with new host inputs give the same output as direct calls."""
    from paged_kv_cache_139_gb300.engine import GraphStep, StagedInputs
    w = _custom(H=8, Hkv=2, ctx=(5, 300, 1000, 77), S=4)
    c = Case(w, cuda_device)
    plan, eng = c.plan, c.eng
    src = {"q": c.query, "key": c.key, "value": c.value, "slots": torch.from_numpy(plan.slots),
           "tables": torch.from_numpy(plan.tables), "ctx": torch.from_numpy(plan.context_lens)}
    stg = StagedInputs({n: (tuple(x.shape), x.dtype) for n, x in src.items()}, cuda_device)
    for n, x in src.items():
        stg.host[n].copy_(x)
    d = stg.dev
    step = type(c.dev)(d["slots"], c.dev.pairs, d["tables"], d["ctx"], c.dev.max_context_len)
    out = torch.empty_like(c.out)
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    g = GraphStep(stg, lambda st: eng.prepare(d["q"], d["key"], d["value"], step, out, stream=st), out, h_out)
    for rep in range(3):
        q2 = workloads.normal(tuple(c.query.shape), w.dtype, 900 + rep)
        stg.host["q"].copy_(q2)
        g.replay()
        torch.cuda.synchronize()
        pkv.check()
        want = eng.attend(q2.to(cuda_device), c.dev)
        pkv.check()
        assert torch.equal(h_out.to(cuda_device), want)


@pytest.mark.parametrize("name,kw", [
    ("tiny", {}), ("opt13b", {}), ("longgqa", dict(num_seqs=2, ctx_len=3000)),
    ("sampling", dict(num_prompts=4, max_suffix=40)),
    ("gqa8", dict(H=16, Hkv=2)), ("gqa4_bf16", dict(H=8, Hkv=2, dtype="bf16")), ("b4_d64", dict(B=4, d=64)),
    ("b128", dict(B=128)),
])
def test_fused_write_matches_separate_calls(cuda_device, name, kw):
    """paged_attention_decode_write (the new tokens written inside the attention
    launch) leaves the caches bit-identical to kv_reshape_and_cache followed by
    paged_attention_decode, gives the same output bit for bit, and matches the
    oracle."""
    if name in ("tiny", "opt13b", "longgqa", "sampling"):
        w = workloads.by_name(name, **kw)
    else:
        base = dict(ctx=(1, 17, 200, 513, 1030), S=5)
        base.update(kw)
        w = _custom(**base)
    sep = Case(w, cuda_device)
    fus = Case(w, cuda_device, fused=True)
    assert torch.equal(sep.eng.key_cache, fus.eng.key_cache) and torch.equal(sep.eng.value_cache, fus.eng.value_cache)
    assert torch.equal(sep.out, fus.out)
    _check(fus, what=f"fused {name}")


def test_fused_write_bad_slot_latches_eindex(cuda_device):
    w = _custom(H=4, Hkv=2, ctx=(5, 40, 300), S=3)
    c = Case(w, cuda_device)
    slots = c.dev.slots.clone()
    slots[1] = w.num_blocks * w.block_size + 3
    out = torch.empty_like(c.q_dev)
    pkv.paged_attention_decode_write(out, c.q_dev, c.k_dev, c.v_dev, c.eng.key_cache, c.eng.value_cache, slots,
                                     c.dev.tables, c.dev.context_lens)
    with pytest.raises(pkv.PkvError) as e:
        pkv.check()
    assert e.value.status == 3


@pytest.mark.parametrize("where", ["other_partition", "other_sequence", "wrong_offset"])
def test_fused_write_slot_contract_latched(cuda_device, where):
    """paged_attention_decode_write only writes a slot that is position
    context_len - 1 of the sequence's own table (no other work item of the
    launch reads it).  A slot elsewhere -- in an earlier partition, in another
    sequence's block, or at another offset of the right block -- is latched as
    PKV_EINDEX and not written."""
    w = _custom(H=4, Hkv=2, ctx=(5, 40, 1300), S=3)
    c = Case(w, cuda_device, partition_size=256)
    B = w.block_size
    tables, ctx = c.plan.tables, c.plan.context_lens
    s = 2
    if where == "other_partition":
        bad = int(tables[s][0]) * B + 3                   # position 3: partition 0 of 6
    elif where == "other_sequence":
        bad = int(tables[1][1]) * B + 7                   # sequence 1's second block
    else:
        last = int(ctx[s]) - 1
        bad = int(tables[s][last // B]) * B + (last + 1) % B
    slots = c.dev.slots.clone()
    slots[s] = bad
    kc0, vc0 = c.eng.key_cache.clone(), c.eng.value_cache.clone()
    out = torch.empty_like(c.q_dev)
    pkv.paged_attention_decode_write(out, c.q_dev, c.k_dev, c.v_dev, c.eng.key_cache, c.eng.value_cache, slots,
                                     c.dev.tables, c.dev.context_lens, partition_size=256)
    with pytest.raises(pkv.PkvError) as e:
        pkv.check()
    assert e.value.status == 3
    assert "context_len - 1" in pkv._lib.load().pkv_last_error_string().decode()
    bb = bad // B
    assert torch.equal(c.eng.key_cache[bb], kc0[bb]) and torch.equal(c.eng.value_cache[bb], vc0[bb])


def _rand_batch(dev, S, H, Hkv, d, B, ctx, dtype, seed):
    ctx = np.asarray(ctx, np.int32)
    mb = int(-(-int(ctx.max()) // B))
    nb = S * mb
    q = workloads.normal((S, H, d), dtype, seed).to(dev)
    kc = workloads.normal((nb, Hkv, B, d), dtype, seed + 1).to(dev)
    vc = workloads.normal((nb, Hkv, B, d), dtype, seed + 2).to(dev)
    perm = np.random.default_rng(seed).permutation(nb).astype(np.int32).reshape(S, mb)
    return q, kc, vc, torch.from_numpy(perm).to(dev), torch.from_numpy(ctx).to(dev)


def test_workspace_shared_by_calls_of_different_sizes(cuda_device):
    """One workspace serving calls of different sizes: the second call's merge
    counters sit where the first call left partials, so the library zeroes
    them when the sizes change.  Every call matches the same call on a fresh
    workspace bit for bit, in both orders and again."""
    a = _rand_batch(cuda_device, 4, 8, 8, 128, 16, [4000, 4096, 3900, 4050], "f16", 41)    # 16 partitions of 256
    b = _rand_batch(cuda_device, 2, 8, 8, 128, 16, [1000, 900], "f16", 43)                 # 4 partitions of 256

    def need(x):
        q, kc, vc, bt, cl = x
        return pkv.paged_attention_workspace_size(q.shape[0], q.shape[1], kc.shape[1], q.shape[2],
                                                  bt.shape[1] * kc.shape[2], 256)

    def run(x, ws):
        q, kc, vc, bt, cl = x
        out = torch.full_like(q, float("nan"))
        pkv.paged_attention_decode(out, q, kc, vc, bt, cl, partition_size=256, workspace=ws)
        pkv.check()
        return out

    want_a = run(a, pkv.make_workspace(cuda_device, need(a)))
    want_b = run(b, pkv.make_workspace(cuda_device, need(b)))
    ws = pkv.make_workspace(cuda_device, max(need(a), need(b)))
    for x, want in [(a, want_a), (b, want_b), (a, want_a), (a, want_a), (b, want_b)]:
        assert torch.equal(run(x, ws), want)
