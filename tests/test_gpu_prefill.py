"""paged_attention_prefill (and the prompt-phase cache write and
copy-on-write before it) against the oracle, through the C ABI.

Every case builds the batch twice (tests/prefill_cases.py): the allocator
plans are compared exactly, the K/V pools bit for bit (NaN-filled before the
writes, so that any read of an unwritten slot would show), and the
attention rows within the allclose tolerance of the decode tests."""
import numpy as np
import pytest
import torch

import paged_kv_cache_139_gb300 as pkv
import workloads
from prefill_cases import PrefillCase, assert_rows_close, custom

pytestmark = pytest.mark.gpu


def _check(c: PrefillCase, what: str, which=None, pools=True):
    c.check_allocator()
    if pools:
        kc, vc = c.oracle_caches()
        gk, gv = c.gpu_caches()
        assert np.array_equal(gk, kc) and np.array_equal(gv, vc), f"{what}: cache pools differ"
    T, H = c.q_dev.shape[0], c.w.num_heads
    if which is None:
        which = [(t, h) for t in range(T) for h in range(H)]
    want = c.oracle_out(which)
    got = c.out.double().cpu().numpy()
    assert_rows_close(got, want, which, what)


def test_plain_prompts(cuda_device):
    """Context = the new tokens: a plain causal prompt, across tile edges."""
    ctx = (1, 5, 127, 128, 129, 300, 700)
    _check(PrefillCase(custom(ctx, ctx, H=4, Hkv=4), cuda_device), "plain prompts")


def test_prompts_after_cached_tokens(cuda_device):
    ctx, new = (40, 300, 1030, 2000, 129), (40, 1, 200, 513, 2)
    _check(PrefillCase(custom(ctx, new, H=8, Hkv=2, d=64, B=8, dtype="bf16"), cuda_device), "after cached tokens")


def test_shared_prefix_small(cuda_device):
    """Five requests fork a 333-token prefix: each copies the prefix's partly
    filled last block on its first write."""
    w = custom([333 + n for n in (1, 17, 128, 255, 300)], (1, 17, 128, 255, 300), H=8, Hkv=2, dtype="bf16",
               prefix_len=333)
    c = PrefillCase(w, cuda_device)
    assert len(c.plan.pairs) == 5
    _check(c, "shared prefix")


def test_prefix_ending_on_a_block_boundary(cuda_device):
    """A 320-token prefix fills whole blocks: nothing is copied."""
    w = custom([320 + n for n in (3, 200)], (3, 200), prefix_len=320)
    c = PrefillCase(w, cuda_device)
    assert len(c.plan.pairs) == 0
    _check(c, "block-aligned prefix")


@pytest.mark.parametrize("B", [4, 8, 16, 32, 64, 128])
@pytest.mark.parametrize("d", [64, 128])
def test_block_and_head_sizes(cuda_device, B, d):
    w = custom((5, 130, 300, 1), (5, 100, 257, 1), H=2, Hkv=1, d=d, B=B, dtype="f16" if B % 8 else "bf16")
    _check(PrefillCase(w, cuda_device), f"B={B} d={d}")


@pytest.mark.parametrize("H,Hkv", [(4, 4), (4, 2), (8, 2), (12, 4), (7, 1), (6, 3)])
def test_head_groupings(cuda_device, H, Hkv):
    w = custom((200, 77, 129), (150, 77, 1), H=H, Hkv=Hkv, d=64, dtype="bf16")
    _check(PrefillCase(w, cuda_device), f"H={H} Hkv={Hkv}")


def test_sequences_without_new_tokens(cuda_device):
    w = custom((50, 10, 300, 7), (20, 0, 130, 0), H=4, Hkv=2)
    c = PrefillCase(w, cuda_device)
    _check(c, "empty sequences")


def test_single_new_token_matches_decode(cuda_device):
    """One new token per sequence is a decode step: the prompt-phase kernel
    and the decode kernel agree (and both match the oracle)."""
    ctx = (1, 33, 500, 1300)
    w = custom(ctx, (1, 1, 1, 1), H=8, Hkv=2, dtype="bf16")
    c = PrefillCase(w, cuda_device)
    _check(c, "single new token")
    dec = torch.empty_like(c.q_dev)
    pkv.paged_attention_decode(dec, c.q_dev, c.eng.key_cache, c.eng.value_cache, c.dev.tables,
                               c.dev.context_lens)
    pkv.check()
    err = (dec.double() - c.out.double()).abs().max().item()
    assert err < 4e-3, err


def test_unwritten_slots_never_weigh(cuda_device):
    """NaN-filled and zero-filled pools give bit-identical outputs."""
    w = custom((29, 250, 1001), (29, 250, 130), H=4, Hkv=2, B=16)
    a = PrefillCase(w, cuda_device, nan_pool=True)
    b = PrefillCase(w, cuda_device, nan_pool=False)
    assert torch.isfinite(a.out.float()).all()
    assert torch.equal(a.out, b.out)


def test_placement_invariance(cuda_device):
    """The same logical blocks at other physical blocks: bit-identical rows."""
    w = custom((400, 130, 900), (400, 64, 300), H=4, Hkv=4, B=16)
    a = PrefillCase(w, cuda_device)
    rev = workloads.free_order(w.num_blocks, w.seed)[::-1].copy()
    b = PrefillCase(w, cuda_device, order=rev)
    assert not np.array_equal(a.plan.tables, b.plan.tables)
    assert torch.equal(a.out, b.out)


def test_repeated_calls_are_identical(cuda_device):
    w = custom((700, 260), (700, 130), H=4, Hkv=2)
    c = PrefillCase(w, cuda_device)
    outs = [c.rerun() for _ in range(3)]
    assert all(torch.equal(c.out, o) for o in outs)


def test_prefix_workload_full_sampled(cuda_device):
    """The 32-request shared-prefix workload (Llama-2-7B layer shapes) in the
    launch the benchmark times: sampled rows against the oracle."""
    c = PrefillCase(workloads.prefix(), cuda_device)
    assert len(c.plan.pairs) == 32
    _check(c, "prefix workload", which=c.sample_rows(n_per_seq=4))


def test_prefix_workload_gqa_bf16_sampled(cuda_device):
    c = PrefillCase(workloads.prefix(num_kv_heads=8, dtype="bf16", num_requests=16, prefix_len=2050,
                                     max_own=1024), cuda_device)
    _check(c, "prefix workload gqa", which=c.sample_rows(n_per_seq=4))


def test_bad_context_is_latched(cuda_device):
    """More new tokens than context: PKV_EINDEX, rows unwritten, and the next
    call works."""
    w = custom((300, 40), (300, 40), H=2, Hkv=2)
    c = PrefillCase(w, cuda_device)
    bad_ctx = c.dev.context_lens.clone()
    bad_ctx[1] = 10                                   # 40 new tokens, context 10
    o = torch.full_like(c.q_dev, 7.0)
    pkv.paged_attention_prefill(o, c.q_dev, c.eng.key_cache, c.eng.value_cache, c.dev.tables, bad_ctx,
                                c.dev.query_start, max_query_len=300)
    with pytest.raises(pkv.PkvError) as e:
        pkv.check()
    assert e.value.status == 3                        # PKV_EINDEX
    assert (o[300:] == 7.0).all()
    assert torch.equal(c.rerun(), c.out)


def test_bad_block_is_latched(cuda_device):
    w = custom((100,), (100,), H=2, Hkv=2)
    c = PrefillCase(w, cuda_device)
    t = c.dev.tables.clone()
    t[0, 2] = w.num_blocks + 5
    o = torch.empty_like(c.q_dev)
    pkv.paged_attention_prefill(o, c.q_dev, c.eng.key_cache, c.eng.value_cache, t, c.dev.context_lens,
                                c.dev.query_start)
    with pytest.raises(pkv.PkvError) as e:
        pkv.check()
    assert e.value.status == 3
    assert torch.equal(c.rerun(), c.out)


def test_max_query_len_bounds_the_rows(cuda_device):
    """max_query_len bounds the work items: rows of a sequence past the tile
    pairs it covers (256 rows each) are left untouched, the rest are computed."""
    w = custom((300,), (300,), H=2, Hkv=2)
    c = PrefillCase(w, cuda_device)
    o = torch.full_like(c.q_dev, 5.0)
    c.rerun(out=o, max_query_len=100)
    assert torch.equal(o[:256], c.out[:256])
    assert (o[256:] == 5.0).all()


def _prefill_abi(c: PrefillCase, out, workspace, nbytes):
    """paged_attention_prefill through the C ABI with an explicit workspace
    pointer (None: the static share per CTA)."""
    from paged_kv_cache_139_gb300 import _lib
    w = c.w
    rc = _lib.load().paged_attention_prefill(
        out.data_ptr(), c.q_dev.data_ptr(), c.eng.key_cache.data_ptr(), c.eng.value_cache.data_ptr(),
        c.dev.tables.data_ptr(), c.dev.context_lens.data_ptr(), c.dev.query_start.data_ptr(), w.num_seqs,
        c.q_dev.shape[0], c.dev.max_query_len, c.dev.tables.shape[1], w.block_size, w.num_blocks, w.num_heads,
        w.num_kv_heads, w.head_dim, float(1.0 / np.sqrt(w.head_dim)), workspace, nbytes,
        1 if w.dtype == "bf16" else 0, torch.cuda.current_stream().cuda_stream)
    assert rc == 0, _lib.load().pkv_last_error_string()


def _many_items(seed, S=16, H=32, Hkv=8, d=64, dtype="bf16"):
    """Several hundred work items (pairs of 128-row tiles x heads x
    sequences) over the GPU's SMs: every CTA runs several, of different
    lengths, one- and two-tile, with the item order mixing sequences."""
    rng = np.random.default_rng(seed)
    new = rng.integers(1, 420, size=S)
    cached = rng.integers(0, 200, size=S)
    return custom(new + cached, new, H=H, Hkv=Hkv, d=d, dtype=dtype, seed=seed)


def _item_rows(c: PrefillCase, seed=0):
    """(token, head) rows covering every work item: per (sequence, head, pair
    of tiles) the first and last row of each tile and one between."""
    rng = np.random.default_rng(seed)
    which = []
    for s in range(c.w.num_seqs):
        a, b = int(c.query_start[s]), int(c.query_start[s + 1])
        for t0 in range(0, b - a, 256):
            for h in range(c.w.num_heads):
                for lo in (t0, t0 + 128):
                    hi = min(lo + 128, b - a)
                    if lo >= hi:
                        continue
                    which += [(a + lo, h), (a + hi - 1, h), (a + int(rng.integers(lo, hi)), h)]
    return sorted(set(which))


@pytest.mark.parametrize("seed,S,H,Hkv,d,dtype", [(11, 16, 32, 8, 64, "bf16"), (12, 24, 24, 24, 128, "f16"),
                                                   (13, 12, 48, 8, 128, "bf16")])
def test_many_items_per_cta(cuda_device, seed, S, H, Hkv, d, dtype):
    """Rows of every work item of a batch whose items outnumber the CTAs
    several times, against the oracle (pools bit for bit); the static round
    robin (no workspace) gives the same bits as the counter."""
    c = PrefillCase(_many_items(seed, S=S, H=H, Hkv=Hkv, d=d, dtype=dtype), cuda_device)
    items = sum(-(-int(n) // 256) for n in c.w.query_lens) * H
    assert items > 3 * torch.cuda.get_device_properties(0).multi_processor_count
    _check(c, f"many items {seed}", which=_item_rows(c, seed))
    o = torch.full_like(c.q_dev, 3.0)
    _prefill_abi(c, o, None, 0)
    pkv.check()
    assert torch.equal(o, c.out)


def test_workspace_counter_left_ready(cuda_device):
    """After a call the workspace's ticket counters are back at zero (magic
    kept), so back-to-back calls and graph replays start from ticket 0."""
    c = PrefillCase(_many_items(21), cuda_device)
    ws = pkv.make_workspace(cuda_device, 256)
    before = ws[:16].clone()
    for _ in range(3):
        o = torch.empty_like(c.q_dev)
        _prefill_abi(c, o, ws.data_ptr(), ws.numel())
        pkv.check()
        assert torch.equal(o, c.out)
    torch.cuda.synchronize()
    assert torch.equal(ws[:16], before)
    assert int(ws[:8].view(torch.int32)[0]) == 0 and int(ws[:8].view(torch.int32)[1]) == 0


def test_unprepared_workspace_is_refused(cuda_device):
    """A workspace that paged_attention_workspace_init never prepared:
    PKV_EINVAL from pkv_check, no row written, and the next call works."""
    c = PrefillCase(custom((300, 40), (300, 40), H=2, Hkv=2), cuda_device)
    raw = torch.zeros(256, dtype=torch.uint8, device=cuda_device)
    o = torch.full_like(c.q_dev, 7.0)
    _prefill_abi(c, o, raw.data_ptr(), raw.numel())
    with pytest.raises(pkv.PkvError) as e:
        pkv.check()
    assert e.value.status == 1
    assert (o == 7.0).all()
    assert torch.equal(c.rerun(), c.out)


@pytest.mark.parametrize("dtype,H,Hkv", [("f16", 4, 4), ("bf16", 8, 2), ("bf16", 6, 2), ("bf16", 3, 3)])
def test_one_tile_items_split_over_both_groups(cuda_device, dtype, H, Hkv):
    """Items with one query tile and two or more key tiles give their key tiles
    alternately to both softmax groups and merge the two outputs.  The
    contexts cover 2 to 8 key tiles, a last key tile ending mid-tile on
    either group (its rows past the context zeroed by that group), rows that
    see no key of the second group's first tile (positions below 128: their
    scores there are all -inf), and the one-tile remainder after a pair of
    tiles.  An even number of query heads per kv head pairs heads instead
    (no one-tile items), so bf16 is also run with groups of 3 and 1."""
    ctx = (200, 259, 484, 1000, 130, 900)
    new = (128, 5, 50, 1, 2, 300)
    _check(PrefillCase(custom(ctx, new, H=H, Hkv=Hkv, dtype=dtype), cuda_device), f"split items {dtype}")


@pytest.mark.parametrize("seed", range(8))
def test_seeded_random_batches(cuda_device, seed):
    """Seeded random prompt-phase batches: 1-7 sequences, 0-600 new tokens
    after 0-1500 cached ones, head dim 64 or 128, block size 4-128, MHA or
    grouped heads, fp16 or bf16 -- pair, split and one-key-tile items mixed in
    one launch, against the oracle."""
    rng = np.random.default_rng(9000 + seed)
    S = int(rng.integers(1, 8))
    new = rng.integers(0, 601, size=S)
    ctx = new + rng.integers(0, 1501, size=S)
    ctx = np.maximum(ctx, 1)
    new = np.minimum(new, ctx)
    d = int(rng.choice([64, 128]))
    B = int(rng.choice([4, 8, 16, 32, 64, 128]))
    Hkv = int(rng.choice([1, 2, 4]))
    H = Hkv * int(rng.choice([1, 2, 4]))
    dtype = str(rng.choice(["f16", "bf16"]))
    w = custom(tuple(int(c) for c in ctx), tuple(int(n) for n in new), H=H, Hkv=Hkv, d=d, B=B, dtype=dtype,
               seed=700 + seed)
    _check(PrefillCase(w, cuda_device), f"random batch {seed}: S={S} d={d} B={B} H={H}/{Hkv} {dtype}")
