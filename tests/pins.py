"""Checks that pin the oracle to facts other than itself.

Each pin is a function that raises AssertionError when the oracle disagrees
with the pages' worked examples, a closed form, an invariant, or a library
routine.  tests/test_oracle_pins.py runs them against the oracle;
tests/test_oracle_mutations.py runs them against copies of the oracle with a
planted mistake and requires each mistake to be caught.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch
import torch.nn.functional as F

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def golden(name: str) -> dict:
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _rand16(shape, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g).to(dtype)


def _pool(NB, Hkv, B, d, dtype, seed):
    return oracle.bits16(_rand16((NB, Hkv, B, d), dtype, seed))


# -- decoding of the 16-bit formats ---------------------------------------------

def pin_decode_f16_all_patterns():
    """Every binary16 pattern decodes as numpy's float16 -> float64."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = oracle.decode16(bits, "f16")
    want = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


def pin_decode_bf16_all_patterns():
    """Every bfloat16 pattern decodes as torch's bfloat16 -> float64."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    want = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.decode16(bits, "bf16")
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


# -- block-table gather --------------------------------------------------------

def pin_block_ranges_worked_example():
    """i = 40, B = 16 visits 3 blocks: tokens 1-16, 17-32, 33-40."""
    g = golden("block_ranges_40_16.json")
    i, B = g["query_position"], g["block_size"]
    phys, off = oracle.locate_tokens([0, 1, 2], B, i)
    assert len(set(phys.tolist())) == g["blocks_visited"]
    ranges = []
    for blk in sorted(set(phys.tolist())):
        toks = np.nonzero(phys == blk)[0] + 1          # 1-based positions
        ranges.append([int(toks.min()), int(toks.max())])
        assert np.array_equal(off[phys == blk], np.arange(len(toks)))
    assert ranges == g["token_ranges_1_based"]


def pin_locate_request_flow():
    """Figure 6: the 8th and 9th tokens of the 7-token prompt's sequence land
    in physical block 1 offset 3, then physical block 3 offset 0."""
    phys, off = oracle.locate_tokens([7, 1, 3], 4, 9)
    assert (phys[7], off[7]) == (1, 3)
    assert (phys[8], off[8]) == (3, 0)
    assert phys[:4].tolist() == [7] * 4 and phys[4:8].tolist() == [1] * 4


# -- cache write -----------------------------------------------------------------

def pin_cache_write_slot_example():
    """Slot 12 with B = 4 is block 3, offset 0 (Figure 6, second decode step);
    nothing else in either cache changes, and a negative slot is skipped."""
    NB, Hkv, B, d = 6, 2, 4, 8
    kc0 = _pool(NB, Hkv, B, d, torch.float16, 1)
    vc0 = _pool(NB, Hkv, B, d, torch.float16, 2)
    kc, vc = kc0.copy(), vc0.copy()
    key = _rand16((2, Hkv, d), torch.float16, 3)
    val = _rand16((2, Hkv, d), torch.float16, 4)
    oracle.cache_write(key, val, kc, vc, [12, -1])
    kb, vb = oracle.bits16(key), oracle.bits16(val)
    assert np.array_equal(kc[3, :, 0, :], kb[0]) and np.array_equal(vc[3, :, 0, :], vb[0])
    mask = np.ones(kc.shape, bool)
    mask[3, :, 0, :] = False
    assert np.array_equal(kc[mask], kc0[mask]) and np.array_equal(vc[mask], vc0[mask])


def pin_cache_write_roundtrip():
    """Tokens written through the slots of an allocated sequence come back,
    bit for bit, when the sequence is read through its block table."""
    B, Hkv, d, NB = 8, 3, 16, 40
    rng = np.random.default_rng(7)
    alloc = oracle.RefAllocator(NB, B, rng.permutation(NB))
    sid = alloc.seq_new(0)
    T = 37
    slots = [alloc.append(sid)[0] for _ in range(T)]
    kc = np.zeros((NB, Hkv, B, d), np.uint16)
    vc = np.zeros_like(kc)
    key = _rand16((T, Hkv, d), torch.bfloat16, 5)
    val = _rand16((T, Hkv, d), torch.bfloat16, 6)
    oracle.cache_write(key, val, kc, vc, slots)
    phys, off = oracle.locate_tokens(alloc.block_table(sid), B, T)
    kb, vb = oracle.bits16(key), oracle.bits16(val)
    for t in range(T):
        assert np.array_equal(kc[phys[t], :, off[t], :], kb[t])
        assert np.array_equal(vc[phys[t], :, off[t], :], vb[t])
    assert int((kc != 0).any(axis=(1, 2, 3)).sum()) <= -(-T // B)


# -- block copy ------------------------------------------------------------------

def pin_copy_blocks_exact():
    """dst := src for every pair, every other block unchanged (a block is all
    Hkv heads x B tokens x d of one tensor)."""
    NB, Hkv, B, d = 10, 2, 4, 8
    c0 = _pool(NB, Hkv, B, d, torch.float16, 9)
    c = c0.copy()
    oracle.copy_blocks(c, [(1, 7), (4, 2), (4, 9)])
    assert np.array_equal(c[7], c0[1]) and np.array_equal(c[2], c0[4]) and np.array_equal(c[9], c0[4])
    for b in (0, 1, 3, 4, 5, 6, 8):
        assert np.array_equal(c[b], c0[b])


# -- attention -------------------------------------------------------------------

def _sdpa_contiguous(q, kc, vc, ctx, dtype, H, Hkv):
    """Textbook attention (torch's scaled_dot_product_attention, fp64) over a
    contiguous copy: with the identity block table, sequence s's tokens are
    pool blocks s*mb .. s*mb+mb-1 in order."""
    S = q.shape[0]
    NB, _, B, d = kc.shape
    mb = NB // S
    G = H // Hkv
    out = np.zeros((S, H, d))
    for s in range(S):
        n = int(ctx[s])
        if n == 0:
            continue
        k = kc[s * mb:(s + 1) * mb].to(torch.float64).permute(1, 0, 2, 3).reshape(Hkv, mb * B, d)[:, :n]
        v = vc[s * mb:(s + 1) * mb].to(torch.float64).permute(1, 0, 2, 3).reshape(Hkv, mb * B, d)[:, :n]
        k = k.repeat_interleave(G, dim=0)
        v = v.repeat_interleave(G, dim=0)
        qq = q[s].to(torch.float64).reshape(H, 1, d)
        out[s] = F.scaled_dot_product_attention(qq[None], k[None], v[None])[0, :, 0].numpy()
    return out


def pin_attention_vs_sdpa(dtype=torch.float16, H=4, Hkv=2, d=32, B=8, ctx=(1, 5, 8, 9, 23, 40)):
    """Identity tables: the paged result equals textbook contiguous attention
    ("the result is identical to attending over one contiguous array")."""
    S = len(ctx)
    mb = -(-max(ctx) // B)
    NB = S * mb
    q = _rand16((S, H, d), dtype, 11)
    kc = _rand16((NB, Hkv, B, d), dtype, 12)
    vc = _rand16((NB, Hkv, B, d), dtype, 13)
    bt = np.arange(NB, dtype=np.int32).reshape(S, mb)
    got = oracle.paged_attention(q, kc, vc, bt, np.array(ctx), dtype)
    want = _sdpa_contiguous(q, kc, vc, ctx, dtype, H, Hkv)
    assert np.allclose(got, want, rtol=1e-12, atol=1e-14), np.abs(got - want).max()


def pin_attention_vs_sdpa_gqa():
    pin_attention_vs_sdpa(dtype=torch.bfloat16, H=8, Hkv=2, d=16, B=4, ctx=(3, 4, 17, 31))


def pin_attention_scale_argument():
    """An explicit scale multiplies q.k: scale c on q equals scale c on the call."""
    S, H, d, B = 2, 2, 16, 4
    ctx = np.array([7, 13])
    q = _rand16((S, H, d), torch.float16, 21)
    kc = _rand16((8, H, B, d), torch.float16, 22)
    vc = _rand16((8, H, B, d), torch.float16, 23)
    bt = np.arange(8, dtype=np.int32).reshape(2, 4)
    a = oracle.paged_attention(q, kc, vc, bt, ctx, "f16", scale=0.5 / math.sqrt(d))
    q2 = (q.to(torch.float64) * 0.5)
    want = np.zeros_like(a)
    for s in range(S):
        k = kc[s * 4:(s + 1) * 4].to(torch.float64).permute(1, 0, 2, 3).reshape(H, 16, d)[:, :ctx[s]]
        v = vc[s * 4:(s + 1) * 4].to(torch.float64).permute(1, 0, 2, 3).reshape(H, 16, d)[:, :ctx[s]]
        want[s] = F.scaled_dot_product_attention(q2[s].reshape(H, 1, d)[None], k[None], v[None])[0, :, 0].numpy()
    assert np.allclose(a, want, rtol=1e-12, atol=1e-14)


def pin_permutation_invariance():
    """Moving the same logical blocks to other physical blocks leaves every
    output bit-identical (blocks need not be adjacent)."""
    S, H, Hkv, d, B = 3, 4, 4, 16, 4
    ctx = np.array([9, 16, 30])
    mb = 8
    NB = 40
    rng = np.random.default_rng(3)
    q = _rand16((S, H, d), torch.float16, 31)
    kc = _pool(NB, Hkv, B, d, torch.float16, 32)
    vc = _pool(NB, Hkv, B, d, torch.float16, 33)
    bt = rng.permutation(NB)[:S * mb].astype(np.int32).reshape(S, mb)
    a = oracle.paged_attention(q, kc, vc, bt, ctx, "f16")
    perm = rng.permutation(NB)          # physical block b moves to perm[b]
    kc2 = np.empty_like(kc)
    vc2 = np.empty_like(vc)
    kc2[perm] = kc
    vc2[perm] = vc
    b = oracle.paged_attention(q, kc2, vc2, perm[bt].astype(np.int32), ctx, "f16")
    assert np.array_equal(a, b)


def pin_identical_keys_mean():
    """All keys equal: the softmax is uniform and the output is the mean of
    the values (closed form)."""
    S, H, d, B, n = 1, 1, 8, 4, 11
    q = _rand16((S, H, d), torch.float16, 41)
    kc = np.zeros((3, H, B, d), np.uint16)
    kc[:] = oracle.bits16(_rand16((d,), torch.float16, 42))
    vc = _pool(3, H, B, d, torch.float16, 43)
    bt = np.array([[2, 0, 1]], np.int32)
    got = oracle.paged_attention(q, kc, vc, bt, np.array([n]), "f16")[0, 0]
    vals = oracle.decode16(vc, "f16")
    toks = [vals[bt[0, t // B], 0, t % B] for t in range(n)]
    assert np.allclose(got, np.mean(toks, axis=0), rtol=1e-13, atol=1e-15)


def pin_single_token_and_empty():
    """ctx = 1 returns v_0 exactly; ctx = 0 returns zeros."""
    q = _rand16((2, 2, 8), torch.bfloat16, 51)
    kc = _pool(4, 2, 4, 8, torch.bfloat16, 52)
    vc = _pool(4, 2, 4, 8, torch.bfloat16, 53)
    bt = np.array([[3, 0], [1, 2]], np.int32)
    got = oracle.paged_attention(q, kc, vc, bt, np.array([1, 0]), "bf16")
    v = oracle.decode16(vc, "bf16")
    assert np.array_equal(got[0, 0], v[3, 0, 0]) and np.array_equal(got[0, 1], v[3, 1, 0])
    assert np.array_equal(got[1], np.zeros((2, 8)))


def pin_one_hot_limit():
    """One key much better aligned with q than the others takes (nearly) all
    the weight: the output tends to that token's value."""
    d, B, n = 16, 4, 10
    q = torch.zeros(1, 1, d, dtype=torch.float16)
    q[0, 0, 5] = 8.0
    kc = np.zeros((3, 1, B, d), np.uint16)
    j = 6                                          # logical token 6 -> block bt[1], offset 2
    bt = np.array([[1, 2, 0]], np.int32)
    kbits = torch.zeros(d, dtype=torch.float16)
    kbits[5] = 8.0
    kc[bt[0, j // B], 0, j % B] = oracle.bits16(kbits)
    vc = _pool(3, 1, B, d, torch.float16, 61)
    got = oracle.paged_attention(q, kc, vc, bt, np.array([n]), "f16")[0, 0]
    want = oracle.decode16(vc, "f16")[bt[0, j // B], 0, j % B]
    # weight of the others is (n-1) e^{-16} relative: under 1e-5
    assert np.allclose(got, want, rtol=0, atol=1e-5 * (1 + np.abs(want).max()))


def pin_which_subset():
    """Computing a subset of (s, h) gives exactly the rows of the full call."""
    S, H, Hkv, d, B = 3, 4, 2, 8, 4
    ctx = np.array([5, 12, 3])
    q = _rand16((S, H, d), torch.float16, 71)
    kc = _pool(12, Hkv, B, d, torch.float16, 72)
    vc = _pool(12, Hkv, B, d, torch.float16, 73)
    bt = np.arange(12, dtype=np.int32).reshape(3, 4)
    full = oracle.paged_attention(q, kc, vc, bt, ctx, "f16")
    part = oracle.paged_attention(q, kc, vc, bt, ctx, "f16", which=[(2, 3), (0, 1)])
    assert np.array_equal(part[2, 3], full[2, 3]) and np.array_equal(part[0, 1], full[0, 1])
    assert np.isnan(part[1]).all()


# -- split context -----------------------------------------------------------------

def pin_partition_merge_identity():
    """Splitting the context into partitions and merging by log-sum-exp gives
    the unsplit result (equal in exact arithmetic)."""
    S, H, Hkv, d, B = 2, 4, 1, 16, 8
    ctx = np.array([1000, 517])
    mb = 128
    NB = S * mb
    q = _rand16((S, H, d), torch.bfloat16, 81)
    kc = _pool(NB, Hkv, B, d, torch.bfloat16, 82)
    vc = _pool(NB, Hkv, B, d, torch.bfloat16, 83)
    bt = np.random.default_rng(8).permutation(NB).astype(np.int32).reshape(S, mb)
    full = oracle.paged_attention(q, kc, vc, bt, ctx, "bf16")
    for P in (16, 96, 512, 4096):
        for s in range(S):
            for h in range(H):
                m, l, o = oracle.partition_stats(q, kc, vc, bt, ctx, "bf16", s, h, P)
                assert len(m) == -(-int(ctx[s]) // P)
                got = oracle.merge_partitions(m, l, o)
                assert np.allclose(got, full[s, h], rtol=1e-12, atol=1e-14)


def pin_partition_stats_definition():
    """A single partition's (m, l, o) are the max score, the sum of
    exp(score - m) and the un-normalised value sum, computed directly."""
    d, B = 8, 4
    q = _rand16((1, 1, d), torch.float16, 91)
    kc = _pool(4, 1, B, d, torch.float16, 92)
    vc = _pool(4, 1, B, d, torch.float16, 93)
    bt = np.array([[2, 3, 0, 1]], np.int32)
    m, l, o = oracle.partition_stats(q, kc, vc, bt, np.array([14]), "f16", 0, 0, 8)
    K = oracle.decode16(kc, "f16")
    V = oracle.decode16(vc, "f16")
    qq = q.to(torch.float64).numpy()[0, 0]
    for p, (t0, t1) in enumerate([(0, 8), (8, 14)]):
        ks = np.array([K[bt[0, t // B], 0, t % B] for t in range(t0, t1)])
        vs = np.array([V[bt[0, t // B], 0, t % B] for t in range(t0, t1)])
        x = ks @ qq / math.sqrt(d)
        assert np.isclose(m[p], x.max(), rtol=1e-14)
        w = np.exp(x - x.max())
        assert np.isclose(l[p], w.sum(), rtol=1e-13)
        assert np.allclose(o[p], w @ vs, rtol=1e-12, atol=1e-14)


# -- sizes from the pages -------------------------------------------------------------

# -- prompt phase (many query tokens per sequence, causal) -------------------------

def _prefill_inputs(ctx, nq, H, Hkv, d, B, dtype, seed, permute=True):
    """A pool, tables and queries for sequences with context ctx[s] whose last
    nq[s] tokens are the new ones."""
    S = len(ctx)
    mb = max(1, -(-max(ctx) // B))
    NB = S * mb + 3
    rng = np.random.default_rng(seed)
    ids = rng.permutation(NB) if permute else np.arange(NB)
    bt = ids[:S * mb].astype(np.int32).reshape(S, mb)
    qs = np.concatenate([[0], np.cumsum(nq)]).astype(np.int32)
    q = _rand16((int(qs[-1]), H, d), dtype, seed + 1)
    kc = _rand16((NB, Hkv, B, d), dtype, seed + 2)
    vc = _rand16((NB, Hkv, B, d), dtype, seed + 3)
    return q, kc, vc, bt, np.array(ctx), qs


def _sdpa_causal(q, kc, vc, bt, ctx, qs, H, Hkv):
    """Textbook masked attention (torch's scaled_dot_product_attention, fp64)
    over each sequence's tokens copied out in logical order; new token j of
    sequence s may see tokens t <= ctx[s] - n_s + j."""
    _, _, B, d = kc.shape
    G = H // Hkv
    out = np.zeros((q.shape[0], H, d))
    for s in range(len(ctx)):
        n, c = int(qs[s + 1] - qs[s]), int(ctx[s])
        if n == 0:
            continue
        rows = [kc[bt[s, t // B], :, t % B] for t in range(c)]
        k = torch.stack(rows, 1).to(torch.float64).repeat_interleave(G, dim=0)      # [H][c][d]
        v = torch.stack([vc[bt[s, t // B], :, t % B] for t in range(c)], 1).to(torch.float64)
        v = v.repeat_interleave(G, dim=0)
        qq = q[qs[s]:qs[s + 1]].to(torch.float64).permute(1, 0, 2)                  # [H][n][d]
        mask = torch.arange(c)[None, :] <= (c - n + torch.arange(n))[:, None]       # [n][c]
        o = F.scaled_dot_product_attention(qq[None], k[None], v[None], attn_mask=mask)[0]
        out[qs[s]:qs[s + 1]] = o.permute(1, 0, 2).numpy()
    return out


def pin_prefill_vs_sdpa_causal():
    """Causal prompt-phase attention equals the library's masked attention on
    the same tokens: plain prompts (context = new tokens), prompts after a
    cached prefix, single new tokens and sequences with none."""
    for dtype, H, Hkv, d, B, ctx, nq in (
            (torch.float16, 4, 4, 16, 4, (7, 9, 30, 5, 12), (7, 2, 30, 1, 0)),
            (torch.bfloat16, 8, 2, 32, 8, (40, 17, 64), (13, 17, 40))):
        q, kc, vc, bt, cl, qs = _prefill_inputs(ctx, nq, H, Hkv, d, B, dtype, 61)
        got = oracle.paged_prefill(q, kc, vc, bt, cl, qs, dtype)
        want = _sdpa_causal(q, kc, vc, bt, cl, qs, H, Hkv)
        assert np.allclose(got, want, rtol=1e-12, atol=1e-14), np.abs(got - want).max()


def pin_prefill_rows_are_truncated_decodes():
    """New token j of sequence s is the decode of a sequence whose context
    stops at its own position (bit-identical: the same sum over the same
    tokens)."""
    H, Hkv, d, B = 4, 2, 16, 4
    ctx, nq = (21, 8, 13), (6, 8, 1)
    q, kc, vc, bt, cl, qs = _prefill_inputs(ctx, nq, H, Hkv, d, B, torch.float16, 71)
    got = oracle.paged_prefill(q, kc, vc, bt, cl, qs, "f16")
    for s in range(len(ctx)):
        for j in range(nq[s]):
            tok = qs[s] + j
            pos = ctx[s] - nq[s] + j
            want = oracle.paged_attention(q[tok:tok + 1], kc, vc, bt[s:s + 1], np.array([pos + 1]), "f16")
            assert np.array_equal(got[tok], want[0]), (s, j)


def pin_prefill_prompt_worked_example():
    """The 7-token prompt of the pages' request walk-through, written into
    physical blocks 7 and 1: with all scores equal, token i averages values
    0..i (hand-computed in the fixture)."""
    g = golden("prefill_prompt_fig6.json")
    B, n, d, NB = g["block_size"], g["prompt_tokens"], g["head_dim"], g["num_blocks"]
    kc = np.zeros((NB, 1, B, d), np.uint16)
    vc = np.zeros((NB, 1, B, d), np.uint16)
    key = _rand16((n, 1, d), torch.float16, 81)
    value = torch.tensor([[[t + 1.0, -2.0 * (t + 1)]] for t in range(n)], dtype=torch.float16)
    blocks = g["physical_blocks"]
    slots = np.array([blocks[t // B] * B + t % B for t in range(n)])
    oracle.cache_write(key, value, kc, vc, slots)
    bt = np.array([blocks], np.int32)
    q = torch.zeros(n, 1, d, dtype=torch.float16)
    got = oracle.paged_prefill(q, kc, vc, bt, np.array([n]), np.array([0, n]), "f16")[:, 0]
    assert np.allclose(got, np.array(g["expected_out_per_token"]), rtol=1e-14, atol=1e-14), got


def pin_prefill_future_tokens_ignored():
    """Changing the keys and values after a token's position leaves its row
    bit-identical; changing its own key and value changes it."""
    H, d, B = 2, 8, 4
    ctx, nq = (19,), (11,)
    q, kc, vc, bt, cl, qs = _prefill_inputs(ctx, nq, H, H, d, B, torch.float16, 91)
    kb, vb = oracle.bits16(kc), oracle.bits16(vc)
    a = oracle.paged_prefill(q, kb, vb, bt, cl, qs, "f16")
    pos = 12                                     # new token j = 4 sits at position 8 + 4
    j = pos - (ctx[0] - nq[0])
    kb2, vb2 = kb.copy(), vb.copy()
    for t in range(pos + 1, ctx[0]):
        kb2[bt[0, t // B], :, t % B] ^= 0x1234
        vb2[bt[0, t // B], :, t % B] ^= 0x0F0F
    b = oracle.paged_prefill(q, kb2, vb2, bt, cl, qs, "f16")
    assert np.array_equal(a[:j + 1], b[:j + 1])
    assert not np.array_equal(a[j + 1:], b[j + 1:])
    vb3 = vb.copy()
    vb3[bt[0, pos // B], :, pos % B] ^= 0x0100
    c = oracle.paged_prefill(q, kb, vb3, bt, cl, qs, "f16")
    assert np.array_equal(a[:j], c[:j]) and not np.array_equal(a[j], c[j])


def pin_prefill_identical_keys_prefix_mean():
    """All keys equal, after a 10-token prefix: new token j averages the
    values of tokens 0..10+j (closed form)."""
    H, d, B = 1, 8, 4
    ctx, nq = (16,), (6,)
    q, kc, vc, bt, cl, qs = _prefill_inputs(ctx, nq, H, H, d, B, torch.bfloat16, 101)
    kb = np.zeros(kc.shape, np.uint16)
    kb[:] = oracle.bits16(_rand16((d,), torch.bfloat16, 102))
    got = oracle.paged_prefill(q, kb, vc, bt, cl, qs, "bf16")[:, 0]
    vals = oracle.decode16(oracle.bits16(vc), "bf16")
    toks = np.array([vals[bt[0, t // B], 0, t % B] for t in range(ctx[0])])
    for j in range(nq[0]):
        assert np.allclose(got[j], toks[:10 + j + 1].mean(axis=0), rtol=1e-13, atol=1e-15)


def pin_prefill_which_subset():
    """Rows asked for by (token, head) equal the same rows of the full run."""
    ctx, nq = (9, 30, 4), (3, 20, 4)
    q, kc, vc, bt, cl, qs = _prefill_inputs(ctx, nq, 4, 2, 16, 8, torch.float16, 111)
    full = oracle.paged_prefill(q, kc, vc, bt, cl, qs, "f16")
    which = [(26, 3), (0, 0), (22, 1), (5, 2), (3, 0)]
    part = oracle.paged_prefill(q, kc, vc, bt, cl, qs, "f16", which=which)
    for t, h in which:
        assert np.array_equal(part[t, h], full[t, h])
    assert np.isnan(part[1, 1]).all()


# -- beam search ------------------------------------------------------------------

def _fig9_tree():
    """Candidates A=[0,1,3,6], B=[0,1,3,7], C=[0,2,4,8], D=[0,1,5] (block size
    2, every block full), built with fork/append in block-id order."""
    a = oracle.RefAllocator(16, 2)
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
    return a, [A, Bc, C, D]


def pin_beam_step_fig9():
    """The width-4 step of the pages' Figure 9: survivors A and B each branch
    in two, C and D are pruned; the four survivors grow into new blocks 9-12
    and the blocks only C and D held (2, 4, 5, 8) return to the pool, while
    block 0 stays shared by all."""
    g = golden("beam_prune_fig9.json")
    a, (A, Bc, C, D) = _fig9_tree()
    new, slots, pairs = a.beam_step([A, Bc, C, D], [0, 0, 1, 1])
    assert new[0] == A and new[2] == Bc and len(set(new)) == 4 and not pairs
    assert [a.block_table(s)[-1] for s in new] == g["new_for_survivors"]
    assert sorted(a.free_list()[:4]) == g["freed_on_prune"]
    assert all(a.block_ref(b) == 0 for b in g["freed_on_prune"])
    assert a.block_ref(g["shared_by_all"]) == 4
    assert slots == [b * 2 for b in g["new_for_survivors"]]


def pin_beam_step_single_block_copy():
    """Children of one parent writing into its shared, partly filled last
    block: every child but the last copies that one block (the last writes in
    place); full shared blocks are never copied."""
    a = oracle.RefAllocator(16, 4)
    p = a.seq_new(6)                           # [b0 full, b1 with 2 of 4]
    b0, b1 = a.block_table(p)
    new, slots, pairs = a.beam_step([p], [0, 0, 0])
    assert len(pairs) == 2 and all(src == b1 for src, _ in pairs)
    tabs = [a.block_table(s) for s in new]
    assert all(t[0] == b0 for t in tabs) and a.block_ref(b0) == 3
    assert sorted(t[1] for t in tabs) == sorted([b1] + [d for _, d in pairs])
    assert a.block_ref(b1) == 1 and all(s % 4 == 2 for s in slots)


def pin_beam_step_all_or_nothing():
    a = oracle.RefAllocator(3, 2)
    p = a.seq_new(3)                            # 2 blocks, 1 free
    before = _alloc_state(a), a._next_id
    try:
        a.beam_step([p], [0, 0, 0])             # needs two copies
        raise AssertionError("a step without room went through")
    except oracle.AllocatorOOM:
        pass
    assert (_alloc_state(a), a._next_id) == before


def pin_beam_memory_closed_form():
    """k beams sharing a P-block prompt, each with its own t-block tail: the
    pool holds P + k t blocks, k (P + t) without sharing."""
    B, P, t, k = 4, 5, 3, 4
    a = oracle.RefAllocator(64, B)
    root = a.seq_new(P * B)
    beams = [root] + [a.fork(root) for _ in range(k - 1)]
    for _ in range(t * B):
        beams, _, _ = a.beam_step(beams, list(range(k)))
    used = a.blocks_in_use()
    unshared = sum(-(-a.seq_len(b) // B) for b in beams)
    assert used == P + k * t and unshared == k * (P + t)


# -- swapping between a GPU and a CPU pool ------------------------------------------

def _alloc_state(a):
    return (list(a.ref), a.free_list(), {k: (list(v["blocks"]), v["len"]) for k, v in a._seqs.items()})


def _sampling_group(a, prompt=10, samples=3, suffix=(2, 0, 5)):
    """A prompt forked into samples that each append a suffix (copy on write
    of the shared, partly filled last block)."""
    root = a.seq_new(prompt)
    ids = [root] + [a.fork(root) for _ in range(samples - 1)]
    for sid, n in zip(ids, suffix):
        for _ in range(n):
            a.append(sid)
    return ids


def pin_swap_all_or_nothing():
    """A group that does not fit in the other pool moves not at all."""
    g = oracle.RefAllocator(16, 4)
    ids = _sampling_group(g)
    need = len({b for s in ids for b in g.block_table(s)})
    c = oracle.RefAllocator(need - 1, 4)
    before_g, before_c = _alloc_state(g), _alloc_state(c)
    try:
        g.move_group(c, ids)
        raise AssertionError("a group larger than the free pool moved")
    except oracle.AllocatorOOM:
        pass
    assert _alloc_state(g) == before_g and _alloc_state(c) == before_c


def pin_swap_preserves_sharing():
    """Moving out and back keeps lengths, the sharing pattern and the
    reference counts; the source pool gets every block back."""
    g = oracle.RefAllocator(32, 4, free_order=np.random.default_rng(5).permutation(32))
    ids = _sampling_group(g, prompt=13, samples=4, suffix=(3, 0, 1, 6))
    tables = [g.block_table(s) for s in ids]
    lens = [g.seq_len(s) for s in ids]
    refs = {b: g.block_ref(b) for t in tables for b in t}
    free0 = g.num_free() + len(refs)
    c = oracle.RefAllocator(24, 4)
    cids, pairs = g.move_group(c, ids)
    assert g.num_free() == free0 and len(pairs) == len(refs)
    remap = dict(pairs)
    assert [c.block_table(s) for s in cids] == [[remap[b] for b in t] for t in tables]
    assert all(c.block_ref(remap[b]) == n for b, n in refs.items())
    assert [c.seq_len(s) for s in cids] == lens
    gids, back = c.move_group(g, cids)
    assert c.num_free() == 24
    # the same structure again (block ids may differ)
    t2 = [g.block_table(s) for s in gids]
    eq = lambda ts: [[ts[i][x] == ts[j][y] for j in range(len(ts)) for y in range(len(ts[j]))]
                     for i in range(len(ts)) for x in range(len(ts[i]))]
    assert eq(t2) == eq(tables) and [g.seq_len(s) for s in gids] == lens


def pin_swap_group_must_hold_all_references():
    """Sequences sharing blocks are evicted together: half a group is refused."""
    g = oracle.RefAllocator(16, 4)
    ids = _sampling_group(g)
    c = oracle.RefAllocator(16, 4)
    before = _alloc_state(g)
    try:
        g.move_group(c, ids[:1])
        raise AssertionError("half of a sharing group moved")
    except ValueError:
        pass
    assert _alloc_state(g) == before


def pin_swap_space_bound():
    """A CPU pool as large as the GPU pool always holds everything swapped out
    (one can never swap out more than exists)."""
    rng = np.random.default_rng(9)
    g = oracle.RefAllocator(40, 4, free_order=rng.permutation(40))
    groups = []
    while True:
        try:
            groups.append(_sampling_group(g, prompt=int(rng.integers(1, 9)), samples=2,
                                          suffix=(int(rng.integers(0, 4)), int(rng.integers(0, 4)))))
        except oracle.AllocatorOOM:
            break
    c = oracle.RefAllocator(40, 4)
    for grp in groups:
        g.move_group(c, grp)
    rest = list(g._seqs)                 # what the last, failed group had created
    if rest:
        g.move_group(c, rest)
    assert g.num_free() == 40 and c.num_free() == 40 - sum(1 for b in range(40) if c.block_ref(b))


def pin_copy_between_exact():
    """Only the destination blocks of the pairs change, each to its source."""
    rng = np.random.default_rng(13)
    src = rng.integers(0, 65536, size=(7, 2, 4, 8), dtype=np.uint16)
    dst = rng.integers(0, 65536, size=(5, 2, 4, 8), dtype=np.uint16)
    pairs = [(6, 0), (2, 3), (6, 4)]
    want = dst.copy()
    for s_, d_ in pairs:
        want[d_] = src[s_]
    oracle.copy_blocks_between(dst, src, pairs)
    assert np.array_equal(dst, want)


def pin_swap_round_trip_attention():
    """Swapping a group out (device copy to the CPU pool), clobbering the GPU
    pool and swapping it back in leaves every sequence's attention output
    bit-identical."""
    H, d, B = 2, 8, 4
    g = oracle.RefAllocator(24, B, free_order=np.random.default_rng(3).permutation(24))
    ids = _sampling_group(g, prompt=9, samples=3, suffix=(4, 1, 0))
    kg = _pool(24, H, B, d, torch.float16, 141)
    vg = _pool(24, H, B, d, torch.float16, 142)
    q = _rand16((3, H, d), torch.float16, 143)
    def attend(a, sids, kc, vc):
        bt = np.full((3, 8), -1, np.int32)
        for i, s_ in enumerate(sids):
            t = a.block_table(s_)
            bt[i, :len(t)] = t
        return oracle.paged_attention(q, kc, vc, bt, np.array([a.seq_len(s_) for s_ in sids]), "f16")
    before = attend(g, ids, kg, vg)
    c = oracle.RefAllocator(16, B)
    kc = np.zeros((16, H, B, d), np.uint16)
    vc = np.zeros((16, H, B, d), np.uint16)
    cids, out_pairs = g.move_group(c, ids)
    oracle.copy_blocks_between(kc, kg, out_pairs)
    oracle.copy_blocks_between(vc, vg, out_pairs)
    kg[:] = 0x7E00                                   # NaN everywhere on the GPU side
    vg[:] = 0x7E00
    gids, in_pairs = c.move_group(g, cids)
    oracle.copy_blocks_between(kg, kc, in_pairs)
    oracle.copy_blocks_between(vg, vc, in_pairs)
    assert np.array_equal(attend(g, gids, kg, vg), before)


def pin_kv_size():
    g = golden("kv_size_opt13b.json")
    per = oracle.kv_bytes_per_token(g["hidden"], g["layers"], g["bytes_per_number"])
    assert per == g["per_token_bytes"]
    assert per / 1024 == g["per_token_kb"]
    assert round(g["request_tokens"] * per / 1024 / 1e6, 1) == g["request_gb_rounded"]


def pin_capacity():
    g = golden("capacity_13b.json")
    slots = g["kv_memory_gib"] * 2 ** g["kv_memory_bytes_exponent"] / (g["per_token_kb"] * 1024)
    assert round(slots / 1000, 1) == g["max_slots_thousands_rounded"]


def pin_waste_example():
    g = golden("waste_100_200.json")
    used = g["prompt_tokens"] + g["output_tokens"]
    assert used == g["used_slots"]
    assert g["reservation_tokens"] - used == g["reservation_waste_slots"]
    assert round(100 * (g["reservation_tokens"] - used) / g["reservation_tokens"]) == \
        g["reservation_waste_percent_rounded"]
    n = oracle.blocks_needed(used, g["block_size"])
    assert n == g["blocks"] and n * g["block_size"] == g["block_slots"]
    assert n * g["block_size"] - used == g["block_waste_slots"]
    a = oracle.RefAllocator(32, g["block_size"])
    sid = a.seq_new(g["prompt_tokens"])
    for _ in range(g["output_tokens"]):
        a.append(sid)
    assert len(a.block_table(sid)) == g["blocks"]


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]


def run_all(lib_path=None):
    """Run every pin (against the oracle build at lib_path, if given) and
    return the names of the pins that failed."""
    if lib_path is not None:
        oracle._lib = oracle.load(lib_path)
    failed = []
    for pin in ALL_PINS:
        try:
            pin()
        except (AssertionError, ValueError):
            failed.append(pin.__name__)
    return failed


if __name__ == "__main__":
    # python tests/pins.py <liboracle.so>: used by the planted-mistake test, one
    # process per mutant, so that a mutant that corrupts memory cannot touch the
    # test process.
    import sys
    print(json.dumps(run_all(sys.argv[1] if len(sys.argv) > 1 else None)))
