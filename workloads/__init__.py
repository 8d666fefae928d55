"""Seeded synthetic inputs for the paged decode workloads.

This module is shared by the CUDA path and by the oracle, so it holds only
random draws and shapes: no attention, no block-table gather, no slot
arithmetic, no allocation rule.  Everything it returns is either a plain
integer/array of sizes or a tensor of N(0, 1) samples.

The five workloads follow the decode settings described on the pages
("PagedAttention and vLLM, annotated" §3 and §7.2 for the 16-token block and
the 100+200 token request; "vLLM & PagedAttention" §V for the per-step decode
and §VII for parallel sampling over shared prompt blocks):

  tiny        4 seqs, MHA 2 x 64, B=16, contexts {1,17,100,300}, 64-block pool
  opt13b      OPT-13B layer (40 x 128 MHA), 64 seqs, lognormal prompt+output
  llama7b     Llama-2-7B layer (32 x 128 MHA), 256 seqs, uniform[1,4096], B swept
  sampling    64 prompts x 4 samples over shared prompt blocks (CoW)
  longgqa     32 q-heads / 8 kv-heads, 8 seqs x 32768 tokens, bf16
  prefix      prompt phase: 32 requests after a shared 1000-token prefix
  swap        32 Llama-2-7B-layer sequences swapped to a CPU pool and back
  beam        16 OPT-13B-layer requests searched with 2-6 beams

The pages give no length distribution for real traffic (their ShareGPT and
Alpaca traces are not available here); the lognormal and uniform models below
stand in for them.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

BASE_SEED = 139

DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16}


@dataclasses.dataclass
class Workload:
    """Sizes and per-sequence lengths of one decode batch (one layer)."""

    name: str
    num_seqs: int
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    dtype: str                      # "f16" or "bf16"
    context_lens: np.ndarray        # int64 [num_seqs], includes the decode token
    max_blocks_per_seq: int         # width of the block table
    num_blocks: int                 # physical blocks in the pool
    seed: int
    partition_size: int = 0         # 0 = let the library choose
    # parallel-sampling workload only
    samples_per_prompt: int = 1
    prompt_lens: Optional[np.ndarray] = None   # int64 [num_prompts]
    suffix_lens: Optional[np.ndarray] = None   # int64 [num_seqs]
    # prompt-phase (shared-prefix) workload only: new tokens per sequence, the
    # last query_lens[s] of context_lens[s], after a prefix of prefix_len
    query_lens: Optional[np.ndarray] = None    # int64 [num_seqs]
    prefix_len: int = 0

    @property
    def torch_dtype(self) -> torch.dtype:
        return DTYPES[self.dtype]

    @property
    def esize(self) -> int:
        return 2

    @property
    def kv_bytes_per_token(self) -> int:
        """K and V bytes of one token of one layer (all kv heads)."""
        return 2 * self.num_kv_heads * self.head_dim * self.esize

    def describe(self) -> dict:
        return {
            "workload": self.name,
            "num_seqs": self.num_seqs,
            "num_heads": self.num_heads,
            "num_kv_heads": self.num_kv_heads,
            "head_dim": self.head_dim,
            "block_size": self.block_size,
            "dtype": self.dtype,
            "num_blocks": self.num_blocks,
            "sum_context": int(self.context_lens.sum()),
            "max_context": int(self.context_lens.max()) if self.num_seqs else 0,
        }


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def lognormal_lengths(rng: np.random.Generator, mean: float, n: int,
                      sigma: float = 1.0) -> np.ndarray:
    """Integer lengths >= 1 from a lognormal with the given arithmetic mean.

    mu is chosen so that E[X] = exp(mu + sigma^2/2) equals `mean`.
    """
    mu = math.log(mean) - 0.5 * sigma * sigma
    x = rng.lognormal(mean=mu, sigma=sigma, size=n)
    return np.maximum(1, np.rint(x)).astype(np.int64)


def uniform_lengths(rng: np.random.Generator, lo: int, hi: int, n: int) -> np.ndarray:
    """Integers uniform on [lo, hi], both ends included."""
    return rng.integers(lo, hi + 1, size=n, dtype=np.int64)


def _ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def free_order(num_blocks: int, seed: int) -> np.ndarray:
    """A seeded permutation of 0..num_blocks-1: the order in which a fresh
    pool hands out its physical blocks."""
    return _rng(seed ^ 0x5EED).permutation(num_blocks).astype(np.int32)


def tiny(seed: int = BASE_SEED * 1000 + 1) -> Workload:
    ctx = np.array([1, 17, 100, 300], dtype=np.int64)
    return Workload("tiny: 4 seqs, MHA 2x64, B=16, ctx {1,17,100,300}, 64-block pool, f16",
                    num_seqs=4, num_heads=2, num_kv_heads=2, head_dim=64, block_size=16,
                    dtype="f16", context_lens=ctx, max_blocks_per_seq=_ceil_div(300, 16),
                    num_blocks=64, seed=seed)


def opt13b(num_seqs: int = 64, seed: int = BASE_SEED * 1000 + 2, max_ctx: int = 2048) -> Workload:
    rng = _rng(seed)
    prompt = lognormal_lengths(rng, 160.0, num_seqs)
    output = lognormal_lengths(rng, 340.0, num_seqs)
    ctx = np.clip(prompt + output, 1, max_ctx)
    B = 16
    nb = int(sum(_ceil_div(int(c), B) for c in ctx))
    return Workload(f"opt13b: {num_seqs} seqs, MHA 40x128, B=16, ctx lognormal(160)+lognormal(340) <= {max_ctx}, f16",
                    num_seqs=num_seqs, num_heads=40, num_kv_heads=40, head_dim=128, block_size=B,
                    dtype="f16", context_lens=ctx, max_blocks_per_seq=_ceil_div(max_ctx, B),
                    num_blocks=nb + 64, seed=seed)


def llama7b(block_size: int = 16, num_seqs: int = 256, max_ctx: int = 4096,
            seed: Optional[int] = None, head_dim: int = 128) -> Workload:
    """Llama-2-7B layer shapes (32 MHA heads).  head_dim 64 (with the same 32
    heads) is the small-head variant of the block-size study."""
    if seed is None:
        seed = BASE_SEED * 1000 + 3
    rng = _rng(seed)             # the same contexts for every block size
    ctx = uniform_lengths(rng, 1, max_ctx, num_seqs)
    nb = int(sum(_ceil_div(int(c), block_size) for c in ctx))
    return Workload(f"llama7b: {num_seqs} seqs, MHA 32x{head_dim}, B={block_size}, ctx uniform[1,{max_ctx}], f16",
                    num_seqs=num_seqs, num_heads=32, num_kv_heads=32, head_dim=head_dim,
                    block_size=block_size, dtype="f16", context_lens=ctx,
                    max_blocks_per_seq=_ceil_div(max_ctx, block_size), num_blocks=nb,
                    seed=seed + block_size + (0 if head_dim == 128 else 1000 * head_dim))


def sampling(num_prompts: int = 64, samples: int = 4, prompt_len: int = 512,
             max_suffix: int = 256, partial_last_block: bool = True,
             seed: int = BASE_SEED * 1000 + 4) -> Workload:
    """Parallel sampling: each prompt is shared by `samples` sequences.

    With partial_last_block, prompt p has length prompt_len - r_p with r_p
    uniform on [1, 15], so its last block is partly filled and shared; the
    companion run (partial_last_block=False) keeps exactly prompt_len tokens.
    Each sample then appends suffix_len tokens, then the decode token.
    """
    B = 16
    rng = _rng(seed)
    if partial_last_block:
        prompts = prompt_len - uniform_lengths(rng, 1, B - 1, num_prompts)
    else:
        prompts = np.full(num_prompts, prompt_len, dtype=np.int64)
    suffix = uniform_lengths(rng, 0, max_suffix, num_prompts * samples)
    ctx = np.repeat(prompts, samples) + suffix + 1
    max_ctx = prompt_len + max_suffix + 1
    # enough blocks if nothing were shared
    nb = int(sum(_ceil_div(int(c), B) for c in ctx)) + 64
    return Workload(f"sampling: {num_prompts} prompts x {samples} samples, MHA 32x128, B=16, "
                    f"prompt {'512-r' if partial_last_block else '512'}, suffix uniform[0,{max_suffix}], f16",
                    num_seqs=num_prompts * samples, num_heads=32, num_kv_heads=32, head_dim=128,
                    block_size=B, dtype="f16", context_lens=ctx,
                    max_blocks_per_seq=_ceil_div(max_ctx, B), num_blocks=nb, seed=seed,
                    samples_per_prompt=samples, prompt_lens=prompts, suffix_lens=suffix)


def longgqa(num_seqs: int = 8, ctx_len: int = 32768, seed: int = BASE_SEED * 1000 + 5,
            partition_size: int = 512) -> Workload:
    B = 16
    ctx = np.full(num_seqs, ctx_len, dtype=np.int64)
    mb = _ceil_div(ctx_len, B)
    return Workload(f"longgqa: {num_seqs} seqs x {ctx_len}, GQA 32q/8kv x 128, B=16, partitions of {partition_size}, bf16",
                    num_seqs=num_seqs, num_heads=32, num_kv_heads=8, head_dim=128, block_size=B,
                    dtype="bf16", context_lens=ctx, max_blocks_per_seq=mb,
                    num_blocks=num_seqs * mb, seed=seed, partition_size=partition_size)


def prefix(num_requests: int = 32, prefix_len: int = 1000, min_own: int = 64, max_own: int = 512,
           num_heads: int = 32, num_kv_heads: int = 32, head_dim: int = 128, block_size: int = 16,
           dtype: str = "f16", seed: int = BASE_SEED * 1000 + 6) -> Workload:
    """Shared prefix ("vLLM & PagedAttention" §VII): one cached prefix (a
    system prompt or few-shot examples) of prefix_len tokens and num_requests
    requests whose own inputs, uniform[min_own, max_own] tokens, follow it.
    The prompt phase runs over the own tokens only; each attends the prefix
    and the own tokens up to itself.  The pool holds the prefix once, each
    request's copy of the prefix's partly filled last block and its new
    blocks, plus slack."""
    B = block_size
    rng = _rng(seed)
    own = uniform_lengths(rng, min_own, max_own, num_requests)
    ctx = prefix_len + own
    shared_full = prefix_len // B
    nb = _ceil_div(prefix_len, B) + int(sum(_ceil_div(int(c), B) - shared_full for c in ctx)) + 64
    return Workload(f"prefix: {num_requests} requests after a shared {prefix_len}-token prefix, own input "
                    f"uniform[{min_own},{max_own}], {'MHA' if num_heads == num_kv_heads else 'GQA'} "
                    f"{num_heads}/{num_kv_heads}x{head_dim}, B={B}, {dtype}",
                    num_seqs=num_requests, num_heads=num_heads, num_kv_heads=num_kv_heads, head_dim=head_dim,
                    block_size=B, dtype=dtype, context_lens=ctx,
                    max_blocks_per_seq=_ceil_div(prefix_len + max_own, B), num_blocks=nb, seed=seed,
                    query_lens=own, prefix_len=prefix_len)


def swap(block_size: int = 16, num_seqs: int = 32, min_ctx: int = 512, max_ctx: int = 4096,
         seed: int = BASE_SEED * 1000 + 7) -> Workload:
    """Swapping ("vLLM & PagedAttention" §VIII): a batch of Llama-2-7B-layer
    sequences (32 x 128 MHA, f16), contexts uniform[min_ctx, max_ctx], all
    evicted to a CPU pool of the same size and brought back; the block size
    is the ablation's variable (§XII)."""
    rng = _rng(seed)
    ctx = uniform_lengths(rng, min_ctx, max_ctx, num_seqs)
    nb = int(sum(_ceil_div(int(c), block_size) for c in ctx))
    return Workload(f"swap: {num_seqs} seqs, MHA 32x128, B={block_size}, ctx uniform[{min_ctx},{max_ctx}], f16",
                    num_seqs=num_seqs, num_heads=32, num_kv_heads=32, head_dim=128, block_size=block_size,
                    dtype="f16", context_lens=ctx, max_blocks_per_seq=_ceil_div(max_ctx, block_size),
                    num_blocks=nb, seed=seed + block_size)


def beam(width: int = 4, num_requests: int = 16, steps: int = 192, seed: int = BASE_SEED * 1000 + 8) -> Workload:
    """Beam search ("vLLM & PagedAttention" §VII, Fig. 9; §XII Fig. 15 for
    widths 2 to 6): OPT-13B-layer requests (40 x 128 MHA, f16, B=16) with
    lognormal(160) prompts, each searched with `width` beams for `steps`
    tokens.  context_lens holds the prompts; parents are drawn by
    beam_parents."""
    rng = _rng(seed)
    prompt = lognormal_lengths(rng, 160.0, num_requests)
    prompt = np.clip(prompt, 1, 1024)
    B = 16
    max_len = int(prompt.max()) + steps + 1
    # room for every beam's own copy of everything (the unshared bound) plus slack
    nb = int(sum(width * _ceil_div(int(p_) + steps + 1, B) for p_ in prompt)) + 64
    return Workload(f"beam: {num_requests} requests x width {width}, OPT-13B layer (MHA 40x128), B=16, "
                    f"prompt lognormal(160), {steps} steps, f16",
                    num_seqs=num_requests, num_heads=40, num_kv_heads=40, head_dim=128, block_size=B, dtype="f16",
                    context_lens=prompt, max_blocks_per_seq=_ceil_div(max_len, B), num_blocks=nb, seed=seed + width,
                    samples_per_prompt=width)


def beam_parents(rng: np.random.Generator, k: int, width: int) -> np.ndarray:
    """Parents of the next `width` candidates among k current beams (ranked
    best first): the better of two uniform draws, so strong beams tend to
    branch and weak ones to die."""
    a = rng.integers(0, k, size=width)
    b = rng.integers(0, k, size=width)
    return np.sort(np.minimum(a, b)).astype(np.int32)


def by_name(name: str, **kw) -> Workload:
    table = {"tiny": tiny, "opt13b": opt13b, "llama7b": llama7b,
             "sampling": sampling, "longgqa": longgqa, "prefix": prefix, "swap": swap, "beam": beam}
    return table[name](**kw)


def normal(shape, dtype: str, seed: int, device="cpu") -> torch.Tensor:
    """N(0,1) samples rounded to fp16/bf16, seeded; generated on `device`."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    x = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    return x.to(DTYPES[dtype])


def tensors(w: Workload, device="cpu") -> dict:
    """The random tensors of one decode step: query, the decode token's key and
    value, and the initial (pre-filled) contents of the K and V pools."""
    S, H, Hkv, d, B = w.num_seqs, w.num_heads, w.num_kv_heads, w.head_dim, w.block_size
    return {
        "query": normal((S, H, d), w.dtype, w.seed + 11, device),
        "key": normal((S, Hkv, d), w.dtype, w.seed + 12, device),
        "value": normal((S, Hkv, d), w.dtype, w.seed + 13, device),
        "key_cache": normal((w.num_blocks, Hkv, B, d), w.dtype, w.seed + 14, device),
        "value_cache": normal((w.num_blocks, Hkv, B, d), w.dtype, w.seed + 15, device),
    }


def prefill_tensors(w: Workload, device="cpu") -> dict:
    """The random tensors of one prompt-phase step: the keys and values of the
    cached prefix (the shared one, or with prefix_len 0 every sequence's
    cached tokens back to back), and the queries, keys and values of every
    request's own tokens (request-major, token-minor)."""
    T = int(w.query_lens.sum())
    Hkv, d = w.num_kv_heads, w.head_dim
    # one shared prefix, or (prefix_len 0) each sequence's own cached tokens
    P = w.prefix_len if w.prefix_len else int((w.context_lens - w.query_lens).sum())
    return {
        "prefix_key": normal((P, Hkv, d), w.dtype, w.seed + 31, device),
        "prefix_value": normal((P, Hkv, d), w.dtype, w.seed + 32, device),
        "query": normal((T, w.num_heads, d), w.dtype, w.seed + 33, device),
        "key": normal((T, Hkv, d), w.dtype, w.seed + 34, device),
        "value": normal((T, Hkv, d), w.dtype, w.seed + 35, device),
    }


def suffix_tensors(w: Workload, device="cpu") -> dict:
    """Keys and values of the tokens each sample appends after its prompt
    (parallel-sampling workload), in sample-major, token-minor order."""
    n = int(w.suffix_lens.sum()) if w.suffix_lens is not None else 0
    return {
        "key": normal((n, w.num_kv_heads, w.head_dim), w.dtype, w.seed + 21, device),
        "value": normal((n, w.num_kv_heads, w.head_dim), w.dtype, w.seed + 22, device),
    }
