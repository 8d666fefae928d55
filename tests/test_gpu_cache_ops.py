"""kv_reshape_and_cache and copy_blocks against the oracle, bit for bit, on
the GPU through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_139_gb300 as pkv
import workloads
from cases import Case

pytestmark = pytest.mark.gpu


def _rand(shape, dtype, seed, device):
    return workloads.normal(shape, dtype, seed, "cpu").to(device)


@pytest.mark.parametrize("B", [4, 8, 16, 32, 64, 128])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_cache_write_matches_oracle(cuda_device, B, d, dtype):
    NB, Hkv, T = 24, 3, 50
    rng = np.random.default_rng(B * 1000 + d)
    slots = rng.choice(NB * B, size=T, replace=False).astype(np.int64)
    slots[rng.random(T) < 0.2] = -1                     # padding tokens are skipped
    kc0 = _rand((NB, Hkv, B, d), dtype, 1, "cpu")
    vc0 = _rand((NB, Hkv, B, d), dtype, 2, "cpu")
    key = _rand((T, Hkv, d), dtype, 3, "cpu")
    val = _rand((T, Hkv, d), dtype, 4, "cpu")
    kc, vc = kc0.to(cuda_device), vc0.to(cuda_device)
    pkv.kv_reshape_and_cache(key.to(cuda_device), val.to(cuda_device), kc, vc,
                             torch.from_numpy(slots).to(cuda_device))
    pkv.check()
    ok, ov = oracle.bits16(kc0), oracle.bits16(vc0)
    oracle.cache_write(key, val, ok, ov, slots)
    assert np.array_equal(oracle.bits16(kc), ok)
    assert np.array_equal(oracle.bits16(vc), ov)


def test_cache_write_bad_slot_latches_eindex(cuda_device):
    NB, Hkv, B, d = 4, 2, 16, 64
    kc = torch.zeros(NB, Hkv, B, d, dtype=torch.float16, device=cuda_device)
    vc = torch.zeros_like(kc)
    key = torch.ones(3, Hkv, d, dtype=torch.float16, device=cuda_device)
    slots = torch.tensor([5, NB * B, 7], dtype=torch.int64, device=cuda_device)
    pkv.kv_reshape_and_cache(key, key, kc, vc, slots)
    with pytest.raises(pkv.PkvError) as e:
        pkv.check()
    assert e.value.status_name == "PKV_EINDEX" and "slot" in str(e.value)
    # the good tokens were written, and the status was cleared
    assert bool((kc[0, :, 5] == 1).all()) and bool((kc[0, :, 7] == 1).all())
    assert int((kc != 0).sum()) == 2 * Hkv * d
    pkv.check()


def test_cache_write_empty_is_a_no_op(cuda_device):
    kc = torch.zeros(2, 1, 16, 64, dtype=torch.bfloat16, device=cuda_device)
    before = pkv.launch_count()
    e = torch.empty(0, 1, 64, dtype=torch.bfloat16, device=cuda_device)
    pkv.kv_reshape_and_cache(e, e, kc, kc.clone(), torch.empty(0, dtype=torch.int64, device=cuda_device))
    assert pkv.launch_count() == before
    pkv.check()


@pytest.mark.parametrize("shape", [(40, 32, 16, 128), (33, 8, 16, 128), (64, 2, 4, 64), (10, 1, 128, 64)])
def test_copy_blocks_matches_oracle(cuda_device, shape):
    NB = shape[0]
    rng = np.random.default_rng(NB)
    perm = rng.permutation(NB)
    n = NB // 3
    pairs = np.stack([perm[:n], perm[n:2 * n]], axis=1).astype(np.int32)   # distinct dst, disjoint from src
    pkv.validate_copy_pairs(pairs, NB)
    c0 = _rand(shape, "f16", 9, "cpu")
    c = c0.to(cuda_device)
    pkv.copy_blocks(c, torch.from_numpy(pairs).to(cuda_device))
    pkv.check()
    oc = oracle.bits16(c0)
    oracle.copy_blocks(oc, pairs)
    assert np.array_equal(oracle.bits16(c), oc)


def test_copy_blocks_bad_pair_latches_eindex(cuda_device):
    c = torch.arange(4 * 256, dtype=torch.float32, device=cuda_device).view(4, 256).to(torch.float16)
    c0 = c.clone()
    pairs = torch.tensor([[0, 1], [2, 9]], dtype=torch.int32, device=cuda_device)
    pkv.copy_blocks(c, pairs)
    with pytest.raises(pkv.PkvError) as e:
        pkv.check()
    assert e.value.status_name == "PKV_EINDEX"
    assert torch.equal(c[1], c0[0]) and torch.equal(c[2:], c0[2:])


def test_sampling_cow_flow_bit_exact(cuda_device):
    """Parallel sampling over shared prompt blocks: fork, suffix appends with
    copy-on-write through copy_blocks, then the decode token; every cache
    byte, table, slot and copy pair equals the oracle's."""
    w = workloads.sampling(num_prompts=6, max_suffix=40)
    c = Case(w, cuda_device)
    c.check_allocator()
    assert len(c.sfx_pairs) + len(c.plan.pairs) == 6 * 3      # 3 copies per prompt, 1 in-place writer
    k, v = c.gpu_cache_blocks()
    ok, ov = c.oracle_caches()
    assert np.array_equal(k, ok) and np.array_equal(v, ov)


def test_sampling_full_prompt_needs_no_copy(cuda_device):
    """A prompt that fills its blocks exactly shares only full blocks: no
    copy-on-write at all."""
    w = workloads.sampling(num_prompts=4, max_suffix=20, partial_last_block=False)
    c = Case(w, cuda_device)
    c.check_allocator()
    assert len(c.sfx_pairs) == 0 and len(c.plan.pairs) == 0


def test_cow_full_size_pairs(cuda_device):
    """The full parallel-sampling workload: 64 prompts x 4 samples gives 192
    copy pairs; the copied blocks equal their sources bit for bit (sampled
    prompts checked against the oracle)."""
    w = workloads.sampling()
    c = Case(w, cuda_device, subset=list(range(0, 256, 37)))
    c.check_allocator()
    assert len(c.sfx_pairs) + len(c.plan.pairs) == 192
    k, v = c.gpu_cache_blocks()
    ok, ov = c.oracle_caches()
    assert np.array_equal(k, ok) and np.array_equal(v, ov)
