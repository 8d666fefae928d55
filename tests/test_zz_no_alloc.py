"""paged_attention_decode_noalloc: the attention entry point for callers that
cannot allocate device memory when they run attention (for example a plugin
called inside a host framework's CUDA-graph capture, or a service whose
device-memory budget is fixed at start-up).  It takes no workspace; the
partition partials live in the library's built-in device array.

Checked through the C ABI against paged_attention_decode with a caller
workspace, on two calls in a row (the array keeps the previous call's
contents).  Both entry points run the same kernels, whose results do not
depend on which CTA takes which work item, so the outputs must be equal bit
for bit -- a stale counter or a scratch overlap would show up here.  The
array is prepared again after check() reported a device-wait timeout, and
that preparation is refused during stream capture.  This file is collected
last so that a run stopping at the first failure has already run every other
test; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cache_139_gb300 as pkv
import workloads
from paged_kv_cache_139_gb300 import _lib

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 16 << 20


def _inputs(dev, S, H, Hkv, d, B, ctx, dtype, seed):
    ctx = np.asarray(ctx, np.int32)
    mb = int(-(-int(ctx.max()) // B))
    nb = S * mb
    q = workloads.normal((S, H, d), dtype, seed).to(dev)
    kc = workloads.normal((nb, Hkv, B, d), dtype, seed + 1).to(dev)
    vc = workloads.normal((nb, Hkv, B, d), dtype, seed + 2).to(dev)
    perm = np.random.default_rng(seed).permutation(nb).astype(np.int32).reshape(S, mb)
    return q, kc, vc, torch.from_numpy(perm).to(dev), torch.from_numpy(ctx).to(dev)


def _noalloc_raw(out, q, kc, vc, bt, cl, partition_size):
    """Direct C-ABI call of paged_attention_decode_noalloc."""
    S, H, d = q.shape
    NB, Hkv, B, _ = kc.shape
    code = pkv.PKV_BF16 if q.dtype == torch.bfloat16 else pkv.PKV_F16
    return _lib.load().paged_attention_decode_noalloc(
        out.data_ptr(), q.data_ptr(), kc.data_ptr(), vc.data_ptr(), bt.data_ptr(), cl.data_ptr(),
        S, bt.shape[1], 0, B, NB, H, Hkv, d, 1.0 / d ** 0.5, partition_size, code,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("S,H,Hkv,d,B,ctx,dtype,P", [
    (2, 32, 8, 128, 16, [4096, 3001], "bf16", 512),             # split contexts: partials in the array
    (4, 8, 8, 64, 32, [1, 700, 64, 2500], "f16", 128),
    (3, 4, 2, 128, 16, [5, 33, 200], "f16", 512),               # one partition each: no scratch needed
])
def test_noalloc_matches_workspace_entry(cuda_device, S, H, Hkv, d, B, ctx, dtype, P):
    q, kc, vc, bt, cl = _inputs(cuda_device, S, H, Hkv, d, B, ctx, dtype, 11 + S)
    ref = torch.empty_like(q)
    ws = pkv.make_workspace(cuda_device, pkv.paged_attention_workspace_size(S, H, Hkv, d, bt.shape[1] * B, P))
    pkv.paged_attention_decode(ref, q, kc, vc, bt, cl, partition_size=P, workspace=ws)
    pkv.check()
    for call in range(2):
        out = torch.full_like(q, float("nan"))
        rc = _noalloc_raw(out, q, kc, vc, bt, cl, P)
        assert rc == 0, _lib.load().pkv_last_error_string()
        pkv.check()
        assert torch.equal(out, ref), f"noalloc call {call} differs from the workspace entry point"


def _latch_and_report_timeout():
    s = torch.cuda.current_stream()
    assert _lib.load().pkv_selftest_wait_timeout(1 << 20, ctypes.c_void_p(s.cuda_stream)) == 0
    with pytest.raises(pkv.PkvError) as e:
        pkv.check()
    assert e.value.status_name == "PKV_ETIMEOUT"


def test_noalloc_prepared_again_after_a_reported_timeout(cuda_device):
    """After check() has reported a device-wait timeout the next call prepares
    the array again (a kernel that gave up may have left its counters
    mid-count) and still matches the workspace entry point bit for bit."""
    S, H, Hkv, d, B, ctx, P = 2, 32, 8, 128, 16, [4096, 3001], 512
    q, kc, vc, bt, cl = _inputs(cuda_device, S, H, Hkv, d, B, ctx, "bf16", 29)
    ref = torch.empty_like(q)
    ws = pkv.make_workspace(cuda_device, pkv.paged_attention_workspace_size(S, H, Hkv, d, bt.shape[1] * B, P))
    pkv.paged_attention_decode(ref, q, kc, vc, bt, cl, partition_size=P, workspace=ws)
    pkv.check()
    _latch_and_report_timeout()
    for call in range(2):
        out = torch.full_like(q, float("nan"))
        assert _noalloc_raw(out, q, kc, vc, bt, cl, P) == 0, _lib.load().pkv_last_error_string()
        pkv.check()
        assert torch.equal(out, ref), f"call {call} after the timeout"


def test_noalloc_preparation_refused_during_capture(cuda_device):
    """A call that must prepare the array (here: the first after a reported
    timeout) inside a CUDA-graph capture returns PKV_EINVAL and records
    nothing; the next call outside capture prepares it and is correct."""
    S, H, Hkv, d, B, ctx, P = 3, 8, 8, 64, 32, [700, 64, 2500], 128
    q, kc, vc, bt, cl = _inputs(cuda_device, S, H, Hkv, d, B, ctx, "f16", 31)
    ref = torch.empty_like(q)
    ws = pkv.make_workspace(cuda_device, pkv.paged_attention_workspace_size(S, H, Hkv, d, bt.shape[1] * B, P))
    pkv.paged_attention_decode(ref, q, kc, vc, bt, cl, partition_size=P, workspace=ws)
    pkv.check()
    # a first call prepares the array, then a reported timeout marks it for preparation again
    out = torch.empty_like(q)
    assert _noalloc_raw(out, q, kc, vc, bt, cl, P) == 0
    pkv.check()
    _latch_and_report_timeout()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    before = pkv.launch_count()
    with torch.cuda.graph(g, stream=side):
        out.zero_()
        rc = _noalloc_raw(out, q, kc, vc, bt, cl, P)
    assert rc == 1                                                # PKV_EINVAL
    assert "capture" in _lib.load().pkv_last_error_string().decode()
    assert pkv.launch_count() == before
    out = torch.full_like(q, float("nan"))
    assert _noalloc_raw(out, q, kc, vc, bt, cl, P) == 0, _lib.load().pkv_last_error_string()
    pkv.check()
    assert torch.equal(out, ref)


def test_noalloc_rejects_sizes_beyond_its_scratch(cuda_device):
    # 256 sequences x 32 heads x 8 partitions of 512 at d 128 need ~34 MB of partials
    S, H, d, B, mb = 256, 32, 128, 16, 256
    assert pkv.paged_attention_workspace_size(S, H, H, d, mb * B, 512) > SCRATCH_BYTES
    q = torch.zeros(S, H, d, dtype=torch.float16, device=cuda_device)
    kc = torch.zeros(4, H, B, d, dtype=torch.float16, device=cuda_device)
    bt = torch.zeros(S, mb, dtype=torch.int32, device=cuda_device)
    cl = torch.ones(S, dtype=torch.int32, device=cuda_device)
    before = pkv.launch_count()
    rc = _noalloc_raw(torch.empty_like(q), q, kc, kc, bt, cl, 512)
    assert rc == 1                                                # PKV_EINVAL
    msg = _lib.load().pkv_last_error_string().decode()
    assert "scratch" in msg and str(SCRATCH_BYTES) in msg
    assert pkv.launch_count() == before                           # nothing was launched
