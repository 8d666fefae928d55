"""Benchmark of the paged decode hot path on GB300.

One step = one decode iteration of one layer over the whole batch: the
copy-on-write block copies (if the step has any), the slot-mapped write of
the batch's new keys and values, and paged decode attention over every
sequence's block table (including the partition merge).  Host allocation is
done once before timing.  The metric is effective KV-read bandwidth:
sum over sequences of context_len x 2 x kv_heads x head_dim x 2 bytes,
divided by the step time.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload llama7b]
                    [--block-size B] [--head-dim D] [--partition-size P] [--impl reference]

--workload prefix times the prompt phase instead: after a shared cached
prefix, the copy-on-write of its last block, the cache write of every
request's own tokens and causal prompt-phase attention, in TFLOP/s
(--block-size, --head-dim, --kv-heads and --dtype vary its shape).

Prints one JSON line (rank 0).  Under torchrun each rank runs an independent
replica (a different seed) on its own GPU; the value is all ranks' bytes over
the slowest rank's time.
"""
from __future__ import annotations

import argparse
import dataclasses
import json
import math
import os
import pathlib
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = pathlib.Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

import workloads  # noqa: E402

METRIC = "paged decode attention effective KV-read GB/s and % of GB300 HBM peak"
PREFILL_METRIC = "prompt-phase paged attention TFLOP/s (causal, after a shared prefix)"
BEAM_METRIC = "beam-search decode effective KV-read GB/s (all beams, shared blocks counted per beam)"
SWAP_METRIC = "swap GB/s (KV blocks GPU -> pinned host -> GPU, both directions)"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
L2_FLUSH_BYTES = 512 << 20
L2_BYTES = 129e6                 # GB300 L2 (nominal)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="llama7b",
                    choices=["tiny", "opt13b", "llama7b", "sampling", "longgqa", "prefix", "swap", "beam"])
    ap.add_argument("--beam-width", type=int, default=4)
    ap.add_argument("--block-size", type=int, default=16)
    ap.add_argument("--head-dim", type=int, default=128, choices=[64, 128])
    ap.add_argument("--partition-size", type=int, default=-1)
    ap.add_argument("--num-seqs", type=int, default=0, help="opt13b / llama7b: batch size (0: the workload's)")
    ap.add_argument("--kv-heads", type=int, default=0, help="prefix workload: kv heads (0: MHA)")
    ap.add_argument("--dtype", default="", choices=["", "f16", "bf16"], help="prefix workload: cache dtype")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


def make_workload(args, rank: int) -> workloads.Workload:
    kw = {}
    if args.workload == "llama7b":
        kw["block_size"] = args.block_size
        kw["head_dim"] = args.head_dim
    if args.workload in ("llama7b", "opt13b") and args.num_seqs > 0:
        kw["num_seqs"] = args.num_seqs
    if args.workload == "swap":
        kw["block_size"] = args.block_size
    if args.workload == "prefix":
        kw["block_size"] = args.block_size
        kw["head_dim"] = args.head_dim
        if args.kv_heads:
            kw["num_kv_heads"] = args.kv_heads
        if args.dtype:
            kw["dtype"] = args.dtype
    if args.workload == "beam":
        kw["width"] = args.beam_width
    w = workloads.by_name(args.workload, **kw)
    if rank:
        w = workloads.by_name(args.workload, seed=w.seed + 7919 * rank, **kw) if args.workload != "tiny" else w
    if args.partition_size >= 0:
        w.partition_size = args.partition_size
    return w


# -- measured peaks and profile figures --------------------------------------------

def hbm_peak():
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        try:
            d = json.loads(p.read_text())
            for k in ("hbm_gbs", "hbm_GBps", "hbm"):
                if k in d and d[k]:
                    return float(d[k]), "measured"
        except (ValueError, TypeError):
            pass
    return FALLBACK_HBM_GBS, "fallback"


def tensor_peak():
    """Dense 16-bit tensor peak for a kernel timed alone (TFLOP/s)."""
    p = ROOT / "MEASURED_PEAKS.json"
    if p.exists():
        try:
            d = json.loads(p.read_text())
            for k in ("bf16_tflops", "bf16_TFLOPs", "bf16"):
                if k in d and d[k]:
                    return float(d[k]), "measured"
        except (ValueError, TypeError):
            pass
    return FALLBACK_BF16_TFLOPS, "fallback"


def profile_traffic(workload_name: str, version: int):
    """DRAM bytes per launch of the attention kernel from a committed ncu
    summary (a line 'traffic_bytes_per_launch[<workload>@<library version>]: N'),
    else None: a figure taken on another kernel version does not count."""
    for f in sorted((ROOT / "profiles").glob("*.md")):
        for line in f.read_text().splitlines():
            key = f"traffic_bytes_per_launch[{workload_name}@{version}]:"
            if line.strip().startswith(key):
                try:
                    return float(line.split(":", 1)[1].split()[0])
                except ValueError:
                    return None
    return None


# -- clocks ------------------------------------------------------------------------

class ClockSampler:
    FIELDS = "index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active," \
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown," \
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap"

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# -- the CPU baseline (the oracle as it stands) -------------------------------------

SAMPLE_KV_BYTES = 1 << 30        # KV held by the CPU baseline's sample of sequences


def decode_config(w: workloads.Workload, kv_bytes: int, world: int) -> dict:
    """The workload as both arms print it (identical keys and values)."""
    if kv_bytes >= 4 * L2_BYTES:
        l2 = (f"inputs larger than L2: {kv_bytes / 1e9:.2f} GB of KV per step against a 129 MB L2, steps back to "
              f"back (the GPU arm's l2_flushed_each_step repeats them with a {L2_FLUSH_BYTES >> 20} MiB memset "
              f"before each)")
    else:
        l2 = f"flushed before every step ({L2_FLUSH_BYTES >> 20} MiB memset, outside the timed events)"
    return {**w.describe(), "l2": l2, "kv_bytes_per_step": kv_bytes, "parallelism": f"replicas x{world}"}


def sample_sequences(w: workloads.Workload, ctx: np.ndarray, max_bytes: int = SAMPLE_KV_BYTES) -> list:
    """A seeded sample of whole sequences holding at most max_bytes of KV
    (at least one)."""
    sel, tot = [], 0
    for s in np.random.default_rng(w.seed).permutation(w.num_seqs):
        b = int(ctx[s]) * w.kv_bytes_per_token
        if sel and tot + b > max_bytes:
            break
        sel.append(int(s))
        tot += b
    return sel


def compact_tables(w: workloads.Workload, sel, tables: np.ndarray, ctx: np.ndarray, slots):
    """The blocks the sampled sequences reference (and their new tokens'
    slots), renumbered in their original order: the physical block ids kept,
    the new tables and slots.  Ids only; the caller fetches the blocks."""
    B = w.block_size
    need = set()
    for s in sel:
        need.update(int(x) for x in tables[s][: -(-int(ctx[s]) // B)] if x >= 0)
        if slots is not None and slots[s] >= 0:
            need.add(int(slots[s]) // B)
    blocks = np.array(sorted(need), np.int64)
    remap = {int(b): i for i, b in enumerate(blocks)}
    t2 = np.full((len(sel), tables.shape[1]), -1, np.int32)
    for i, s in enumerate(sel):
        for j, x in enumerate(tables[s]):
            if x >= 0 and int(x) in remap:
                t2[i, j] = remap[int(x)]
    sl2 = None
    if slots is not None:
        sl2 = np.array([remap[int(slots[s]) // B] * B + int(slots[s]) % B if slots[s] >= 0 else -1 for s in sel],
                       np.int64)
    return blocks, t2, np.asarray(ctx, np.int32)[sel], sl2


def cpu_baseline(w: workloads.Workload, kc: np.ndarray, vc: np.ndarray, q, key, value, tables: np.ndarray,
                 ctx: np.ndarray, slots, what: str, budget_s=12.0):
    """The oracle, as it stands, on a compact sample of whole sequences (pools
    kc/vc of raw 16-bit patterns, tables/ctx/slots and q/key/value of the
    sampled sequences only): the new tokens' cache write, then attention of
    one sequence (all heads) per call, in a seeded order, for about half the
    budget on one thread and half on every host core (the C oracle runs
    outside the GIL)."""
    import oracle
    oracle.cache_write(key, value, kc, vc, slots)
    n = len(ctx)
    bpt = w.kv_bytes_per_token
    G = w.num_heads // w.num_kv_heads
    order = np.random.default_rng(w.seed + 1).permutation(n)

    def one(i):
        which = [(int(i), h) for h in range(w.num_heads)]
        oracle.paged_attention(q, kc, vc, tables, ctx, w.dtype, which=which)
        return int(ctx[i]) * bpt                         # every kv head's K and V read once

    done_bytes, t0, seqs = 0, time.perf_counter(), 0
    for i in order:
        done_bytes += one(i)
        seqs += 1
        if time.perf_counter() - t0 > budget_s / 2:
            break
    dt1 = time.perf_counter() - t0
    single = done_bytes / dt1 / 1e9
    from concurrent.futures import ThreadPoolExecutor
    cores = os.cpu_count() or 1
    par_bytes, t0, pseqs = 0, time.perf_counter(), 0
    with ThreadPoolExecutor(max_workers=cores) as ex:
        k = 0
        while time.perf_counter() - t0 < budget_s / 2:
            batch = [order[(k + j) % n] for j in range(cores)]
            k += cores
            par_bytes += sum(ex.map(one, batch))
            pseqs += len(batch)
    dt2 = time.perf_counter() - t0
    return {"value": par_bytes / dt2 / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{what}; {pseqs} sequence calls (all {w.num_heads} heads, G={G}) on {cores} threads in "
                      f"{dt2:.1f} s; single thread: {seqs} sequences in {dt1:.1f} s",
            "single_thread_value": single}


def gpu_arm_cpu_baseline(w: workloads.Workload, eng, q, key, value, plan, budget_s=12.0):
    """The CPU baseline of our arm: the sampled sequences' blocks copied from
    the device pools (their state after the timed steps; the oracle writes the
    new tokens again at the same slots, which leaves them unchanged)."""
    import oracle
    sel = sample_sequences(w, plan.context_lens)
    blocks, t2, c2, sl2 = compact_tables(w, sel, plan.tables, plan.context_lens, plan.slots)
    idx = torch.from_numpy(blocks).to(eng.key_cache.device)
    kc = oracle.bits16(eng.key_cache.index_select(0, idx))
    vc = oracle.bits16(eng.value_cache.index_select(0, idx))
    si = torch.tensor(sel, device=q.device)
    kvb = int(c2.astype(np.int64).sum()) * w.kv_bytes_per_token
    what = (f"{len(sel)} of {w.num_seqs} sequences ({kvb / 1e9:.2f} GB of KV), seeded, their blocks copied from "
            f"the device pool")
    return cpu_baseline(w, kc, vc, q.index_select(0, si).cpu(), key.index_select(0, si).cpu(),
                        value.index_select(0, si).cpu(), t2, c2, sl2, what, budget_s)


def reference_plan(w: workloads.Workload):
    """The decode step's block tables, context lengths and new-token slots as
    the oracle's allocator lays them out: every sequence created with its
    cached tokens (or, for parallel sampling, each prompt forked into its
    samples, which append their suffixes), then one append each."""
    import oracle
    ref = oracle.RefAllocator(w.num_blocks, w.block_size, workloads.free_order(w.num_blocks, w.seed))
    if w.prompt_lens is None:
        ids = [ref.seq_new(int(c) - 1) for c in w.context_lens]
    else:
        ids = []
        for plen in w.prompt_lens:
            root = ref.seq_new(int(plen))
            ids += [root] + [ref.fork(root) for _ in range(w.samples_per_prompt - 1)]
        ref.append_batch([sid for i, sid in enumerate(ids) for _ in range(int(w.suffix_lens[i]))])
    slots, _ = ref.append_batch(ids)
    tables = np.full((len(ids), w.max_blocks_per_seq), -1, np.int32)
    for i, sid in enumerate(ids):
        bt = ref.block_table(sid)
        tables[i, :len(bt)] = bt
    ctx = np.array([ref.seq_len(s) for s in ids], np.int32)
    return tables, ctx, np.asarray(slots, np.int64)


def run_reference(args, rank: int, world: int):
    if rank != 0:
        return
    w = make_workload(args, 0)
    if w.query_lens is not None:
        return run_reference_prefill(args, w)
    if args.workload == "swap":
        return run_reference_swap(args, w)
    if args.workload == "beam":
        print(json.dumps({"impl": "reference", "unavailable": "reference arm runs the decode workloads (tiny, "
                          "opt13b, llama7b, sampling, longgqa), the prompt phase and swapping"}))
        return
    tables, ctx, slots = reference_plan(w)
    sel = sample_sequences(w, ctx)
    blocks, t2, c2, sl2 = compact_tables(w, sel, tables, ctx, slots)
    # the sample's pool: N(0, 1) values of the workload's type, only the blocks it uses
    import oracle
    shape = (len(blocks), w.num_kv_heads, w.block_size, w.head_dim)
    kc = oracle.bits16(workloads.normal(shape, w.dtype, w.seed + 14))
    vc = oracle.bits16(workloads.normal(shape, w.dtype, w.seed + 15))
    t = workloads.tensors(dataclasses.replace(w, num_blocks=0), "cpu")
    si = torch.tensor(sel)
    kvb = int(c2.astype(np.int64).sum()) * w.kv_bytes_per_token
    what = f"{len(sel)} of {w.num_seqs} sequences ({kvb / 1e9:.2f} GB of KV), seeded, their blocks generated"
    per_step = max(2.0, 60.0 / max(1, args.steps + args.warmup))
    vals = []
    for i in range(args.warmup + args.steps):
        cb = cpu_baseline(w, kc, vc, t["query"][si], t["key"][si], t["value"][si], t2, c2, sl2, what,
                          budget_s=per_step)
        if i >= args.warmup:
            vals.append(cb)
    v = statistics.median([c["value"] for c in vals])
    total_bytes = int(ctx.astype(np.int64).sum()) * w.kv_bytes_per_token
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_bytes / (v * 1e9) * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": decode_config(w, total_bytes, args.gpus),
            "kernel": "oracle (fp64 C, CPU)",
            "cpu_baseline": {**vals[-1], "value": v},
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def sampling_setup(eng, w: workloads.Workload, dev):
    """Parallel sampling: each prompt's sequence is forked into its samples
    (shared blocks), every sample appends its suffix -- the first append into
    the shared, partly filled last block copies it (copy_blocks) -- and the
    suffix keys and values are written.  Returns the sample ids and the
    measured copy-on-write step."""
    import paged_kv_cache_139_gb300 as pkv
    n = w.samples_per_prompt
    ids = []
    for plen in w.prompt_lens:
        root = eng.new_sequence(int(plen))
        ids += [root] + [eng.fork(root) for _ in range(n - 1)]
    order = []
    for i, sid in enumerate(ids):
        order += [sid] * int(w.suffix_lens[i])
    plan = eng.plan_step(order)
    dev_plan = eng.upload(plan)
    sfx = workloads.suffix_tensors(w, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    # the copies are idempotent until the suffix is written: one untimed run
    # (first launch of the kernel), then the timed one
    eng.copy_on_write(dev_plan.pairs)
    flush.zero_()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    eng.copy_on_write(dev_plan.pairs)
    b.record()
    eng.write(sfx["key"], sfx["value"], dev_plan.slots)
    torch.cuda.synchronize(dev)
    pkv.check()
    npairs = int(plan.pairs.shape[0])
    block_bytes = eng.num_kv_heads * eng.block_size * eng.head_dim * eng.key_cache.element_size()
    ms = a.elapsed_time(b)
    moved = 2 * 2 * npairs * block_bytes            # K and V, read + write
    return ids, {"pairs": npairs, "block_bytes": block_bytes, "ms": ms,
                 "gbs": moved / (ms * 1e-3) / 1e9 if ms > 0 else None, "bytes_moved": moved,
                 "note": "both copy_blocks launches (K and V) of the suffix step, L2 flushed before"}


def time_loop(stream, fn, n: int, flush=None) -> float:
    """Mean milliseconds per call of fn on `stream`: n calls back to back
    between two events, or (flush given) an event pair around each call with
    the L2 flushed before it (the flush also keeps the GPU busy while the host
    enqueues the call, so no host latency lands between the events)."""
    if flush is None:
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(n):
            fn()
        b.record(stream)
        b.synchronize()
        return a.elapsed_time(b) / n
    ev = []
    for _ in range(n):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        ev.append((a, b))
    ev[-1][1].synchronize()
    return statistics.fmean(a.elapsed_time(b) for a, b in ev)


def aggregate(t_step_ms: float, nbytes: float, dist=None, device="cpu"):
    """Whole-job figures over the ranks: the slowest rank's step time and the
    sum of every rank's bytes (host control traffic only; no data moves)."""
    if dist is None:
        return t_step_ms, float(nbytes)
    t = torch.tensor([t_step_ms], dtype=torch.float64, device=device)
    b = torch.tensor([float(nbytes)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(b, op=dist.ReduceOp.SUM)
    return float(t.item()), float(b.item())


# -- our arm -----------------------------------------------------------------------------

def run_ours(args, rank: int, world: int):
    import paged_kv_cache_139_gb300 as pkv
    from paged_kv_cache_139_gb300.engine import PagedKVCache

    dist = None
    if world > 1:
        import torch.distributed as dist
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    w = make_workload(args, rank)
    t_gpu = workloads.tensors(w, device=dev)
    order = workloads.free_order(w.num_blocks, w.seed)
    eng = PagedKVCache(w.num_blocks, w.num_kv_heads, w.head_dim, w.block_size, w.torch_dtype, dev,
                       w.max_blocks_per_seq, order, key_cache=t_gpu["key_cache"], value_cache=t_gpu["value_cache"])
    cow = None
    if w.prompt_lens is not None:
        ids, cow = sampling_setup(eng, w, dev)
    else:
        ids = [eng.new_sequence(int(c) - 1) for c in w.context_lens]
    plan = eng.plan_step(ids)
    step = eng.upload(plan)
    q, key, value = t_gpu["query"], t_gpu["key"], t_gpu["value"]
    out = torch.empty_like(q)
    P = w.partition_size
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    kv_bytes = int(plan.context_lens.astype(np.int64).sum()) * w.kv_bytes_per_token

    # the step's C-ABI calls, marshalled once (a decode loop reuses its buffers)
    prep = eng.prepare(q, key, value, step, out, partition_size=P)

    def device_step():
        prep()

    # Clocks are sampled from the start of the warm-up to the end of the e2e
    # leg (the GPU runs the same step throughout); the warm-up runs at least W
    # steps and at least one second so that the sampler sees the GPU under load.
    clk = ClockSampler(dev.index).__enter__()
    t_w = time.perf_counter()
    n_w = 0
    while n_w < args.warmup or time.perf_counter() - t_w < 1.0:
        flush.zero_()
        device_step()
        n_w += 1
        if n_w % 16 == 0:
            torch.cuda.synchronize(dev)
    pkv.check()

    # Timed region: K steps.  A batch whose KV bytes exceed the L2 several
    # times runs its steps back to back between two events (each step reads
    # what the previous one evicted); a smaller one flushes the L2 before every
    # step, with an event pair around each.
    back_to_back = kv_bytes >= 4 * L2_BYTES
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    launches0 = pkv.launch_count()
    wall0 = time.perf_counter()
    t_step = time_loop(stream, prep, args.steps, None if back_to_back else flush)
    wall = time.perf_counter() - wall0
    if dist:
        dist.barrier()
    launches = pkv.launch_count() - launches0
    pkv.check()
    # the attention call alone (the step minus its copy-on-write copies), same policy
    t_attn = time_loop(stream, prep.back, args.steps, None if back_to_back else flush)
    # both with the L2 flushed before every step (an event pair around each)
    t_step_fl = time_loop(stream, prep, args.steps, flush)
    t_attn_fl = time_loop(stream, prep.back, args.steps, flush)
    pkv.check()

    # paged vs contiguous placement of the same batch (identity block tables)
    nblk = -(-plan.context_lens.astype(np.int64) // w.block_size)
    ident = np.full_like(plan.tables, -1)
    base = 0
    for i, n in enumerate(nblk):
        ident[i, :n] = np.arange(base, base + n)
        base += n
    ident_dev = torch.from_numpy(ident).to(dev)
    istep = type(step)(step.slots, step.pairs, ident_dev, step.context_lens, step.max_context_len)
    iprep = eng.prepare(q, key, value, istep, torch.empty_like(out), partition_size=P)
    iprep.attend()
    t_contig = time_loop(stream, iprep.attend, max(3, args.steps // 2), None if back_to_back else flush)
    pkv.check()

    # end to end through the public API from pinned host buffers: the step's inputs
    # staged in one pinned buffer (one host-to-device copy), the output read back
    e2e = None
    if not args.no_e2e:
        from paged_kv_cache_139_gb300.engine import StagedInputs
        src = {"q": q, "key": key, "value": value, "slots": torch.from_numpy(plan.slots),
               "tables": torch.from_numpy(plan.tables), "ctx": torch.from_numpy(plan.context_lens)}
        stg = StagedInputs({n: (tuple(x.shape), x.dtype) for n, x in src.items()}, dev)
        for n, x in src.items():
            stg.host[n].copy_(x.cpu())
        h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        d = stg.dev
        dstep = type(step)(d["slots"], step.pairs, d["tables"], d["ctx"], step.max_context_len)
        from paged_kv_cache_139_gb300.engine import GraphStep
        gstep = GraphStep(stg, lambda st: eng.prepare(d["q"], d["key"], d["value"], dstep, out, partition_size=P,
                                                      stream=st), out, h_out)
        h2d = stg.nbytes
        d2h = h_out.numel() * h_out.element_size()
        times = []
        for i in range(args.warmup + args.steps):
            flush.zero_()
            torch.cuda.synchronize(dev)
            t0 = time.perf_counter()
            gstep.replay()
            torch.cuda.synchronize(dev)
            if i >= args.warmup:
                times.append(time.perf_counter() - t0)
        t_e2e = sum(times) / len(times)
        e2e = {"value": kv_bytes / t_e2e / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": t_e2e * 1e3,
               "note": "engine.GraphStep: one staged host-to-device copy, the step's calls and the output "
                       "read-back replayed as one CUDA graph; host time from before the replay to after the sync"}
        pkv.check()

    clk.__exit__(None, None, None)
    t_step_max, total_bytes = aggregate(t_step, kv_bytes, dist, dev)
    if rank != 0:
        return

    peak, peak_src = hbm_peak()
    value = total_bytes / (t_step_max * 1e-3) / 1e9
    attn_gbs = kv_bytes / (t_attn * 1e-3) / 1e9
    traffic = profile_traffic(args.workload if args.workload != "llama7b"
                              else f"llama7b_B{w.block_size}_d{w.head_dim}", pkv.version())
    # the block-size trade-off: slots held by the batch vs tokens stored
    held = int((-(-plan.context_lens.astype(np.int64) // w.block_size)).sum()) * w.block_size
    frag = {"slots_held": held, "tokens": int(plan.context_lens.sum()),
            "internal_fragmentation_pct": 100.0 * (1.0 - plan.context_lens.sum() / held)}
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t_step_max, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "kv_dtype": w.dtype, "data": "synthetic",
        "config": decode_config(w, kv_bytes, world),
        "partition_size": pkv.paged_attention_partition_size(
            w.num_seqs, w.num_heads, w.num_kv_heads, w.head_dim, step.max_context_len, P),
        "pct_of_hbm_peak": 100.0 * value / world / peak,
        "tokens_per_s": w.num_seqs * world / (t_step_max * 1e-3),
        "roofline": {"bound": "hbm", "achieved": attn_gbs, "peak": peak, "unit": "GB/s", "frac": attn_gbs / peak,
                     "traffic": traffic, "kernel": ("paged_attention_decode_write (new tokens written in the launch, "
                                                    "partition kernel + merge)" if prep._fused else
                                                    "paged_attention_decode (partition kernel + merge)"),
                     "peak_source": f"{peak_src} {'MEASURED_PEAKS.json hbm_gbs' if peak_src == 'measured' else '6.8 TB/s'}",
                     "ms_per_launch": t_attn},
        "paged_overhead": {"contiguous_ms": t_contig, "paged_ms": t_attn,
                           "slowdown_pct": 100.0 * (t_attn / t_contig - 1.0)},
        "l2_flushed_each_step": {"ms_per_step": t_step_fl, "value": kv_bytes / (t_step_fl * 1e-3) / 1e9,
                                 "attention_ms": t_attn_fl,
                                 "attention_gbs": kv_bytes / (t_attn_fl * 1e-3) / 1e9},
        "block_fill": frag,
        "gpu_launches": launches,
        "clocks": {**clk.summary(), "window": "warm-up + timed + e2e legs"},
        "wall_s_timed_region": wall,
        "e2e": e2e,
    }
    if cow is not None:
        B = w.block_size
        distinct = len({int(b) for row, n in zip(plan.tables, plan.context_lens) for b in row[:-(-int(n) // B)]})
        unique = distinct * B * w.kv_bytes_per_token
        line["sharing"] = {"copy_blocks": cow, "unique_kv_bytes_per_step": unique,
                           "unique_gbs": unique / (t_step_max * 1e-3) / 1e9,
                           "note": "unique bytes count every distinct physical block in full"}
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = gpu_arm_cpu_baseline(w, eng, q, t_gpu["key"], t_gpu["value"], plan)
    print(json.dumps(line), flush=True)


# -- prompt phase after a shared prefix --------------------------------------------------

def prefill_flops(ctx: np.ndarray, n: np.ndarray, H: int, d: int) -> float:
    """Algorithmic FLOPs of causal prompt-phase attention: new token j of a
    sequence (position ctx - n + j) sees ctx - n + j + 1 keys, each costing
    2d for q.k and 2d for the weighted value, per query head."""
    ctx = ctx.astype(np.float64)
    n = n.astype(np.float64)
    keys = n * (ctx - n + 1) + n * (n - 1) / 2
    return float(4.0 * d * H * keys.sum())


def prefill_cpu_baseline(w, t, tables, ctx, qs, cached_slots, pairs, slots, budget_s=12.0):
    import oracle
    shape = (w.num_blocks, w.num_kv_heads, w.block_size, w.head_dim)
    kc = np.zeros(shape, np.uint16)
    vc = np.zeros(shape, np.uint16)
    oracle.cache_write(t["prefix_key"], t["prefix_value"], kc, vc, cached_slots)
    if len(pairs):
        oracle.copy_blocks(kc, pairs)
        oracle.copy_blocks(vc, pairs)
    oracle.cache_write(t["key"], t["value"], kc, vc, slots)
    q = t["query"].cpu()
    rng = np.random.default_rng(w.seed)
    T = int(qs[-1])
    seq_of = np.repeat(np.arange(w.num_seqs), np.diff(qs))

    def one(tok):
        which = [(tok, h) for h in range(w.num_heads)]
        oracle.paged_prefill(q, kc, vc, tables, ctx, qs, w.dtype, which=which)
        s = seq_of[tok]
        pos = int(ctx[s]) - int(qs[s + 1] - qs[s]) + (tok - int(qs[s]))
        return 4.0 * w.head_dim * w.num_heads * (pos + 1)

    # random new tokens (all heads), half the budget on one thread, half on every host core
    # (the C oracle runs outside the GIL)
    flops, rows, t0 = 0.0, 0, time.perf_counter()
    while time.perf_counter() - t0 < budget_s / 2:
        flops += one(int(rng.integers(T)))
        rows += w.num_heads
    dt1 = time.perf_counter() - t0
    single = flops / dt1 / 1e12
    from concurrent.futures import ThreadPoolExecutor
    cores = os.cpu_count() or 1
    pflops, prows, t0 = 0.0, 0, time.perf_counter()
    with ThreadPoolExecutor(max_workers=cores) as ex:
        while time.perf_counter() - t0 < budget_s / 2:
            pflops += sum(ex.map(one, [int(x) for x in rng.integers(T, size=cores)]))
            prows += cores * w.num_heads
    dt2 = time.perf_counter() - t0
    return {"value": pflops / dt2 / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{prows} (token, head) rows of {T * w.num_heads} (random new tokens, all heads) on {cores} "
                      f"threads in {dt2:.1f} s; single thread: {rows} rows in {dt1:.1f} s",
            "single_thread_value": single}


def run_reference_prefill(args, w):
    """The oracle's prompt-phase attention, as it stands, on bounded samples of
    the shared-prefix workload (same allocator plan as our arm)."""
    import oracle
    B = w.block_size
    ref = oracle.RefAllocator(w.num_blocks, B, workloads.free_order(w.num_blocks, w.seed))
    root = ref.seq_new(w.prefix_len)
    rt = ref.block_table(root)
    cached = np.array([rt[i // B] * B + i % B for i in range(w.prefix_len)], np.int64)
    kids = [ref.fork(root) for _ in range(w.num_seqs)]
    slots, pairs = ref.append_batch(np.repeat(np.asarray(kids, np.int32), w.query_lens))
    tables = np.full((w.num_seqs, w.max_blocks_per_seq), -1, np.int32)
    for i, k in enumerate(kids):
        bt = ref.block_table(k)
        tables[i, :len(bt)] = bt
    ctx = np.array([ref.seq_len(k) for k in kids], np.int32)
    qs = np.concatenate([[0], np.cumsum(w.query_lens)]).astype(np.int32)
    t = workloads.prefill_tensors(w, "cpu")
    per_step = max(2.0, 60.0 / max(1, args.steps + args.warmup))
    vals = []
    for i in range(args.warmup + args.steps):
        cb = prefill_cpu_baseline(w, t, tables, ctx, qs, cached, pairs, np.asarray(slots, np.int64),
                                  budget_s=per_step)
        if i >= args.warmup:
            vals.append(cb)
    v = statistics.median([c["value"] for c in vals])
    flops = prefill_flops(ctx, w.query_lens, w.num_heads, w.head_dim)
    line = {"impl": "reference", "metric": PREFILL_METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": flops / (v * 1e12) * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {**w.describe(), "prefix_len": w.prefix_len,
                                            "kernel": "oracle (fp64 C, CPU)"},
            "cpu_baseline": {**vals[-1], "value": v},
            "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def run_reference_swap(args, w):
    """The oracle's block copy between two pools, as it stands, on a bounded
    sample of the swap workload's blocks."""
    import oracle
    t = workloads.tensors(w, "cpu")
    kb = oracle.bits16(t["key_cache"][: min(w.num_blocks, 2048)])
    dst = np.zeros_like(kb)
    n = kb.shape[0]
    block_bytes = kb[0].nbytes
    prs = np.stack([np.arange(n), np.arange(n)[::-1]], 1).astype(np.int32)
    vals = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        oracle.copy_blocks_between(dst, kb, prs)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            vals.append(n * block_bytes / dt / 1e9)
    v = statistics.median(vals)
    line = {"impl": "reference", "metric": SWAP_METRIC, "value": v, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": n * block_bytes / (v * 1e9) * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8", "data": "synthetic",
            "config": {**w.describe(), "kernel": "oracle (C, CPU)"},
            "cpu_baseline": {"value": v, "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": f"{n} blocks of {block_bytes} B per step, single thread"},
            "e2e": {"value": v, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def run_prefill(args, rank: int, world: int):
    """One step: the copy-on-write copies of the shared prefix's last block,
    the cache write of every request's own tokens, and prompt-phase attention
    of those tokens over the paged cache."""
    import paged_kv_cache_139_gb300 as pkv
    from paged_kv_cache_139_gb300.engine import PagedKVCache

    dist = None
    if world > 1:
        import torch.distributed as dist
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    w = make_workload(args, rank)
    t = workloads.prefill_tensors(w, device=dev)
    eng = PagedKVCache(w.num_blocks, w.num_kv_heads, w.head_dim, w.block_size, w.torch_dtype, dev,
                       w.max_blocks_per_seq, workloads.free_order(w.num_blocks, w.seed))
    B = w.block_size
    root = eng.new_sequence(w.prefix_len)
    rt = eng.alloc.block_table(root)
    cached_slots = np.array([rt[i // B] * B + i % B for i in range(w.prefix_len)], np.int64)
    eng.write(t["prefix_key"], t["prefix_value"], torch.from_numpy(cached_slots).to(dev))
    kids = [eng.fork(root) for _ in range(w.num_seqs)]
    plan = eng.plan_prefill(kids, w.query_lens)
    step = eng.upload_prefill(plan)
    q, key, value = t["query"], t["key"], t["value"]
    out = torch.empty_like(q)
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flops = prefill_flops(plan.context_lens, np.diff(plan.query_start), w.num_heads, w.head_dim)
    T = int(plan.query_start[-1])
    prep = eng.prepare_prefill(q, key, value, step, out)

    clk = ClockSampler(dev.index).__enter__()
    t_w, n_w = time.perf_counter(), 0
    while n_w < args.warmup or time.perf_counter() - t_w < 1.0:
        flush.zero_()
        prep()
        n_w += 1
        if n_w % 16 == 0:
            torch.cuda.synchronize(dev)
    pkv.check()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize(dev)
    launches0 = pkv.launch_count()
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush.zero_()
        ev[i][0].record(stream)
        prep.copy()
        prep.write()
        ev[i][1].record(stream)
        prep.attend()
        ev[i][2].record(stream)
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - wall0
    if dist:
        dist.barrier()
    launches = pkv.launch_count() - launches0
    pkv.check()
    t_step = statistics.fmean(a.elapsed_time(c) for a, _, c in ev)
    t_attn = statistics.fmean(b.elapsed_time(c) for _, b, c in ev)
    t_front = statistics.fmean(a.elapsed_time(b) for a, b, _ in ev)

    e2e = None
    if not args.no_e2e:
        from paged_kv_cache_139_gb300.engine import StagedInputs
        src = {"q": q, "key": key, "value": value, "slots": torch.from_numpy(plan.slots),
               "tables": torch.from_numpy(plan.tables), "ctx": torch.from_numpy(plan.context_lens),
               "qs": torch.from_numpy(plan.query_start)}
        stg = StagedInputs({n: (tuple(x.shape), x.dtype) for n, x in src.items()}, dev)
        for n, x in src.items():
            stg.host[n].copy_(x.cpu())
        h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        d = stg.dev
        dstep = type(step)(d["slots"], step.pairs, d["tables"], d["ctx"], d["qs"], step.max_query_len)
        from paged_kv_cache_139_gb300.engine import GraphStep
        gstep = GraphStep(stg, lambda st: eng.prepare_prefill(d["q"], d["key"], d["value"], dstep, out, stream=st),
                          out, h_out)
        h2d = stg.nbytes
        d2h = h_out.numel() * h_out.element_size()
        times = []
        for i in range(args.warmup + args.steps):
            flush.zero_()
            torch.cuda.synchronize(dev)
            t0 = time.perf_counter()
            gstep.replay()
            torch.cuda.synchronize(dev)
            if i >= args.warmup:
                times.append(time.perf_counter() - t0)
        t_e2e = statistics.fmean(times)
        e2e = {"value": flops / t_e2e / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": t_e2e * 1e3,
               "note": "engine.GraphStep: one staged host-to-device copy, the step's calls and the output "
                       "read-back replayed as one CUDA graph; host time from before the replay to after the sync"}
        pkv.check()
    clk.__exit__(None, None, None)
    t_step_max, total_flops = aggregate(t_step, flops, dist, dev)
    if rank != 0:
        return
    peak, peak_src = tensor_peak()
    achieved = flops / (t_attn * 1e-3) / 1e12
    esz = 2
    write_bytes = 2 * 2 * T * w.num_kv_heads * w.head_dim * esz + 8 * T
    copy_bytes = 2 * 2 * len(plan.pairs) * w.num_kv_heads * B * w.head_dim * esz
    line = {
        "metric": PREFILL_METRIC, "value": total_flops / (t_step_max * 1e-3) / 1e12, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_step_max,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "kv_dtype": w.dtype,
        "data": "synthetic",
        "config": {**w.describe(), "prefix_len": w.prefix_len, "new_tokens": T,
                   "l2": f"flushed before every step ({L2_FLUSH_BYTES >> 20} MiB memset, outside the timed events)",
                   "flops_per_step": flops, "parallelism": f"replicas x{world}"},
        "tokens_per_s": T * world / (t_step_max * 1e-3),
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": profile_traffic("prefix", pkv.version()),
                     "kernel": "paged_attention_prefill (tcgen05, TMEM accumulators)",
                     "peak_source": f"{peak_src} {'MEASURED_PEAKS.json bf16_tflops' if peak_src == 'measured' else '1.9 PFLOP/s bf16 burst'}",
                     "ms_per_launch": t_attn},
        "write_and_copy": {"ms": t_front, "copy_pairs": int(len(plan.pairs)), "bytes": write_bytes + copy_bytes,
                           "gbs": (write_bytes + copy_bytes) / (t_front * 1e-3) / 1e9},
        "gpu_launches": launches,
        "clocks": {**clk.summary(), "window": "warm-up + timed + e2e legs"},
        "wall_s_timed_region": wall,
        "e2e": e2e,
    }
    if not args.no_cpu_baseline:
        tc = workloads.prefill_tensors(w, "cpu")
        line["cpu_baseline"] = prefill_cpu_baseline(w, tc, plan.tables, plan.context_lens, plan.query_start,
                                                    cached_slots, plan.pairs, plan.slots)
    print(json.dumps(line), flush=True)


# -- beam search --------------------------------------------------------------------------

def run_beam(args, rank: int, world: int):
    """A beam search over every request: each step plans the next beams on
    the host (fork / prune / copy-on-write), then the device copies the
    written shared blocks, writes the new tokens and runs decode attention
    over all beams.  The search first runs `steps0` untimed steps so that
    the beams' histories branch and share."""
    import paged_kv_cache_139_gb300 as pkv
    from paged_kv_cache_139_gb300.engine import PagedKVCache

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    w = make_workload(args, rank)
    k = w.samples_per_prompt
    B = w.block_size
    rng = np.random.default_rng(w.seed)
    kc = workloads.normal((w.num_blocks, w.num_kv_heads, B, w.head_dim), w.dtype, w.seed + 14, dev)
    vc = workloads.normal((w.num_blocks, w.num_kv_heads, B, w.head_dim), w.dtype, w.seed + 15, dev)
    eng = PagedKVCache(w.num_blocks, w.num_kv_heads, w.head_dim, B, w.torch_dtype, dev, w.max_blocks_per_seq,
                       workloads.free_order(w.num_blocks, w.seed), key_cache=kc, value_cache=vc)
    beams = [[eng.new_sequence(int(p_))] for p_ in w.context_lens]
    nq = w.num_seqs * k
    q = workloads.normal((nq, w.num_heads, w.head_dim), w.dtype, w.seed + 11, dev)
    key = workloads.normal((nq, w.num_kv_heads, w.head_dim), w.dtype, w.seed + 12, dev)
    value = workloads.normal((nq, w.num_kv_heads, w.head_dim), w.dtype, w.seed + 13, dev)
    out = torch.empty_like(q)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def host_step():
        all_new, slots, pairs = [], [], []
        for r in range(w.num_seqs):
            par = workloads.beam_parents(rng, len(beams[r]), k)
            new, sl, pr = eng.alloc.beam_step(beams[r], par)
            beams[r] = new
            all_new += new
            slots.append(sl)
            pairs.append(pr)
        s_ = np.asarray(all_new, np.int32)
        tables, ctx = eng.alloc.build_block_tables(s_, w.max_blocks_per_seq)
        from paged_kv_cache_139_gb300.engine import StepPlan
        return StepPlan(s_, np.concatenate(slots), np.concatenate(pairs).reshape(-1, 2).astype(np.int32), tables, ctx)

    def memory():
        used = eng.alloc.blocks_in_use()
        unshared = sum(-(-eng.alloc.seq_len(b) // B) for g in beams for b in g)
        return used, unshared

    steps0 = 64
    mem_trace, host_ms, dev_ms, kvb = [], [], [], []
    launches = 0
    clk = ClockSampler(dev.index).__enter__()
    for i in range(steps0 + args.warmup + args.steps):
        t0 = time.perf_counter()
        plan = host_step()
        t_host = time.perf_counter() - t0
        step = eng.upload(plan)
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        l0 = pkv.launch_count()
        a.record(stream)
        eng.copy_on_write(step.pairs)
        eng.write(key, value, step.slots)
        eng.attend(q, step, out=out)
        b.record(stream)
        if i >= steps0 + args.warmup:
            torch.cuda.synchronize(dev)
            launches += pkv.launch_count() - l0
            dev_ms.append(a.elapsed_time(b))
            host_ms.append(t_host * 1e3)
            kvb.append(int(plan.context_lens.astype(np.int64).sum()) * w.kv_bytes_per_token)
            mem_trace.append(memory())
    torch.cuda.synchronize(dev)
    pkv.check()
    clk.__exit__(None, None, None)
    used = np.array([m[0] for m in mem_trace], np.float64)
    unshared = np.array([m[1] for m in mem_trace], np.float64)
    t_dev = statistics.fmean(dev_ms)
    value = statistics.fmean(kvb) / (t_dev * 1e-3) / 1e9
    peak, peak_src = hbm_peak()
    line = {
        "metric": BEAM_METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t_dev, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "kv_dtype": w.dtype, "data": "synthetic",
        "config": {**w.describe(), "beam_width": k, "beams": nq, "untimed_steps_before": steps0 + args.warmup,
                   "l2": f"flushed before every step ({L2_FLUSH_BYTES >> 20} MiB memset, outside the timed events)"},
        "memory": {"blocks_in_use": float(used.mean()), "blocks_without_sharing": float(unshared.mean()),
                   "saving_pct": float(100.0 * (1.0 - used.sum() / unshared.sum())),
                   "note": "blocks held with block sharing vs every beam holding its own copy of its history"},
        "host_beam_step_ms": statistics.fmean(host_ms),
        "roofline": {"bound": "hbm", "achieved": value, "peak": peak, "unit": "GB/s", "frac": value / peak,
                     "traffic": None, "kernel": "copy_blocks + kv_reshape_and_cache + paged_attention_decode",
                     "peak_source": f"{peak_src}", "note": "shared prompt blocks are read once per beam; L2 serves the repeats"},
        "gpu_launches": launches,
        "clocks": {**clk.summary(), "window": "the whole search"},
        "e2e": None,
    }
    print(json.dumps(line), flush=True)


# -- swapping between the GPU pool and a pinned host pool ----------------------------------

def run_swap(args, rank: int, world: int):
    """One step: every sequence's K and V blocks swapped out to the host pool
    and back in (two swap_blocks launches each way), the pairs planned once."""
    import paged_kv_cache_139_gb300 as pkv
    from paged_kv_cache_139_gb300.engine import HostKVPool, PagedKVCache

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", 0)))
    torch.cuda.set_device(dev)
    w = make_workload(args, rank)
    t = workloads.tensors(w, device=dev)
    eng = PagedKVCache(w.num_blocks, w.num_kv_heads, w.head_dim, w.block_size, w.torch_dtype, dev,
                       w.max_blocks_per_seq, workloads.free_order(w.num_blocks, w.seed),
                       key_cache=t["key_cache"], value_cache=t["value_cache"])
    host = HostKVPool(w.num_blocks, w.num_kv_heads, w.head_dim, w.block_size, w.torch_dtype)
    ids = [eng.new_sequence(int(c)) for c in w.context_lens]
    # the device copies of one round trip: plan the moves once (block ids only)
    probe_g = pkv.BlockAllocator(w.num_blocks, w.block_size, workloads.free_order(w.num_blocks, w.seed))
    pids = [probe_g.seq_new(int(c)) for c in w.context_lens]
    probe_c = pkv.BlockAllocator(w.num_blocks, w.block_size)
    cids, out_pairs = probe_g.move_group(probe_c, pids)
    _, in_pairs = probe_c.move_group(probe_g, cids)
    po = torch.from_numpy(out_pairs).to(dev)
    pi = torch.from_numpy(in_pairs).to(dev)
    nblk = out_pairs.shape[0]
    block_bytes = w.num_kv_heads * w.block_size * w.head_dim * 2
    moved = 2 * nblk * block_bytes                  # K and V, one direction
    stream = torch.cuda.current_stream(dev)

    def out_copy():
        pkv.swap_blocks(host.key_cache, eng.key_cache, po, stream)
        pkv.swap_blocks(host.value_cache, eng.value_cache, po, stream)

    def in_copy():
        pkv.swap_blocks(eng.key_cache, host.key_cache, pi, stream)
        pkv.swap_blocks(eng.value_cache, host.value_cache, pi, stream)

    clk = ClockSampler(dev.index).__enter__()
    for _ in range(max(3, args.warmup)):
        out_copy()
        in_copy()
    torch.cuda.synchronize(dev)
    pkv.check()
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    launches0 = pkv.launch_count()
    for i in range(args.steps):
        ev[i][0].record(stream)
        out_copy()
        ev[i][1].record(stream)
        in_copy()
        ev[i][2].record(stream)
    torch.cuda.synchronize(dev)
    launches = pkv.launch_count() - launches0
    pkv.check()
    t_out = statistics.fmean(a.elapsed_time(b) for a, b, _ in ev)
    t_in = statistics.fmean(b.elapsed_time(c) for _, b, c in ev)
    # the link's own rate: one contiguous copy of the same bytes each way (copy engine)
    hbuf = torch.empty(moved, dtype=torch.uint8).pin_memory()
    dbuf = torch.empty(moved, dtype=torch.uint8, device=dev)
    ce = []
    for i in range(3 + args.steps):
        a, b, c = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        a.record(stream)
        hbuf.copy_(dbuf, non_blocking=True)
        b.record(stream)
        dbuf.copy_(hbuf, non_blocking=True)
        c.record(stream)
        ce.append((a, b, c))
    torch.cuda.synchronize(dev)
    ce_d2h = statistics.median(a.elapsed_time(b) for a, b, _ in ce[3:])
    ce_h2d = statistics.median(b.elapsed_time(c) for _, b, c in ce[3:])
    peak = 2 * moved / ((ce_d2h + ce_h2d) * 1e-3) / 1e9
    # end to end through the engine: the group moves (host bookkeeping) and the copies
    e2e_t = []
    gids = ids
    for i in range(args.warmup + args.steps):
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        hids, _ = eng.swap_out(gids, host)
        gids, _ = eng.swap_in(hids, host)
        torch.cuda.synchronize(dev)
        if i >= args.warmup:
            e2e_t.append(time.perf_counter() - t0)
    pkv.check()
    clk.__exit__(None, None, None)
    t_e2e = statistics.fmean(e2e_t)
    value = 2 * moved / ((t_out + t_in) * 1e-3) / 1e9
    line = {
        "metric": SWAP_METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t_out + t_in, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "u8", "kv_dtype": w.dtype, "data": "synthetic",
        "config": {**w.describe(), "blocks_moved": nblk, "block_bytes": block_bytes,
                   "bytes_per_direction": moved, "host_pool": "pinned host memory, addressed by the kernel"},
        "swap_out": {"ms": t_out, "gbs": moved / (t_out * 1e-3) / 1e9},
        "swap_in": {"ms": t_in, "gbs": moved / (t_in * 1e-3) / 1e9},
        "roofline": {"bound": "link", "achieved": value, "peak": peak, "unit": "GB/s", "frac": value / peak,
                     "traffic": profile_traffic("swap", pkv.version()) if w.block_size == 16 else None,
                     "traffic_note": "DRAM bytes of one device-to-host launch (keys), from profiles/",
                     "kernel": "swap_blocks",
                     "peak_source": "one contiguous cudaMemcpyAsync of the same bytes each way, measured here",
                     "copy_engine_d2h_gbs": moved / (ce_d2h * 1e-3) / 1e9,
                     "copy_engine_h2d_gbs": moved / (ce_h2d * 1e-3) / 1e9},
        "gpu_launches": launches,
        "clocks": {**clk.summary(), "window": "warm-up + timed + e2e legs"},
        "e2e": {"value": 2 * moved / t_e2e / 1e9, "unit": "GB/s", "h2d_bytes_per_step": moved,
                "d2h_bytes_per_step": moved, "ms_per_step": t_e2e * 1e3,
                "note": "engine.swap_out + swap_in: the allocator moves and the copies"},
    }
    if not args.no_cpu_baseline:
        import oracle
        kb = oracle.bits16(t["key_cache"][: min(w.num_blocks, 2048)])
        dst = np.zeros_like(kb)
        n = kb.shape[0]
        prs = np.stack([np.arange(n), np.arange(n)[::-1]], 1).astype(np.int32)
        t0 = time.perf_counter()
        reps = 0
        while time.perf_counter() - t0 < 5.0:
            oracle.copy_blocks_between(dst, kb, prs)
            reps += 1
        dt = time.perf_counter() - t0
        line["cpu_baseline"] = {"value": reps * n * block_bytes / dt / 1e9, "unit": "GB/s", "cores": 1,
                                "kind": "oracle", "sample": f"{reps} x {n} blocks of {block_bytes} B copied "
                                                            f"between two host pools, single thread, {dt:.1f} s"}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
        dist.init_process_group("nccl")
    if args.impl == "reference":
        run_reference(args, rank, world)
    elif args.workload == "prefix":
        run_prefill(args, rank, world)
    elif args.workload == "swap":
        run_swap(args, rank, world)
    elif args.workload == "beam":
        run_beam(args, rank, world)
    else:
        run_ours(args, rank, world)
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
