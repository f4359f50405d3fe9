#!/usr/bin/env python
"""Benchmark of the paged KV-cache decode hot path on one GB300.

One step = one decode layer-step of the whole hot path over a seeded synthetic
batch: copy-on-write pairs are applied (copy_blocks, when the workload has
any), the new token of every sequence is written into its slot and the decode
attention (+ its split merge) runs over every sequence's context.  By default
the write is part of the attention call (paged_attention_decode_append: the
newest token's K/V taken from the step's input and stored into its slot by
the same kernel); with --step two-call, or for the shared-prefix entry point,
reshape_and_cache writes it first.  The block tables and slot mappings come
from the C++ block manager (set-up, host).

Default workload: OPT-13B-shaped decode layer (64 sequences, 40 heads x 128,
fp16 K/V, block size 16, lognormal context lengths with median 300 clipped to
[1, 2048]); 40 per-layer pools are rotated so consecutive steps read cold K/V
(each layer's K/V is larger than the 129 MB L2).

Metric: achieved HBM GB/s of algorithmic bytes, where the bytes of a step are
sum_s ctx_s * H * D * 2 (K and V) * 2 B + q and out (2 * S * H * D * 2 B) +
the block-table entries read (sum_s ceil(ctx_s / B) * 4 B) + context_lens
(4 S B) + the new-token write (2 * S * H * D * 2 B read and the same written).

``--impl reference`` times the CPU fp64 oracle (the only reference there is)
on the host cores over a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_kv_cache_05_gb300 import workloads as W  # noqa: E402

METRIC = "paged-attn decode: achieved HBM GB/s (% of GB300 peak), us/layer-step at OPT-13B"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_NOTE = "fallback (MEASURED_PEAKS.json absent): one earlier GB300 copy measurement"


# ------------------------------------------------------------------ helpers
def read_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, copy burst)"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_NOTE


def kernel_source_digest(files=("decode_kernel.cuh", "decode_api.cu", "pkv_internal.h")) -> str:
    import hashlib
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "paged_kv_cache_05_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


PREFILL_SOURCES = ("prefill.cu", "pkv_internal.h")


def profiled_traffic(workload: str, profile: str = None, sources=None):
    """DRAM bytes per launch from the committed ncu summary (the decode
    kernel's for the workload, or the named profile), if it was taken on the
    current kernel source (else None)."""
    p = os.path.join(ROOT, "profiles", profile or ("paged_decode_main_%s.md" % workload))
    if not os.path.exists(p):
        return None
    kv = {}
    for line in open(p):
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            kv[k.strip()] = v.strip().strip("`")
    digest = kernel_source_digest(sources) if sources else kernel_source_digest()
    if kv.get("kernel_source_sha256_16") != digest:
        return None
    try:
        return float(kv["dram_bytes_per_launch_full_size"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi SM clock / throttle-reason sampling while the GPU is busy."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ workload
class Workload:
    """Device-resident inputs of one workload plus the algorithmic byte counts."""

    def __init__(self, name: str, device, partition=None, block_size=None, layers=None,
                 placement: str = "scattered", decode: str = "auto", step: str = "append"):
        import torch
        import paged_kv_cache_05_gb300 as pkv
        self.pkv = pkv
        spec = W.SPECS[name]
        self.spec = spec
        self.name = name
        B = block_size or spec.block_size
        self.B = B
        S, H, D = spec.num_seqs, spec.num_heads, spec.head_dim
        self.S, self.H, self.D = S, H, D
        self.partition = spec.partition_size if partition is None else partition
        ctx = W.context_lens(spec)
        self.ctx_host = ctx
        nb = W.pool_blocks(spec, ctx, B)
        self.nb = nb
        dt = W.torch_dtype(spec.dtype)
        self.dtype = spec.dtype
        # block manager: every sequence holds ctx-1 tokens, then one decode
        # step reserves the slot of its new token (position ctx-1)
        bm = pkv.BlockManager(nb, B, spec.seed)
        ids = list(range(S))
        pairs = np.zeros((0, 2), np.int32)
        if name == "shared_prefix":
            p_len, s_len = W.prompt_and_suffix_lens(spec)
            g = spec.extra["per_group"]
            for gi in range(len(p_len)):
                bm.add_sequence(gi * g, int(p_len[gi]))
                for c in range(1, g):
                    bm.fork(gi * g, gi * g + c)
            # all but the last suffix token of each sequence, round-robin; the
            # copy-on-write pairs this emits (first suffix token of the first
            # five samples of a group whose prompt ends mid-block) are applied
            # by copy_blocks in every timed step
            got = []
            for t in range(int(s_len.max()) - 1):
                act = [s for s in ids if t < s_len[s] - 1]
                sl, pr = bm.append_slots(act)
                got.append(pr)
            slots, pr = bm.append_slots(ids)
            got.append(pr)
            pairs = np.concatenate(got).astype(np.int32).reshape(-1, 2)
        else:
            for s in ids:
                bm.add_sequence(s, int(ctx[s]) - 1)
            slots, pairs = bm.append_slots(ids)
        self.max_blocks = max(1, max(-(-int(c) // B) for c in ctx))
        tables, ctx2 = bm.export(ids, self.max_blocks)
        assert np.array_equal(ctx2, ctx)
        self.placement = placement
        if placement == "contiguous":
            # every sequence's blocks consecutive in the pool, in logical order
            # (the contiguous-allocation baseline the pages compare against)
            if name == "shared_prefix":
                raise SystemExit("bench.py: contiguous placement is not defined with sharing")
            nxt = 0
            tables = np.full_like(tables, -1)
            for s_ in ids:
                n = -(-int(ctx[s_]) // B)
                tables[s_, :n] = np.arange(nxt, nxt + n)
                nxt += n
            pos = ctx.astype(np.int64) - 1
            slots = tables[np.arange(len(ids)), pos // B].astype(np.int64) * B + pos % B
            pairs = np.zeros((0, 2), np.int32)
        self.tables_host = tables
        self.slots_host = slots
        self.pairs_host = pairs
        self.bm = bm
        dev = device
        self.layers = layers or spec.layers
        self.kc, self.vc = [], []
        if name == "long":
            # an 80 GB pool, uninitialised except the blocks the batch uses
            kc = torch.empty((nb, H, B, D), dtype=dt, device=dev)
            vc = torch.empty((nb, H, B, D), dtype=dt, device=dev)
            used = torch.from_numpy(np.unique(np.concatenate(
                [tables[s, :-(-int(ctx[s]) // B)] for s in ids]))).long().to(dev)
            for pool, seed in ((kc, spec.seed + 1), (vc, spec.seed + 2)):
                vals = W.device_normal((used.numel(), H, B, D), spec.dtype, seed, dev)
                pool.index_copy_(0, used, vals)
                del vals
            self.kc.append(kc)
            self.vc.append(vc)
        else:
            for layer in range(self.layers):
                self.kc.append(W.device_normal((nb, H, B, D), spec.dtype,
                                               spec.seed * 1000 + 2 * layer, dev))
                self.vc.append(W.device_normal((nb, H, B, D), spec.dtype,
                                               spec.seed * 1000 + 2 * layer + 1, dev))
        self.q = W.device_normal((S, H, D), spec.dtype, spec.seed * 1000 + 900, dev)
        self.k_new = W.device_normal((S, H, D), spec.dtype, spec.seed * 1000 + 901, dev)
        self.v_new = W.device_normal((S, H, D), spec.dtype, spec.seed * 1000 + 902, dev)
        self.out = torch.empty_like(self.q)
        self.tables = torch.from_numpy(tables).to(dev)
        self.ctx = torch.from_numpy(ctx).to(dev)
        self.slots = torch.from_numpy(slots).to(dev)
        self.pairs = torch.from_numpy(pairs).to(dev)
        # the shared-prefix entry point (each group's common prefix read once)
        # for the workload whose sequences are forks of shared prompts
        self.shared = decode == "shared" or (decode == "auto" and name == "shared_prefix")
        self.decode_fn = (pkv.paged_attention_decode_shared if self.shared
                          else pkv.paged_attention_decode)
        # the new token written by the attention call itself (not with the
        # shared-prefix entry point)
        self.append = step == "append" and not self.shared
        if self.shared:
            self.ws = torch.empty(pkv.decode_shared_workspace_size(
                S, H, D, B, self.max_blocks, self.partition), dtype=torch.uint8, device=dev)
        else:
            self.ws = pkv.alloc_workspace(S, H, D, B, self.max_blocks, self.partition, dev)
        self.scale = spec.scale
        e = 2
        self.kv_bytes = int(ctx.astype(np.int64).sum()) * H * D * 2 * e
        self.attn_bytes = (self.kv_bytes + 2 * S * H * D * e
                           + sum(-(-int(c) // B) for c in ctx) * 4 + 4 * S)
        self.reshape_bytes = 2 * (2 * S * H * D * e)
        self.copy_bytes = len(pairs) * 2 * 2 * H * B * D * e
        self.step_bytes = self.attn_bytes + self.reshape_bytes + self.copy_bytes
        self.launches_per_step = ((2 if self.append else 3) + (1 if len(pairs) else 0)
                                  + (1 if self.shared else 0))
        self.unique_kv_bytes = None
        if name == "shared_prefix":
            blocks = set()
            for s in ids:
                blocks.update(tables[s, :-(-int(ctx[s]) // B)].tolist())
            self.unique_kv_bytes = len(blocks) * H * B * D * 2 * e

    def step(self, i: int, append=None):
        pkv = self.pkv
        layer = i % self.layers
        kc, vc = self.kc[layer], self.vc[layer]
        if len(self.pairs_host):
            pkv.copy_blocks(kc, vc, self.pairs)
        if self.append if append is None else append:
            pkv.paged_attention_decode_append(self.out, self.q, self.k_new, self.v_new, kc, vc,
                                              self.tables, self.ctx, self.scale, self.partition,
                                              self.ws)
            return
        pkv.reshape_and_cache(self.k_new, self.v_new, kc, vc, self.slots)
        self.decode_fn(self.out, self.q, kc, vc, self.tables, self.ctx, self.scale,
                       self.partition, self.ws)

    def attention(self, i: int):
        layer = i % self.layers
        self.decode_fn(self.out, self.q, self.kc[layer], self.vc[layer], self.tables, self.ctx,
                       self.scale, self.partition, self.ws)

    def describe(self) -> str:
        sp = self.spec
        c = self.ctx_host
        return ("%s: %d seqs x %d heads x %d, %s K/V, B=%d, ctx %d..%d (sum %d), pool %d blocks"
                " x %d layer pool(s), split %s, %s placement%s" % (
                    self.name, self.S, self.H, self.D, sp.dtype, self.B, int(c.min()),
                    int(c.max()), int(c.sum()), self.nb, self.layers,
                    "balanced" if self.partition == 0 else "%d tokens" % self.partition,
                    self.placement,
                    ", shared prefixes read once (paged_attention_decode_shared)"
                    if self.shared else ""))


# ------------------------------------------------------------------ oracle leg
def host_case(name: str, block_size=None):
    """The workload's block tables and context lengths built on the host
    only, by the oracle's own model of the block manager (the same seeded
    policy and the same sequence of operations as the device workload: every
    sequence holds ctx - 1 tokens, then one decode step appends its newest;
    shared prefixes are forked and their suffixes appended round-robin).  No
    product library is loaded."""
    from oracle.block_manager import BlockManagerModel
    spec = W.SPECS[name]
    B = block_size or spec.block_size
    ctx = W.context_lens(spec)
    m = BlockManagerModel(W.pool_blocks(spec, ctx, B), B, spec.seed)
    S = spec.num_seqs
    if name == "shared_prefix":
        p_len, s_len = W.prompt_and_suffix_lens(spec)
        g = spec.extra["per_group"]
        for gi in range(len(p_len)):
            m.add_sequence(gi * g, int(p_len[gi]))
            for c in range(1, g):
                m.fork(gi * g, gi * g + c)
        for t in range(int(s_len.max())):
            for s_ in range(S):
                if t < s_len[s_]:
                    m.append_slot(s_)
    else:
        for s_ in range(S):
            m.add_sequence(s_, int(ctx[s_]) - 1)
        for s_ in range(S):
            m.append_slot(s_)
    tables = [m.block_table(s_) for s_ in range(S)]
    assert [m.context_len(s_) for s_ in range(S)] == [int(c) for c in ctx]
    return dict(spec=spec, B=B, ctx=ctx, tables=tables)


def oracle_sample(hc: dict, seqs=None, tile_blocks: int = 256):
    """Oracle inputs for a subset of a host case's sequences (all heads):
    their tables renumbered over the blocks they use, and pools of seeded
    host values (tile_blocks random blocks repeated over the blocks in use:
    the oracle's cost does not depend on the values)."""
    spec, B, ctx = hc["spec"], hc["B"], hc["ctx"]
    pick = list(range(spec.num_seqs)) if seqs is None else sorted(seqs)
    used = sorted(set(int(b) for s in pick for b in hc["tables"][s]))
    remap = {b: i for i, b in enumerate(used)}
    H, D = spec.num_heads, spec.head_dim
    n = len(used)
    kc, vc = (np.resize(W.normal_words((min(n, tile_blocks), H, B, D), spec.dtype, spec.seed,
                                       40 + k), (n, H, B, D)) for k in range(2))
    q = W.normal_words((len(pick), H, D), spec.dtype, spec.seed, 42)
    mb = max(1, max(len(hc["tables"][s]) for s in pick))
    bt = np.full((len(pick), mb), -1, np.int32)
    for i, s in enumerate(pick):
        bt[i, :len(hc["tables"][s])] = [remap[int(b)] for b in hc["tables"][s]]
    cl = ctx[pick].astype(np.int32)
    e = 2
    nbytes = (int(cl.astype(np.int64).sum()) * H * D * 2 * e + 2 * len(pick) * H * D * e
              + sum(-(-int(c) // B) for c in cl) * 4 + 4 * len(pick))
    return dict(q=q, kc=kc, vc=vc, bt=bt, cl=cl, bytes=nbytes, seqs=len(pick), heads=H,
                scale=spec.scale, dtype=spec.dtype)


def run_oracle(sample, threads):
    import oracle
    dt = oracle.F16 if sample["dtype"] == "f16" else oracle.BF16
    t0 = time.perf_counter()
    oracle.paged_attention_decode_threaded(sample["q"], sample["kc"], sample["vc"], sample["bt"],
                                           sample["cl"], float(np.float32(sample["scale"])), dt,
                                           threads=threads)
    return time.perf_counter() - t0


def sized_sample(hc: dict, budget_s: float, threads: int):
    """The largest length-spread subset of sequences whose oracle pass is
    expected to fit in budget_s (calibrated on a small subset), at least one."""
    ctx, S = hc["ctx"], hc["spec"].num_seqs
    order = [int(i) for i in np.argsort(ctx, kind="stable")]
    probe = sorted(order[::max(1, S // 8)])
    p = oracle_sample(hc, probe)
    t = run_oracle(p, threads)
    per_byte = t / p["bytes"] * max(1, min(threads, len(probe))) / max(1, min(threads, S))
    allowed = budget_s / max(per_byte, 1e-15)
    take = []
    spec = hc["spec"]
    for k in range(1, S + 1):
        sel = sorted(order[::max(1, S // k)])[:k]
        b = sum(int(ctx[s]) for s in sel) * spec.num_heads * spec.head_dim * 4
        if b > allowed and take:
            break
        take = sel
    return take

def max_over_ranks(x: float, dist) -> float:
    """The maximum of x over all ranks (x itself without a process group)."""
    if dist is None:
        return x
    import torch
    if dist.get_backend() == "nccl":
        dev = torch.device("cuda", torch.cuda.current_device())
    else:
        dev = torch.device("cpu")
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(bytes_per_rank: int, seconds: float, world: int) -> float:
    """Weak scaling: every rank processes the same per-rank work; the job's
    rate is all ranks' bytes over the slowest rank's time, in GB/s."""
    return world * bytes_per_rank / seconds / 1e9


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


# ------------------------------------------------------------------ main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--op", choices=["step", "swap", "sharing", "prefill", "layout"],
                    default="step",
                    help="step: the decode layer-step (default); swap: block swap GPU<->CPU; "
                         "sharing: memory saved by block sharing (host only); prefill: the "
                         "prompt phase; layout: paged against contiguous-layout decode")
    ap.add_argument("--workload", default="opt13b", choices=sorted(W.SPECS))
    ap.add_argument("--dtype", choices=["f16", "bf16"], default="f16",
                    help="storage type of q and the caches for --op prefill")
    ap.add_argument("--partition", type=int, default=None,
                    help="split length in tokens (0 = balanced); default: the workload's")
    ap.add_argument("--block-size", type=int, default=None)
    ap.add_argument("--layers", type=int, default=None)
    ap.add_argument("--placement", choices=["scattered", "contiguous"], default="scattered",
                    help="physical block placement: the block manager's scattered free list, "
                         "or every sequence's blocks consecutive (contiguous baseline)")
    ap.add_argument("--decode", choices=["auto", "plain", "shared"], default="auto",
                    help="decode entry point: plain, shared (groups of sequences sharing "
                         "prefix blocks read them once), auto = shared for the shared-prefix "
                         "workload")
    ap.add_argument("--step", choices=["append", "two-call"], default="append",
                    help="how a step writes the new tokens: inside the attention call "
                         "(paged_attention_decode_append, default) or by reshape_and_cache "
                         "before it")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--roofline-seconds", type=float, default=0.5,
                    help="length of the roofline region (back-to-back attention calls; at "
                         "least --steps calls)")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the other workloads' block (long, short, shared prefix, prompt "
                         "phase)")
    args = ap.parse_args()

    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)

    if args.op == "sharing":
        from paged_kv_cache_05_gb300 import build
        build.build()
        print(json.dumps({"op": "sharing", "metric": "KV blocks saved by sharing (fraction)",
                          "block_size": 16, "data": "synthetic (seeded)",
                          "results": sharing_savings()}), flush=True)
        return
    if args.impl == "reference":
        return reference_arm(args, world, rank, dist)
    if args.op == "swap":
        return bench_swap(args)
    if args.op == "prefill":
        return bench_prefill(args)
    if args.op == "layout":
        return bench_layout(args)

    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    from paged_kv_cache_05_gb300 import build
    build.build()
    wl = Workload(args.workload, device, args.partition, args.block_size, args.layers,
                  args.placement, args.decode, args.step)
    stream = torch.cuda.current_stream()

    K = args.steps
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(device.index if device.index is not None else 0)
    sampler.start()
    time.sleep(0.3)                       # let the sampler start before the GPU work
    # the W warm-up steps run right before the timed region, so that the GPU
    # is not left idle (clocks ramping down) between them
    for i in range(args.warmup):
        wl.step(i)
    torch.cuda.synchronize()
    if wl.pkv.get_device_error() != 0:
        raise SystemExit("bench.py: device error bits after warm-up")
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    # timed region 1: K whole steps back to back (no events between kernels,
    # which would break the programmatic-dependent-launch chain)
    t_start.record(stream)
    for i in range(K):
        wl.step(args.warmup + i)
    t_end.record(stream)
    torch.cuda.synchronize()
    # timed region 2: back-to-back launches of the dominant operation alone
    # (at least K, and at least --roofline-seconds of them, so that the
    # clock record covers it), bracketed by events on the launching stream:
    # its average duration per launch
    n_attn = attention_calls(wl, K, args.roofline_seconds, stream)
    a_start, a_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a_start.record(stream)
    for i in range(n_attn):
        wl.attention(args.warmup + i)
    a_end.record(stream)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    clocks = sampler.stop()
    ms_total = max_over_ranks(t_start.elapsed_time(t_end), dist)
    attn_avg = a_start.elapsed_time(a_end) / n_attn
    ms_step = ms_total / K
    value = whole_job_rate(wl.step_bytes, ms_step * 1e-3, world)

    # ---- the cache operations on their own, and a per-call median of the
    # attention (each call bracketed by its own events, which also breaks the
    # programmatic launch chain, so these calls cannot overlap their neighbours)
    parts = measure_parts(wl, device, args.warmup)
    if wl.append:
        # the same step as two calls (reshape_and_cache, then the attention), K steps
        for i in range(3):
            wl.step(i, append=False)
        torch.cuda.synchronize()
        t_start.record(stream)
        for i in range(K):
            wl.step(args.warmup + i, append=False)
        t_end.record(stream)
        torch.cuda.synchronize()
        parts["two_call_step_us"] = round(t_start.elapsed_time(t_end) / K * 1e3, 2)
        parts["two_call_step_note"] = ("the same step with the new tokens written by "
                                       "reshape_and_cache before the attention call")

    # ---- end to end: host (pinned) inputs -> C ABI -> host output, every step
    e2e = api = None
    if args.e2e_steps > 0:
        api = measure_e2e_api(wl, args.e2e_steps, device, dist)
        api["seconds"] = max_over_ranks(api["seconds"], dist)
        e2e = measure_e2e(wl, args.e2e_steps, device, dist)
        e2e["seconds"] = max_over_ranks(e2e["seconds"], dist)

    if wl.pkv.get_device_error() != 0:
        raise SystemExit("bench.py: device error bits after the timed region")

    peak, peak_note = read_peaks()
    achieved = wl.attn_bytes / (attn_avg * 1e-3) / 1e9
    # the committed capture is of the workload as specified (its block size,
    # the balanced split, scattered blocks)
    traffic = (profiled_traffic(args.workload)
               if args.block_size in (None, W.SPECS[args.workload].block_size)
               and args.partition in (None, W.SPECS[args.workload].partition_size)
               and args.placement == "scattered" else None)
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5),
        "us_per_layer_step": round(ms_step * 1e3, 2),
        "attention_us_per_call": round(attn_avg * 1e3, 2),
        "pct_of_peak": round(100 * value / world / peak, 1),
        "seq_heads_per_s": round(world * wl.S * wl.H / (ms_step * 1e-3), 1),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded; N(0,1) K/V/q, lognormal/uniform context lengths)",
        "config": {
            "workload": wl.describe(),
            "storage": wl.dtype,
            "num_seqs": wl.S, "num_heads": wl.H, "head_dim": wl.D, "block_size": wl.B,
            "partition_size": wl.partition,
            "algorithmic_bytes_per_step": wl.step_bytes,
            "attention_bytes_per_call": wl.attn_bytes,
            "l2": "inputs larger than L2: %.0f MB of K/V per layer, %d layer pools rotated" % (
                wl.attn_bytes / 1e6, wl.layers),
            "parallelism": "replicas" if world > 1 else "1 GPU",
        },
        "roofline": {
            "bound": "hbm",
            "kernel": "paged_attention_decode (paged_decode_main + paged_decode_merge)",
            "achieved": round(achieved, 1),
            "peak": peak,
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": traffic,
            "peak_source": peak_note,
        },
        "gpu_launches": K * wl.launches_per_step,
        "gpu_launches_note": "timed region 1: %d per step (%s); region 2 adds %d attention "
                             "launches (2 kernels each) for the roofline" % (
                                 wl.launches_per_step,
                                 "copy_blocks, " * bool(len(wl.pairs_host))
                                 + "reshape_and_cache, " * (not wl.append)
                                 + "paged_decode_groups, " * wl.shared
                                 + "paged_decode_main, paged_decode_merge",
                                 n_attn),
        "roofline_region": {"calls": n_attn, "ms": round(attn_avg * n_attn, 2)},
        "clocks": clocks,
        "parts": parts,
    }
    if wl.unique_kv_bytes is not None:
        line["config"]["unique_kv_bytes"] = wl.unique_kv_bytes
    if e2e is not None:
        api_us = 1e6 * api["seconds"] / api["steps"]
        line["api_us_per_step"] = round(api_us, 2)
        line["e2e"] = {"value": round(whole_job_rate(wl.step_bytes, api["seconds"] / api["steps"],
                                                    world), 1),
                       "unit": "GB/s", "h2d_bytes_per_step": api["h2d"],
                       "d2h_bytes_per_step": api["d2h"], "steps": api["steps"],
                       "us_per_step": round(api_us, 2),
                       "host_issue_us_per_step": round(api["host_issue_us_per_step"], 2),
                       "graph_us_per_step": round(1e6 * e2e["seconds"] / e2e["steps"], 2),
                       "graph_value": round(whole_job_rate(
                           wl.step_bytes, e2e["seconds"] / e2e["steps"], world), 1),
                       "serial_us_per_step": round(e2e["serial_us_per_step"], 2),
                       "how": "every step issued from the host through the public API (the "
                              "Python binding of the C ABI: " + (
                                  "paged_attention_decode_append" if wl.append else
                                  "copy_blocks, reshape_and_cache, paged_attention_decode")
                              + "), pipelined over two input and two "
                              "output buffers: a copy stream brings step i+1's inputs from "
                              "pinned host memory and copies step i-1's output to pinned host "
                              "memory while step i's kernels run; the host reads every byte of "
                              "each step's output (a checksum) two steps later; wall clock "
                              "over all steps.  graph_us_per_step: the same pipeline with each "
                              "step's calls captured once in a CUDA graph and replayed; "
                              "serial_us_per_step: copy in, kernels, copy out, full sync, step "
                              "by step (graphs)"}
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.workload)
        line["cpu_baseline_single_thread"] = cpu_baseline(args.workload, single_thread=True)
    if not args.no_configs and args.placement == "scattered" and args.workload == "opt13b" \
            and args.block_size is None and args.partition is None:
        del wl
        import gc
        gc.collect()
        torch.cuda.empty_cache()
        line["configs"] = measure_configs(device, args.roofline_seconds, args.warmup, dist,
                                          attn_avg * 1e3)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def attention_calls(wl: Workload, at_least: int, seconds: float, stream) -> int:
    """How many back-to-back attention calls fill `seconds` (from a short
    timed probe), at least `at_least`."""
    import torch
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for i in range(20):
        wl.attention(i)
    b.record(stream)
    torch.cuda.synchronize()
    per = a.elapsed_time(b) / 20 * 1e-3
    return max(at_least, int(math.ceil(seconds / max(per, 1e-7))))


def timed_attention(wl: Workload, seconds: float, warmup: int, device, partition=None,
                    ws=None) -> dict:
    """Back-to-back attention calls (about `seconds` of them) between two events
    on the launching stream, with nvidia-smi clock samples over the region."""
    import torch
    stream = torch.cuda.current_stream()

    def call(i):
        layer = i % wl.layers
        wl.decode_fn(wl.out, wl.q, wl.kc[layer], wl.vc[layer], wl.tables, wl.ctx, wl.scale,
                     wl.partition if partition is None else partition, wl.ws if ws is None else ws)

    for i in range(max(3, warmup)):
        call(i)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for i in range(20):
        call(i)
    b.record(stream)
    torch.cuda.synchronize()
    n = max(20, int(math.ceil(seconds / max(a.elapsed_time(b) / 20 * 1e-3, 1e-7))))
    sampler = ClockSampler(device.index if device.index is not None else 0)
    sampler.start()
    time.sleep(0.3)
    torch.cuda.synchronize()
    a.record(stream)
    for i in range(n):
        call(i)
    b.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    if wl.pkv.get_device_error() != 0:
        raise SystemExit("bench.py: device error bits in the configs block")
    us = a.elapsed_time(b) / n * 1e3
    return {"calls": n, "us": us, "clocks": clocks}


def timed_contiguous(name: str, device, seconds: float, warmup: int) -> dict:
    """The decode attention over a contiguous [S][H][T][D] K/V layout (T = the
    batch's longest context; no block table) for the workload's batch, split
    and dtype, timed like the paged call.  Algorithmic bytes: the paged
    call's without the table entries."""
    import torch
    import paged_kv_cache_05_gb300 as pkv
    spec = W.SPECS[name]
    ctx = W.context_lens(spec)
    S, H, D = spec.num_seqs, spec.num_heads, spec.head_dim
    T = int(ctx.max())
    q = W.device_normal((S, H, D), spec.dtype, spec.seed * 1000 + 900, device)
    k = W.device_normal((S, H, T, D), spec.dtype, spec.seed * 1000 + 903, device)
    v = W.device_normal((S, H, T, D), spec.dtype, spec.seed * 1000 + 904, device)
    cl = torch.from_numpy(ctx).to(device)
    part = spec.partition_size
    ws = torch.empty(pkv.contiguous_workspace_size(S, H, D, T, part), dtype=torch.uint8,
                     device=device)
    out = torch.empty_like(q)
    stream = torch.cuda.current_stream()

    def call():
        pkv.contiguous_attention_decode(out, q, k, v, cl, spec.scale, part, ws)

    for _ in range(max(3, warmup)):
        call()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(20):
        call()
    b.record(stream)
    torch.cuda.synchronize()
    n = max(20, int(math.ceil(seconds / max(a.elapsed_time(b) / 20 * 1e-3, 1e-7))))
    sampler = ClockSampler(device.index if device.index is not None else 0)
    sampler.start()
    time.sleep(0.3)
    a.record(stream)
    for _ in range(n):
        call()
    b.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    if pkv.get_device_error() != 0:
        raise SystemExit("bench.py: device error bits (contiguous layout)")
    us = a.elapsed_time(b) / n * 1e3
    nbytes = int(ctx.astype(np.int64).sum()) * H * D * 2 * 2 + 2 * S * H * D * 2 + 4 * S
    peak, _ = read_peaks()
    gbs = nbytes / (us * 1e-6) / 1e9
    return {"workload": "%s batch, contiguous [S][H][T][D] layout (T = %d), %s, split %s" % (
                name, T, spec.dtype, "balanced" if part == 0 else "%d tokens" % part),
            "attention_us_per_call": round(us, 2), "attention_bytes_per_call": nbytes,
            "GB/s": round(gbs, 1), "frac": round(gbs / peak, 4), "calls": n, "clocks": clocks}


def measure_configs(device, seconds: float, warmup: int, dist, headline_attn_us: float) -> dict:
    """The other workloads of the decode path, each on its own: the attention
    call (main + merge) timed back to back for about `seconds`, its
    algorithmic GB/s and fraction of the measured copy peak, with the clock
    record of its region; and the prompt phase.  Long context: split length
    512 (the workload's) and the balanced split; short: bf16, B = 16;
    shared prefix: GB/s of the metric's logical bytes and of the unique
    blocks' bytes."""
    import torch
    peak, _ = read_peaks()
    out = {}

    def entry(wl, t, extra=None):
        gbs = wl.attn_bytes / (t["us"] * 1e-6) / 1e9
        e = {"workload": wl.describe(), "attention_us_per_call": round(t["us"], 2),
             "attention_bytes_per_call": wl.attn_bytes, "GB/s": round(gbs, 1),
             "frac": round(gbs / peak, 4), "calls": t["calls"], "clocks": t["clocks"]}
        if extra:
            e.update(extra)
        return e

    for name, parts, decode in (("long", (512, 0), "auto"), ("short", (None,), "auto"),
                                ("shared_prefix", (None,), "plain"),
                                ("shared_prefix", (None,), "shared")):
        wl = Workload(name, device, decode=decode)
        for part in parts:
            ws = None
            if part is not None and part != wl.partition:
                ws = wl.pkv.alloc_workspace(wl.S, wl.H, wl.D, wl.B, wl.max_blocks, part, device)
                assert not wl.shared
            t = timed_attention(wl, seconds, warmup, device, part, ws)
            key = name if part is None else "%s_split_%s" % (
                name, "balanced" if part == 0 else str(part))
            if wl.shared:
                key += "_groups"
            extra = None
            if wl.unique_kv_bytes is not None:
                ub = wl.unique_kv_bytes + (wl.attn_bytes - wl.kv_bytes)
                extra = {"unique_bytes_per_call": ub,
                         "unique_GB/s": round(ub / (t["us"] * 1e-6) / 1e9, 1),
                         "unique_frac": round(ub / (t["us"] * 1e-6) / 1e9 / peak, 4)}
            out[key] = entry(wl, t, extra)
            p_ = wl.partition if part is None else part
            out[key]["split"] = "balanced" if p_ == 0 else "%d tokens" % p_
            del ws
        del wl
        torch.cuda.empty_cache()
    # the contiguous-layout kernel on the same batches (paging's cost)
    for name, paged_key in (("opt13b", None), ("short", "short"), ("long", "long_split_512")):
        c = timed_contiguous(name, device, seconds, warmup)
        ref_us = headline_attn_us if paged_key is None else out[paged_key]["attention_us_per_call"]
        c["paged_attention_us_per_call"] = round(ref_us, 2)
        c["paged_over_contiguous"] = round(ref_us / c["attention_us_per_call"], 4)
        out[name + "_contiguous"] = c
        torch.cuda.empty_cache()
    out["prefill"] = measure_prefill("f16", max(3, warmup), seconds)
    out["note"] = ("each workload alone, after the headline runs; attention = paged_decode_main "
                   "+ paged_decode_merge back to back; frac of the measured copy peak "
                   "(%s GB/s); *_contiguous: the same kernel over a contiguous layout with no "
                   "block table, paged_over_contiguous = paged / contiguous call time; "
                   "prefill: tensor-core TFLOP/s of the prompt phase" % peak)
    return out


def measure_e2e_api(wl: Workload, steps: int, device, dist):
    """End to end through the public API with host buffers, every step issued
    by the host: the step's inputs (q, new K/V, the slot mapping when the
    writes are a call of their own, block tables, context lengths, copy
    pairs) are copied from pinned host memory in one transfer, the step's
    calls run on the compute stream, and its
    output is copied to pinned host memory and read, every byte, by the host.

    Pipelined over two device input buffers and two output buffers: while
    step i's kernels run, a copy stream copies step i-1's output out and
    then brings step i+1's inputs into the other input buffer (both after
    step i-1's kernels are done with that buffer); before issuing step i+1
    the host reads step i-1's output.  The first step's inputs are copied
    before the timed region (the copy of step K's inputs, made in the timed
    region and not used, stands in for it) and the last output is copied and
    read after the loop, inside the timed region.  Returns the wall-clock
    seconds and the host's own issue time per step."""
    import torch
    # (the slot mapping only when reshape_and_cache writes the new tokens)
    parts = [("q", wl.q), ("k_new", wl.k_new), ("v_new", wl.v_new)]
    parts += [] if wl.append else [("slots", wl.slots)]
    parts += [("tables", wl.tables), ("ctx", wl.ctx), ("pairs", wl.pairs)]
    sizes = [t.numel() * t.element_size() for _, t in parts]
    offs, o = [], 0
    for n in sizes:
        offs.append(o)
        o += (n + 255) // 256 * 256
    host = torch.empty(o, dtype=torch.uint8).pin_memory()
    devs = [torch.empty(o, dtype=torch.uint8, device=device) for _ in range(2)]
    views = [{}, {}]
    for (name, t), off, n in zip(parts, offs, sizes):
        host[off:off + n].copy_(t.detach().cpu().contiguous().view(-1).view(torch.uint8))
        for b in range(2):
            views[b][name] = devs[b][off:off + n].view(t.dtype).view(t.shape)
    out_hosts = [torch.empty(wl.out.shape, dtype=wl.out.dtype).pin_memory() for _ in range(2)]
    out_words = [h.view(-1).view(torch.uint8).numpy().view(np.uint64) for h in out_hosts]
    outs = [torch.empty_like(wl.out), torch.empty_like(wl.out)]
    h2d = sum(sizes)
    d2h = out_hosts[0].numel() * out_hosts[0].element_size()
    pkv = wl.pkv
    comp = torch.cuda.current_stream()
    cps = torch.cuda.Stream(device=device)
    in_ready = [torch.cuda.Event(), torch.cuda.Event()]
    done = [torch.cuda.Event(), torch.cuda.Event()]
    out_ready = [torch.cuda.Event(), torch.cuda.Event()]
    check = [0]

    def issue(i):
        p, layer = i % 2, i % wl.layers
        v = views[p]
        kc, vc = wl.kc[layer], wl.vc[layer]
        comp.wait_event(in_ready[p])
        if len(wl.pairs_host):
            pkv.copy_blocks(kc, vc, v["pairs"], stream=comp)
        if wl.append:
            pkv.paged_attention_decode_append(outs[p], v["q"], v["k_new"], v["v_new"], kc, vc,
                                              v["tables"], v["ctx"], wl.scale, wl.partition,
                                              wl.ws, stream=comp)
        else:
            pkv.reshape_and_cache(v["k_new"], v["v_new"], kc, vc, v["slots"], stream=comp)
            wl.decode_fn(outs[p], v["q"], kc, vc, v["tables"], v["ctx"], wl.scale,
                         wl.partition, wl.ws, stream=comp)
        done[p].record(comp)
        # the copy stream: step i-1's output out, then step i+1's inputs in
        # (step i-1's kernels are done with input buffer 1-p)
        cps.wait_event(done[1 - p])
        with torch.cuda.stream(cps):
            if i > 0:
                out_hosts[1 - p].copy_(outs[1 - p], non_blocking=True)
                out_ready[1 - p].record(cps)
            devs[1 - p].copy_(host, non_blocking=True)
            in_ready[1 - p].record(cps)

    def read(j):
        out_ready[j % 2].synchronize()
        check[0] ^= int(np.bitwise_xor.reduce(out_words[j % 2]))

    def run(n):
        torch.cuda.synchronize()
        with torch.cuda.stream(cps):
            devs[0].copy_(host, non_blocking=True)
            in_ready[0].record(cps)
        done[1].record(comp)
        torch.cuda.synchronize()
        host_s = 0.0
        t0 = time.perf_counter()
        for i in range(n):
            h0 = time.perf_counter()
            issue(i)
            host_s += time.perf_counter() - h0
            if i >= 2:
                read(i - 2)                    # copied out while step i-1 ran
        last = (n - 1) % 2
        cps.wait_event(done[last])
        with torch.cuda.stream(cps):
            out_hosts[last].copy_(outs[last], non_blocking=True)
            out_ready[last].record(cps)
        for j in range(max(0, n - 2), n):
            read(j)
        torch.cuda.synchronize()
        return time.perf_counter() - t0, host_s

    run(3)
    if dist is not None:
        dist.barrier()
    sec, host_s = run(steps)
    if pkv.get_device_error() != 0:
        raise SystemExit("bench.py: device error bits in the end-to-end leg")
    return {"seconds": sec, "steps": steps, "h2d": h2d, "d2h": d2h,
            "host_issue_us_per_step": 1e6 * host_s / steps, "checksum": check[0]}


def measure_e2e(wl: Workload, steps: int, device, dist):
    """End to end through the public API with host buffers.  Every step copies
    its inputs (q, new K/V, slot mapping, block tables, context lengths, copy
    pairs) from pinned host memory in one transfer, runs the step's kernels and
    copies the output back to pinned host memory, where the host reads it.

    Pipelined (the value reported): two device input buffers and two device
    output buffers; step i's graph runs its kernels on input buffer i % 2 into
    output buffer i % 2 while a copy stream fills the other input buffer with
    step i + 1's inputs and copies step i - 1's output to pinned host memory;
    the host reads step i - 1's output once step i's graph is done, and step
    K - 1's output is copied after the loop, inside the timed region.  The
    first step's inputs are copied before the timed region and the last
    step's copy of the next inputs stands in for it; the first graph's output
    copy (of no step) is an extra one, so the timed region holds one input
    copy per step and one output copy per step plus one; the host reads every
    step's output.  Serial (reported beside it): one graph per step, copy in,
    kernels, copy out, then a full stream synchronise before the next step."""
    import torch
    # (the slot mapping only when reshape_and_cache writes the new tokens)
    parts = [("q", wl.q), ("k_new", wl.k_new), ("v_new", wl.v_new)]
    parts += [] if wl.append else [("slots", wl.slots)]
    parts += [("tables", wl.tables), ("ctx", wl.ctx), ("pairs", wl.pairs)]
    sizes = [t.numel() * t.element_size() for _, t in parts]
    offs, o = [], 0
    for n in sizes:
        offs.append(o)
        o += (n + 255) // 256 * 256
    host = torch.empty(o, dtype=torch.uint8).pin_memory()
    devs = [torch.empty(o, dtype=torch.uint8, device=device) for _ in range(2)]
    views = [{}, {}]
    for (name, t), off, n in zip(parts, offs, sizes):
        host[off:off + n].copy_(t.detach().cpu().contiguous().view(-1).view(torch.uint8))
        for b in range(2):
            views[b][name] = devs[b][off:off + n].view(t.dtype).view(t.shape)
    out_hosts = [torch.empty(wl.out.shape, dtype=wl.out.dtype).pin_memory() for _ in range(2)]
    outs = [wl.out, torch.empty_like(wl.out)]
    h2d = sum(sizes)
    d2h = out_hosts[0].numel() * out_hosts[0].element_size()
    pkv = wl.pkv
    layers = max(1, min(wl.layers, steps))

    def kernels(layer, v, out):
        kc, vc = wl.kc[layer], wl.vc[layer]
        if len(wl.pairs_host):
            pkv.copy_blocks(kc, vc, v["pairs"])
        if wl.append:
            pkv.paged_attention_decode_append(out, v["q"], v["k_new"], v["v_new"], kc, vc,
                                              v["tables"], v["ctx"], wl.scale, wl.partition,
                                              wl.ws)
        else:
            pkv.reshape_and_cache(v["k_new"], v["v_new"], kc, vc, v["slots"])
            wl.decode_fn(out, v["q"], kc, vc, v["tables"], v["ctx"], wl.scale, wl.partition,
                         wl.ws)

    side = torch.cuda.Stream(device=device)
    cps = torch.cuda.Stream(device=device)

    def body_pipelined(layer, p):
        cur = torch.cuda.current_stream()
        start = torch.cuda.Event()
        start.record(cur)
        cps.wait_event(start)
        with torch.cuda.stream(cps):
            devs[1 - p].copy_(host, non_blocking=True)       # the next step's inputs
            out_hosts[1 - p].copy_(outs[1 - p], non_blocking=True)   # the previous step's output
        copied = torch.cuda.Event()
        copied.record(cps)
        kernels(layer, views[p], outs[p])
        cur.wait_event(copied)

    def body_serial(layer):
        devs[0].copy_(host, non_blocking=True)
        kernels(layer, views[0], outs[0])
        out_hosts[0].copy_(outs[0], non_blocking=True)

    # first calls outside capture, then one graph per (layer, buffer parity)
    # the timed loop meets, and one per layer for the serial form
    keys = sorted({(i % layers, i % 2) for i in range(steps + 3)})
    for layer, p in keys:
        body_pipelined(layer, p)
    for layer in range(layers):
        body_serial(layer)
    torch.cuda.synchronize()
    pg, sg = {}, []
    for key in keys:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            body_pipelined(*key)
        pg[key] = g
    for layer in range(layers):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            body_serial(layer)
        sg.append(g)
    torch.cuda.synchronize()
    evs = [torch.cuda.Event(), torch.cuda.Event()]
    seen = 0.0

    def run_pipelined(n):
        nonlocal seen
        devs[0].copy_(host)                                   # step 0's inputs
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(n):
            pg[(i % layers, i % 2)].replay()
            evs[i % 2].record()
            if i > 1:
                # graph i - 1 is done: step i - 2's output is on the host
                evs[(i - 1) % 2].synchronize()
                seen += float(out_hosts[i % 2].view(-1)[0])
        last = (n - 1) % 2
        out_hosts[last].copy_(outs[last], non_blocking=True)   # step n - 1's output
        torch.cuda.current_stream().synchronize()
        seen += float(out_hosts[last].view(-1)[0])
        if n > 1:
            seen += float(out_hosts[1 - last].view(-1)[0])        # step n - 2's
        return time.perf_counter() - t0

    run_pipelined(3)
    if dist is not None:
        dist.barrier()
    sec = run_pipelined(steps)
    for i in range(3):
        sg[i % layers].replay()
        torch.cuda.current_stream().synchronize()
    t0 = time.perf_counter()
    for i in range(steps):
        sg[i % layers].replay()
        torch.cuda.current_stream().synchronize()
        seen += float(out_hosts[0].view(-1)[0])
    sec_serial = time.perf_counter() - t0
    return {"seconds": sec, "steps": steps, "h2d": h2d, "d2h": d2h,
            "serial_us_per_step": 1e6 * sec_serial / steps}


def measure_parts(wl: Workload, device, warmup: int) -> dict:
    """reshape_and_cache and copy_blocks timed alone (back to back between two
    events; their algorithmic bytes: the new tokens' K/V read and written, the
    pairs' blocks read and written), and the attention call's median duration
    over 60 calls each bracketed by its own events."""
    import torch
    pkv = wl.pkv
    stream = torch.cuda.current_stream()
    n = 200
    out = {}

    def timed(fn):
        for i in range(max(3, warmup)):
            fn(i)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        a.record(stream)
        for i in range(n):
            fn(i)
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / n

    out["note"] = ("cache operations repeated on the same few-MB buffers (and, with one layer "
                   "pool, the same blocks): L2-resident and launch-latency-bound, not HBM "
                   "figures; inside the step they overlap their neighbours")
    ms = timed(lambda i: pkv.reshape_and_cache(wl.k_new, wl.v_new, wl.kc[i % wl.layers],
                                               wl.vc[i % wl.layers], wl.slots))
    out["reshape_and_cache"] = {"us": round(ms * 1e3, 2), "bytes": wl.reshape_bytes,
                                "GB/s": round(wl.reshape_bytes / (ms * 1e-3) / 1e9, 1)}
    if len(wl.pairs_host):
        ms = timed(lambda i: pkv.copy_blocks(wl.kc[i % wl.layers], wl.vc[i % wl.layers],
                                             wl.pairs))
        out["copy_blocks"] = {"us": round(ms * 1e3, 2), "bytes": wl.copy_bytes,
                              "pairs": int(len(wl.pairs_host)),
                              "GB/s": round(wl.copy_bytes / (ms * 1e-3) / 1e9, 1)}
    ts = []
    for i in range(60 + 5):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        wl.attention(i)
        b.record(stream)
        b.synchronize()
        if i >= 5:
            ts.append(a.elapsed_time(b))
    med = float(np.median(ts))
    out["attention_median_us_per_call_events"] = round(med * 1e3, 2)
    out["attention_median_GB/s"] = round(wl.attn_bytes / (med * 1e-3) / 1e9, 1)
    return out


def cpu_baseline(name: str, single_thread: bool = False) -> dict:
    """The oracle, as it stands, on the host cores over the whole batch of the
    workload (inputs built on the host: host_case), repeated until about 10 s
    of CPU work has been done; single_thread: one thread over the longest
    sequences holding about an eighth of the batch's bytes."""
    hc = host_case(name)
    ctx, S = hc["ctx"], hc["spec"].num_seqs
    threads = 1 if single_thread else min(host_cores(), S)
    seqs = None
    if single_thread:
        order = np.argsort(ctx)
        budget, seqs, acc = int(ctx.sum()) // 8, [], 0
        for s_ in order[::-1]:
            if acc >= budget and seqs:
                break
            seqs.append(int(s_))
            acc += int(ctx[s_])
    sample = oracle_sample(hc, seqs)
    first = run_oracle(sample, threads)
    reps = max(1, min(30, int(10.0 / max(first, 1e-3))))
    total, done = first, 1
    while done < reps and total < 10.0:
        total += run_oracle(sample, threads)
        done += 1
    return {"value": round(sample["bytes"] * done / total / 1e9, 4), "unit": "GB/s",
            "cores": threads, "kind": "oracle",
            "sample": "%d of %d sequences x %d heads, %d pass(es), %.1f s; tables from the "
                      "oracle's block-manager model, values from the seeded host generator" % (
                          S if seqs is None else len(seqs), S, hc["spec"].num_heads, done, total)}


def bench_swap(args):
    """Block swap GPU pool <-> pinned CPU pool at the OPT-13B layer shape (40 heads
    x 128, fp16) for block sizes 8..64: pkv_swap_blocks (one launch for every
    block) against the copy engine (one cudaMemcpyAsync per block and pool, and
    one bulk copy of the same bytes as its best case)."""
    import torch
    import paged_kv_cache_05_gb300 as pkv
    from paged_kv_cache_05_gb300 import build
    build.build()
    dev = torch.device("cuda", 0)
    H, D = 40, 128
    total = 512 << 20                       # bytes of K+V moved per direction
    rows = []
    for B in ([args.block_size] if args.block_size else [8, 16, 32, 64]):
        per_pool = H * B * D * 2
        n = total // (2 * per_pool)
        gk = W.device_normal((n, H, B, D), "f16", 11, dev)
        gv = W.device_normal((n, H, B, D), "f16", 12, dev)
        ck = torch.empty((n, H, B, D), dtype=torch.float16).pin_memory()
        cv = torch.empty_like(ck).pin_memory()
        perm = np.random.default_rng(B).permutation(n).astype(np.int32)
        p_out = torch.from_numpy(np.stack([np.arange(n, dtype=np.int32), perm], 1)).to(dev)
        p_in = torch.from_numpy(np.stack([perm, np.arange(n, dtype=np.int32)], 1)).to(dev)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

        def timed(fn, reps):
            for _ in range(2):
                fn()
            torch.cuda.synchronize()
            a.record()
            for _ in range(reps):
                fn()
            b.record()
            torch.cuda.synchronize()
            return a.elapsed_time(b) / reps * 1e-3

        reps = max(3, args.steps // 100)
        t_out = timed(lambda: pkv.swap_blocks(ck, cv, gk, gv, p_out), reps)
        t_in = timed(lambda: pkv.swap_blocks(gk, gv, ck, cv, p_in), reps)
        if pkv.get_device_error() != 0:
            raise SystemExit("bench.py --op swap: device error bits")

        def per_block_out():
            for i in range(n):
                ck[int(perm[i])].copy_(gk[i], non_blocking=True)
                cv[int(perm[i])].copy_(gv[i], non_blocking=True)
        t_ce_blocks = timed(per_block_out, 1)
        flat_g = gk.view(-1)
        flat_c = ck.view(-1)
        t_ce_bulk = timed(lambda: (flat_c.copy_(flat_g, non_blocking=True),
                                   cv.view(-1).copy_(gv.view(-1), non_blocking=True)), reps)
        nbytes = 2 * n * per_pool
        rows.append({"block_size": B, "blocks": int(n), "block_bytes_kv": 2 * per_pool,
                     "swap_out_gbs": round(nbytes / t_out / 1e9, 1),
                     "swap_in_gbs": round(nbytes / t_in / 1e9, 1),
                     "copy_engine_per_block_gbs": round(nbytes / t_ce_blocks / 1e9, 1),
                     "copy_engine_bulk_gbs": round(nbytes / t_ce_bulk / 1e9, 1)})
        del gk, gv, ck, cv
        torch.cuda.empty_cache()
    print(json.dumps({"op": "swap_blocks", "metric": "block swap GB/s (K+V bytes moved)",
                      "unit": "GB/s", "value": rows[-1]["swap_out_gbs"],
                      "config": {"heads": H, "head_dim": D, "dtype": "f16",
                                 "bytes_per_direction": total},
                      "results": rows}), flush=True)


def bench_layout(args):
    """Paged against contiguous-layout decode attention on the OPT-13B, short
    and long batches: three alternating rounds of back-to-back calls of each
    in one process (attention call only; the contiguous K/V are [S][H][T][D]
    with T the batch's longest context, no block table)."""
    import torch
    from paged_kv_cache_05_gb300 import build
    build.build()
    dev = torch.device("cuda", 0)
    out_all = {}
    for name in ("opt13b", "short", "long"):
        wl = Workload(name, dev, layers=(8 if name == "opt13b" else None))
        spec = W.SPECS[name]
        ctx = W.context_lens(spec)
        S, H, D = spec.num_seqs, spec.num_heads, spec.head_dim
        T = int(ctx.max())
        k = W.device_normal((S, H, T, D), spec.dtype, spec.seed * 1000 + 903, dev)
        v = W.device_normal((S, H, T, D), spec.dtype, spec.seed * 1000 + 904, dev)
        ws = torch.empty(wl.pkv.contiguous_workspace_size(S, H, D, T, wl.partition),
                         dtype=torch.uint8, device=dev)
        out = torch.empty_like(wl.q)

        def contig(i):
            wl.pkv.contiguous_attention_decode(out, wl.q, k, v, wl.ctx, wl.scale, wl.partition,
                                               ws)

        def timed(fn, n):
            for i in range(10):
                fn(i)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            a.record()
            for i in range(n):
                fn(i)
            b.record()
            torch.cuda.synchronize()
            return a.elapsed_time(b) / n * 1e3

        n = 600 if name == "long" else 1500
        pg, ct = [], []
        for _ in range(3):
            pg.append(timed(wl.attention, n))
            ct.append(timed(contig, n))
        if wl.pkv.get_device_error() != 0:
            raise SystemExit("bench.py --op layout: device error bits")
        cbytes = wl.attn_bytes - sum(-(-int(c) // wl.B) for c in ctx) * 4
        pm, cm = float(np.median(pg)), float(np.median(ct))
        out_all[name] = {"paged_us": [round(x, 2) for x in pg],
                         "contiguous_us": [round(x, 2) for x in ct],
                         "paged_over_contiguous": round(pm / cm, 4),
                         "paged_GB/s": round(wl.attn_bytes / (pm * 1e-6) / 1e9, 1),
                         "contiguous_GB/s": round(cbytes / (cm * 1e-6) / 1e9, 1),
                         "contiguous_T": T, "paged_pool_blocks": wl.nb}
        del wl, k, v, ws
        torch.cuda.empty_cache()
    print(json.dumps({"op": "layout", "metric": "paged / contiguous decode attention time",
                      "results": out_all}), flush=True)


def bench_prefill(args):
    """--op prefill: the prompt phase on its own (measure_prefill)."""
    from paged_kv_cache_05_gb300 import build
    build.build()
    r = measure_prefill(getattr(args, "dtype", "f16"), max(3, args.warmup),
                        args.roofline_seconds, min_calls=max(10, args.steps // 20))
    print(json.dumps(dict({"op": "prefill", "metric": "prompt-phase paged attention TFLOP/s",
                           "unit": "TFLOP/s"}, **r)), flush=True)


def measure_prefill(dt: str, warmup: int, seconds: float, min_calls: int = 10) -> dict:
    """The prompt phase at the OPT-13B shape: every prompt's K/V written into
    the pool (reshape_and_cache), then causal paged attention of all prompt
    tokens (tensor cores).  FLOPs = sum over query rows of 4 * D * H * (p + 1)
    (Q K^T and P V, causal); peak = the measured dense bf16 tensor rate
    (fp16 runs at the same nominal rate).  The whole step and the attention
    alone are each timed back to back for about `seconds`."""
    import torch
    import paged_kv_cache_05_gb300 as pkv
    dev = torch.device("cuda", 0)
    spec = W.SPECS["prefill"]
    ctx = W.context_lens(spec)
    S, H, D, B = spec.num_seqs, spec.num_heads, spec.head_dim, spec.block_size
    nb = W.pool_blocks(spec, ctx)
    bm = pkv.BlockManager(nb, B, spec.seed)
    slots = np.concatenate([bm.add_sequence(s_, int(ctx[s_])) for s_ in range(S)])
    maxb = max(-(-int(c) // B) for c in ctx)
    tables, _ = bm.export(list(range(S)), maxb)
    T = int(ctx.sum())
    kc = torch.zeros((nb, H, B, D), dtype=W.torch_dtype(dt), device=dev)
    vc = torch.zeros_like(kc)
    k = W.device_normal((T, H, D), dt, spec.seed + 1, dev)
    v = W.device_normal((T, H, D), dt, spec.seed + 2, dev)
    q = W.device_normal((T, H, D), dt, spec.seed + 3, dev)
    out = torch.empty_like(q)
    qs = torch.from_numpy(np.concatenate([[0], np.cumsum(ctx)]).astype(np.int32)).to(dev)
    bt = torch.from_numpy(tables).to(dev)
    cl = torch.from_numpy(ctx).to(dev)
    sl = torch.from_numpy(slots).to(dev)
    maxq = int(ctx.max())

    def step():
        pkv.reshape_and_cache(k, v, kc, vc, sl)
        pkv.paged_attention_prefill(out, q, kc, vc, bt, cl, qs, spec.scale, maxq)

    def attn():
        pkv.paged_attention_prefill(out, q, kc, vc, bt, cl, qs, spec.scale, maxq)

    def fused():
        # the same step in one kernel: the cache write beside the attention
        pkv.paged_attention_prefill_write(out, q, k, v, kc, vc, bt, cl, qs, spec.scale, maxq)

    for _ in range(max(3, warmup)):
        step()
        fused()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(5):
        step()
    b.record()
    torch.cuda.synchronize()
    K = max(min_calls, int(math.ceil(seconds / (a.elapsed_time(b) / 5 * 1e-3))))
    sampler = ClockSampler(0)
    sampler.start()
    time.sleep(0.3)                       # let the sampler start before the timed region
    a.record()
    for _ in range(K):
        step()
    b.record()
    torch.cuda.synchronize()
    t_step = a.elapsed_time(b) / K * 1e-3
    a.record()
    for _ in range(K):
        attn()
    b.record()
    torch.cuda.synchronize()
    t_attn = a.elapsed_time(b) / K * 1e-3
    a.record()
    for _ in range(K):
        fused()
    b.record()
    torch.cuda.synchronize()
    t_fused = a.elapsed_time(b) / K * 1e-3
    clocks = sampler.stop()
    if pkv.get_device_error() != 0:
        raise SystemExit("bench.py prefill: device error bits")
    flops = float(sum(4.0 * D * H * (c * (c + 1) / 2.0) for c in ctx))
    try:
        mp = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
        peak = float(mp["bf16_tflops"])
        src = "measured (MEASURED_PEAKS.json bf16_tflops, cuBLAS burst)"
        peak_sus = float(mp["bf16_tflops_sustained"]) if "bf16_tflops_sustained" in mp else None
    except Exception:
        peak, src, peak_sus = 1900.0, "fallback", 1700.0
    tf = flops / t_attn / 1e12
    return {
        "value": round(tf, 1), "us_per_call": round(t_attn * 1e6, 1), "calls": K,
        "us_per_step_with_cache_write": round(t_step * 1e6, 1),
        "us_per_step_fused": round(t_fused * 1e6, 1),
        "tokens_per_s": round(T / t_fused, 1),
        "tokens_per_s_two_step": round(T / t_step, 1), "dtype": "%s in, f32 accumulate" % dt,
        "step_note": "us_per_step_with_cache_write: reshape_and_cache then paged_attention_prefill; "
                     "us_per_step_fused: paged_attention_prefill_write (the cache write in the "
                     "attention kernel); tokens_per_s from the fused step",
        "config": {"workload": "prefill: %d prompts, lengths %d..%d (sum %d), 40 heads x 128, "
                               "B=16, %s" % (S, int(ctx.min()), int(ctx.max()), T,
                                             {"f16": "fp16", "bf16": "bf16"}[dt]),
                   "flops_per_call": flops},
        "roofline": {"bound": "tensor", "achieved": round(tf, 1), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(tf / peak, 4), "peak_source": src,
                     "traffic": profiled_traffic("prefill", "paged_prefill_tc_prefill.md",
                                                 PREFILL_SOURCES) if dt == "f16" else None,
                     "peak_sustained": peak_sus,
                     "frac_sustained": round(tf / peak_sus, 4) if peak_sus else None,
                     "note": "tcgen05.mma kind::f16 from shared-memory descriptors, S and O in "
                             "tensor memory, TMA tiled copies through the block table; frac "
                             "against the cuBLAS burst peak, frac_sustained against its "
                             "power-capped sustained rate (each timed region runs back to back "
                             "for about 0.4 s after the previous one: see clocks.reasons)"},
        "clocks": clocks,
    }


def sharing_savings(seed: int = 2024, block_size: int = 16):
    """Memory the block manager saves by sharing, on synthetic decoding runs
    (host only).  Parallel sampling: k samples of one prompt share the prompt's
    blocks, the partial last one copied on write.  Beam-search-like churn:
    every step each of W beams appends a token, then W survivors are drawn at
    random (no model decides) and forked from their parents while the old
    beams are freed.  Saving = 1 - blocks in use / blocks needed if every
    sequence held its own copy, averaged over the run's steps."""
    import paged_kv_cache_05_gb300 as pkv
    rng = np.random.default_rng(seed)
    B = block_size
    out = {"parallel_sampling": {}, "beam_search": {}}
    for k in (2, 4, 6):
        bm = pkv.BlockManager(200_000, B, seed)
        savings = []
        for g in range(16):
            P = int(rng.integers(128, 1025))
            O = rng.integers(1, 513, size=k)
            base = g * 100
            bm.add_sequence(base, P)
            for c in range(1, k):
                bm.fork(base, base + c)
            for t in range(int(O.max())):
                act = [base + c for c in range(k) if t < O[c]]
                bm.append_slots(act)
            used_before = 200_000 - bm.num_free()
            unshared = sum(-(-(P + int(o)) // B) for o in O)
            shared = sum(len(bm.block_table(base + c)) for c in range(k))
            distinct = len({b for c in range(k) for b in bm.block_table(base + c)})
            savings.append(1 - distinct / unshared)
            assert shared == unshared and used_before > 0
            for c in range(k):
                bm.free_sequence(base + c)
        out["parallel_sampling"][k] = round(float(np.mean(savings)), 4)
    for W_ in (4, 8):
        bm = pkv.BlockManager(200_000, B, seed + W_)
        savings = []
        for g in range(8):
            P = int(rng.integers(128, 1025))
            nxt = g * 100_000
            bm.add_sequence(nxt, P)
            beams = [nxt]
            nxt += 1
            for c in range(1, W_):
                bm.fork(beams[0], nxt)
                beams.append(nxt)
                nxt += 1
            for t in range(256):
                bm.append_slots(beams)
                parents = rng.integers(0, W_, size=W_)
                new = []
                for p_ in parents:
                    bm.fork(beams[int(p_)], nxt)
                    new.append(nxt)
                    nxt += 1
                for b_ in beams:
                    bm.free_sequence(b_)
                beams = new
                distinct = len({b for s_ in beams for b in bm.block_table(s_)})
                unshared = W_ * -(-(P + t + 1) // B)
                savings.append(1 - distinct / unshared)
            for b_ in beams:
                bm.free_sequence(b_)
            assert bm.num_free() == 200_000
        out["beam_search"][W_] = round(float(np.mean(savings)), 4)
    return out


def reference_arm(args, world, rank, dist):
    """The CPU fp64 oracle as the reference arm, on the host cores: W warm-up
    and K timed steps, each over a length-spread subset of the workload sized
    so that the whole run takes about a minute.  Its inputs are built on the
    host (host_case: the oracle's block-manager model and the seeded host
    generator), so the product library is never loaded."""
    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return
    hc = host_case(args.workload, args.block_size)
    spec = hc["spec"]
    threads = host_cores()
    K, Wu = max(1, args.steps), max(0, args.warmup)
    seqs = sized_sample(hc, 60.0 / (K + Wu), threads)
    sample = oracle_sample(hc, seqs)
    threads = min(threads, len(seqs))
    for _ in range(Wu):
        run_oracle(sample, threads)
    times = [run_oracle(sample, threads) for _ in range(K)]
    sec = statistics.mean(times)
    v = sample["bytes"] / sec / 1e9
    desc = "%d of %d sequences (length-spread), all %d heads, per step" % (
        len(seqs), spec.num_seqs, spec.num_heads)
    c = hc["ctx"]
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(v, 4), "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": Wu,
        "ms_per_step": round(sec * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": {"workload": "%s: %d seqs x %d heads x %d, %s K/V, B=%d, ctx %d..%d (sum %d)"
                               % (args.workload, spec.num_seqs, spec.num_heads, spec.head_dim,
                                  spec.dtype, hc["B"], int(c.min()), int(c.max()), int(c.sum())),
                   "sample": desc},
        "cpu_baseline": {"value": round(v, 4), "unit": "GB/s", "cores": threads,
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": round(v, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
