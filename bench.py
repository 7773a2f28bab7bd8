"""Paged decode benchmark: one decode step of a Llama-3-8B-shaped layer.

Workload (the headline configuration): 64 sequences, 32 query / 8 KV heads,
head_dim 128, bf16 cache, block size 16; context lengths are prompt + output
of the first 64 requests of the seeded request mix (sum 121,416 tokens,
732..3360); blocks are a seeded permutation of a pool 1.2x the blocks used.
One step = the host slot mapping of the 64 new tokens, then one library call
(pa_write_and_decode): the cache write of their K/V and paged decode over
all 64 sequences.  The decode call alone and the write alone are also timed.

Metric: achieved HBM GB/s on the algorithmic bytes a step must move
(K and V of every context token once, q, out, block-table entries, lengths,
the new tokens' K/V write) and microseconds per step.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
Under torchrun every rank runs an independent replica on its own GPU (the
path has no cross-GPU exchange); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged decode attention: achieved HBM GB/s (% of GB300 peak) and µs/step"
L2_FLUSH_BYTES = 512 << 20
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--partition", type=int, default=0, help="split-K partition (0 = auto)")
    ap.add_argument("--kernel", type=int, default=0, help="decode kernel (0 auto, 1 SIMT, 2 tcgen05)")
    ap.add_argument("--kv-dtype", choices=["bf16", "fp8"], default="bf16",
                    help="KV cache type: bf16, or fp8-e4m3 with per-tensor scales")
    ap.add_argument("--workload", choices=list(WORKLOADS), default="llama8b",
                    help="llama8b: the headline layer (batch 64); longctx: 8 sequences of "
                         "4K..128K tokens; serving: 256 MHA sequences in groups of 8 sharing "
                         "a 1024-token prefix")
    ap.add_argument("--new-tokens", type=int, default=1,
                    help="tokens each sequence adds per step (> 1: multi-token step through "
                         "pa_varlen_attention, e.g. speculative decoding)")
    ap.add_argument("--shared-prefix-group", type=int, default=0,
                    help="decode through pa_decode_shared_prefix with groups of this many "
                         "sequences (serving workload: 8); 0 = pa_decode")
    ap.add_argument("--block-size", type=int, default=16,
                    help="tokens per physical block (llama8b workload: 1, 16, 64, 256)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


# ---------------------------------------------------------------- ranks

def slowest_over_ranks(values, dist, device):
    """Each per-rank time replaced by its maximum over all ranks (the job
    finishes with its slowest replica); identity without a process group."""
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    if dist is not None:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t]


def job_throughput(world, bytes_per_replica_step, seconds_per_step):
    """Whole-job rate: every replica moves its own bytes in the slowest
    replica's step time (weak scaling)."""
    return world * bytes_per_replica_step / seconds_per_step


# ---------------------------------------------------------------- workload

# steps adding at least this many tokens per sequence run as prefill chunks
# (pa_varlen_attention: tensor-core prefill tiles, a tensor-bound roofline)
PREFILL_TOKENS = 16

WORKLOADS = {
    "llama8b": "llama8b-layer decode, batch 64, 32q/8kv heads, d=128",
    "longctx": "long-context decode, 8 sequences of 4K-128K tokens, 32q/8kv heads, d=128",
    "serving": "serving step, 256 MHA sequences (32q/32kv, d=128) in 32 groups of 8 sharing "
               "a 1024-token prefix, suffixes U[16, 2048]",
}


def build_workload(name, block_size, kv_dtype):
    """Shapes, lengths and block tables of a workload (no K/V values).
    Returns (workload, unique_tokens): the tokens whose K/V are stored once
    (fewer than sum(context_lens) when sequences share prefix blocks)."""
    from paged_kv_cache_108_gb300 import synth
    if name == "llama8b":
        w = synth.llama8b(block_size=block_size, kv_dtype=kv_dtype, with_data=False)
        return w, int(np.sum(w.context_lens))
    if name == "longctx":
        w = synth.longctx(kv_dtype=kv_dtype, with_data=False)
        return w, int(np.sum(w.context_lens))
    # serving mix: each group's prefix blocks appear in all its members' tables
    mix = synth.serving()
    B, P = mix.block_size, mix.prefix_len
    lens = (P + mix.suffix_lens).astype(np.int32)
    pre_blocks = -(-P // B)
    priv = [-(-int(n) // B) - P // B for n in lens]
    used = mix.num_groups * pre_blocks + sum(priv)
    num_blocks = int(math.ceil(1.2 * used))
    perm = np.random.default_rng(mix.seed).permutation(num_blocks).astype(np.int32)
    tables = np.zeros((mix.num_seqs, max(P // B + c for c in priv)), dtype=np.int32)
    at = 0
    for grp in range(mix.num_groups):
        prefix = perm[at:at + pre_blocks]
        at += pre_blocks
        for i in range(grp * mix.group_size, (grp + 1) * mix.group_size):
            tables[i, :P // B] = prefix[:P // B]
            tables[i, P // B:P // B + priv[i]] = perm[at:at + priv[i]]
            at += priv[i]
    w = synth.Workload("serving", mix.num_heads, mix.num_kv_heads, mix.head_dim, B, kv_dtype,
                       num_blocks, lens, tables, 1.0 / math.sqrt(mix.head_dim), mix.seed)
    unique = mix.num_groups * P + int(np.sum(lens - P))
    return w, unique


def causal_pairs(context_lens, new_tokens) -> int:
    """(new token, visible key) pairs of a step in which every sequence adds
    its last ``new_tokens`` positions: token j of a sequence of n sees the
    n - T + j + 1 keys up to and including itself."""
    T = int(new_tokens)
    return sum(int(n - T) * T + T * (T + 1) // 2 for n in context_lens)


def decode_bytes_of(w, kv_bytes, new_tokens, tokens) -> int:
    """Algorithmic bytes of one decode call (what the method must move): the
    K/V rows of ``tokens`` stored tokens once per KV head (rows stored once
    are read once, so shared prefix blocks count once), q and out, the
    block-table entries and the lengths."""
    kv = tokens * w.num_kv_heads * w.head_dim * kv_bytes * 2
    qo = 2 * w.num_seqs * new_tokens * w.num_heads * w.head_dim * 2
    table = int(sum(math.ceil(n / w.block_size) for n in w.context_lens)) * 4
    return kv + qo + table + w.num_seqs * 4


def write_bytes_of(w, kv_bytes, new_tokens) -> int:
    """Algorithmic bytes of the step's cache write: the new tokens' bf16 K
    and V read, their cache rows written, and their slots."""
    n = w.num_seqs * new_tokens
    return 2 * n * w.num_kv_heads * w.head_dim * (2 + kv_bytes) + n * 4


def step_config(args, w, unique_tokens, fp8, new_tokens, group, sbytes, dbytes, world):
    """The ``config`` object of the JSON line (both arms print the same one)."""
    cfg = {"workload": f"{WORKLOADS[args.workload]}, "
                       + (f"{new_tokens} new tokens per sequence "
                          + ("(chunked prefill, pa_varlen_attention tiles), "
                             if new_tokens >= PREFILL_TOKENS else
                             "(pa_decode_multi), ") if new_tokens > 1 else "")
                       + (f"shared-prefix groups of {group} "
                          "(pa_decode_shared_prefix), " if group else "")
                       + f"{'e4m3 (per-tensor scale)' if fp8 else 'bf16'} KV, "
                       f"block {w.block_size}, sum ctx {int(np.sum(w.context_lens))}",
           "num_seqs": w.num_seqs,
           "num_heads": w.num_heads, "num_kv_heads": w.num_kv_heads,
           "head_dim": w.head_dim, "block_size": w.block_size,
           "num_blocks": w.num_blocks, "sum_context": int(np.sum(w.context_lens)),
           "partition_tokens": args.partition or "auto", "kernel": args.kernel or "auto",
           "bytes_per_step": sbytes, "decode_bytes_per_step": dbytes}
    if unique_tokens != int(np.sum(w.context_lens)):
        cfg["decode_bytes_logical"] = decode_bytes_of(w, 1 if fp8 else 2, new_tokens,
                                                      int(np.sum(w.context_lens)))
        cfg["unique_context_tokens"] = unique_tokens
    cfg["l2"] = (f"flushed between steps by reading a {L2_FLUSH_BYTES >> 20} MB buffer "
                 "(untimed)")
    cfg["parallelism"] = "replicas" if world > 1 else "single GPU"
    return cfg


class Step:
    """Device-resident state of one decode step of a workload."""

    def __init__(self, device, partition=0, kernel=0, kv_dtype="bf16", workload="llama8b",
                 block_size=16, new_tokens=1, shared_prefix_group=0):
        import torch

        from paged_kv_cache_108_gb300 import ops, pool, synth
        self.torch, self.ops, self.pool = torch, ops, pool
        w, self.unique_tokens = build_workload(workload, block_size, kv_dtype)
        self.workload = workload
        self.w = w
        self.device = device
        self.partition, self.kernel = partition, kernel
        self.fp8 = kv_dtype == "fp8"
        self.kv_bytes = 1 if self.fp8 else 2
        B, hkv, d, H = w.block_size, w.num_kv_heads, w.head_dim, w.num_heads
        gen = torch.Generator(device=device)
        gen.manual_seed(w.seed)
        shape = (w.num_blocks, B, hkv, d)
        self.k_scale = self.v_scale = None
        if self.fp8:
            # N(0,1) quantised to e4m3 with scale amax / 448 (per tensor)
            caches, scales = [], []
            for _ in range(2):
                x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
                sc = (x.abs().max() / 448.0).reshape(1)
                caches.append((x / sc).to(torch.float8_e4m3fn).view(torch.uint8))
                scales.append(sc)
                del x
            self.k_cache, self.v_cache = caches
            self.k_scale, self.v_scale = scales
        else:
            self.k_cache = torch.randn(shape, generator=gen, device=device, dtype=torch.bfloat16)
            self.v_cache = torch.randn(shape, generator=gen, device=device, dtype=torch.bfloat16)
        S = w.num_seqs
        T = new_tokens
        self.new_tokens = T
        self.q = torch.randn((S * T, H, d), generator=gen, device=device).to(torch.bfloat16)
        self.k_new = torch.randn((S * T, hkv, d), generator=gen, device=device).to(torch.bfloat16)
        self.v_new = torch.randn((S * T, hkv, d), generator=gen, device=device).to(torch.bfloat16)
        # the step's tokens: the last T positions of every context, sequence-major
        self.token_seq = np.repeat(np.arange(S, dtype=np.int32), T)
        self.positions = (np.repeat(w.context_lens, T) - T +
                          np.tile(np.arange(T, dtype=np.int32), S)).astype(np.int32)
        slots = pool.slot_mapping(w.block_tables, B, self.positions, self.token_seq)
        self.qsl = torch.arange(0, S * T + 1, T, dtype=torch.int32, device=device)
        self.slots = torch.from_numpy(slots).to(device)
        self.block_tables = torch.from_numpy(w.block_tables).to(device)
        self.context_lens = torch.from_numpy(w.context_lens).to(device)
        self.out = torch.empty_like(self.q)
        self.group = shared_prefix_group
        if T == 1 and self.group:
            n = max(ops.decode_shared_prefix_workspace_size(S, self.group, H, d, w.max_blocks, B),
                    ops.decode_workspace_size(S, H, d, w.max_blocks, B))
            self.ws = torch.empty(n, dtype=torch.uint8, device=device)
        elif T == 1:
            self.ws = ops.alloc_workspace(S, H, d, w.max_blocks, B, partition, device=device)
        elif T >= PREFILL_TOKENS:
            n = ops.varlen_workspace_size(S * T, H, d, w.max_blocks, B)
            self.ws = torch.empty(n, dtype=torch.uint8, device=device)
        else:
            n = ops.decode_multi_workspace_size(S, T, H, d, w.max_blocks, B)
            self.ws = torch.empty(n, dtype=torch.uint8, device=device)
        # the tensor-core decode (one launch, merge inside) serves this shape
        # unless the SIMT kernel is forced; SIMT adds a combine launch
        simt = kernel == 1
        G = H // hkv
        tc = kernel == 2 or (kernel == 0 and d == 128 and S <= 1024 and G in (1, 2, 4, 8)
                                   and (B >= 8 or T > 1))
        splits = int(np.max(w.context_lens)) > (partition or 256)
        self.launches_per_step = 2 + (1 if not tc and splits else 0)
        if shared_prefix_group:
            # metadata, prefix pass, suffix pass, merge -- plus the cache write
            self.launches_per_step = 5
        if T >= PREFILL_TOKENS:
            self.launches_per_step = 2  # cache write, prefill tiles

    def decode_bytes(self, logical=False) -> int:
        tokens = int(np.sum(self.w.context_lens)) if logical else self.unique_tokens
        return decode_bytes_of(self.w, self.kv_bytes, self.new_tokens, tokens)

    # causal attention flops of one step: per query head, 4 d per visible
    # (new token, key) pair -- the tensor-core prefill tiles' algorithmic work
    def decode_flops(self) -> float:
        w = self.w
        return 4.0 * w.head_dim * w.num_heads * causal_pairs(w.context_lens, self.new_tokens)

    def write_bytes(self) -> int:
        return write_bytes_of(self.w, self.kv_bytes, self.new_tokens)

    def run_write(self, slots=None, k=None, v=None):
        self.ops.reshape_and_cache(self.k_new if k is None else k, self.v_new if v is None else v,
                                   self.k_cache, self.v_cache, self.slots if slots is None else slots,
                                   self.k_scale, self.v_scale)

    def run_step(self, slots=None, k=None, v=None, q=None, bt=None, cl=None):
        """The step as one call: cache write of the new tokens, then decode."""
        w = self.w
        if self.new_tokens > 1 or self.group:
            self.run_write(slots, k, v)
            self.run_decode(q, bt, cl)
            return
        self.ops.write_and_decode(self.k_new if k is None else k, self.v_new if v is None else v,
                                  self.slots if slots is None else slots, self.out,
                                  self.q if q is None else q, self.k_cache, self.v_cache,
                                  self.block_tables if bt is None else bt,
                                  self.context_lens if cl is None else cl, w.scale,
                                  self.k_scale, self.v_scale, workspace=self.ws)

    def run_decode(self, q=None, bt=None, cl=None):
        w = self.w
        if self.group:
            self.ops.decode_shared_prefix(self.out, self.q if q is None else q, self.k_cache,
                                          self.v_cache, self.block_tables if bt is None else bt,
                                          self.context_lens if cl is None else cl, self.group,
                                          w.scale, self.k_scale, self.v_scale, workspace=self.ws)
            return
        if self.new_tokens >= PREFILL_TOKENS:
            self.ops.varlen_attention(self.out, self.q if q is None else q, self.k_cache,
                                      self.v_cache, self.block_tables if bt is None else bt,
                                      self.context_lens if cl is None else cl, self.qsl,
                                      w.scale, self.k_scale, self.v_scale, workspace=self.ws)
            return
        if self.new_tokens > 1:
            self.ops.decode_multi(self.out, self.q if q is None else q, self.k_cache,
                                  self.v_cache, self.block_tables if bt is None else bt,
                                  self.context_lens if cl is None else cl, self.new_tokens,
                                  w.scale, self.k_scale, self.v_scale, workspace=self.ws)
            return
        self.ops.decode(self.out, self.q if q is None else q, self.k_cache, self.v_cache,
                        self.block_tables if bt is None else bt,
                        self.context_lens if cl is None else cl, w.scale, self.k_scale,
                        self.v_scale, workspace=self.ws, partition_tokens=self.partition,
                        kernel=self.kernel)


# ---------------------------------------------------------------- helpers

def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:  # noqa: BLE001
        return FALLBACK_HBM_GBS, "fallback"


def measured_tensor_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:  # noqa: BLE001
        return FALLBACK_BF16_TFLOPS, "fallback"


def recorded_traffic(step_bytes, kv_dtype="bf16"):
    """ncu DRAM bytes per decode call, if recorded for the current kernel source."""
    name = "decode_traffic.json" if kv_dtype == "bf16" else f"decode_traffic_{kv_dtype}.json"
    path = os.path.join(ROOT, "profiles", name)
    try:
        with open(path) as f:
            rec = json.load(f)
    except Exception:  # noqa: BLE001
        return None
    import hashlib
    h = hashlib.sha256()
    for rel in rec.get("sources", []):
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    if h.hexdigest() != rec.get("sources_sha256"):
        return None
    return rec.get("dram_bytes_per_call")


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:  # noqa: BLE001
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:  # noqa: BLE001
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[3:7]):
                if val.lower() in ("active", "1"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


def cpu_baseline_oracle(step, budget_s=10.0):
    """Time the fp64 oracle on this step's data on the host cores."""
    from oracle import core as ocore
    torch = step.torch
    w = step.w
    if step.fp8:
        kc = step.k_cache.cpu().numpy()
        vc = step.v_cache.cpu().numpy()
        ks, vs = float(step.k_scale.item()), float(step.v_scale.item())
    else:
        kc = step.k_cache.view(torch.int16).cpu().numpy().view(np.uint16)
        vc = step.v_cache.view(torch.int16).cpu().numpy().view(np.uint16)
        ks = vs = 1.0
    q = step.q.view(torch.int16).cpu().numpy().view(np.uint16)
    threads = os.cpu_count() or 1
    units = [(i, g) for i in range(w.num_seqs) for g in range(w.num_kv_heads)]
    # bounded sample: the first sequences' units until the budget is spent
    bytes_done, t_total, reps = 0, 0.0, 0
    per_unit_bytes = {(i, g): int(w.context_lens[i]) * w.head_dim * step.kv_bytes * 2
                      for i, g in units}
    chunk = max(threads, 32)
    at = 0
    while t_total < budget_s and reps < 100000:
        sel = units[at:at + chunk]
        if not sel:
            at = 0
            continue
        t0 = time.perf_counter()
        ocore.decode(q, kc, vc, w.block_tables, w.context_lens, w.scale, ks, vs, units=sel,
                     nthreads=threads)
        t_total += time.perf_counter() - t0
        bytes_done += sum(per_unit_bytes[u] for u in sel)
        at += chunk
        reps += 1
    gbs = bytes_done / t_total / 1e9
    return {"value": gbs, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{reps} batches of {chunk} (sequence, kv-head) units of the {step.workload} step "
                      f"({bytes_done / 1e6:.0f} MB of KV, {t_total:.1f} s), fp64, {threads} threads"}


# ---------------------------------------------------------------- arms

def run_ours(args, rank, world, local_rank):
    import torch
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    step = Step(device, args.partition, args.kernel, args.kv_dtype, args.workload,
                args.block_size, args.new_tokens, args.shared_prefix_group)
    stream = torch.cuda.current_stream()
    # L2 flush: read a buffer 4x the L2 size.  Reading (not writing) leaves
    # only clean lines behind, so the timed kernels do not pay for writing
    # back another kernel's dirty data.
    flush = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    flush_sink = torch.empty((), dtype=torch.float32, device=device)

    def flush_l2():
        torch.sum(flush, dim=0, out=flush_sink)

    dist = None
    if world > 1:
        import torch.distributed as dist

    def one_step():
        if step.kernel == 0:
            step.run_step()
        else:  # a forced kernel choice goes through the separate calls
            step.run_write()
            step.run_decode()

    for _ in range(max(args.warmup, 3)):
        one_step()
        step.run_decode()
    torch.cuda.synchronize()

    # device-resident timing.  Loop 1 times the step (value); loop 2 times
    # the decode call alone (roofline of the dominant kernel); loop 3 the
    # cache write alone.  Each timed call follows an untimed L2 flush.
    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(K)]
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    def host_ahead():
        # a few ms of GPU sleep ahead of a timed loop: the host enqueues the
        # first iterations while the GPU waits, so host-side latency (the
        # clock sampler starting, a first call through a code path) never
        # shows between a start event and its kernels
        torch.cuda._sleep(int(4e6))

    with ClockSampler(local_rank) as clk:
        time.sleep(0.3)  # the sampler's own start-up (NVML) is over before timing
        host_ahead()
        # after an idle GPU the first call runs with cold clocks (measured
        # 160-280 us against 87 us for the batch-64 step): a few untimed
        # steps, queued back to back with the timed ones, wake it first
        for _ in range(3):
            flush_l2()
            one_step()
        for k in range(K):
            flush_l2()
            ev[k][0].record(stream)
            one_step()
            ev[k][1].record(stream)
        host_ahead()
        for k in range(K):
            flush_l2()
            ev[k][2].record(stream)
            step.run_decode()
            ev[k][3].record(stream)
        host_ahead()
        for k in range(K):
            flush_l2()
            ev[k][4].record(stream)
            step.run_write()
            ev[k][5].record(stream)
        torch.cuda.synchronize()
    if dist:
        dist.barrier()
    step_ms = [ev[k][0].elapsed_time(ev[k][1]) for k in range(K)]
    dec_ms = [ev[k][2].elapsed_time(ev[k][3]) for k in range(K)]
    wr_ms = [ev[k][4].elapsed_time(ev[k][5]) for k in range(K)]
    mean_step = sum(step_ms) / K
    mean_dec = sum(dec_ms) / K
    mean_step, mean_dec = slowest_over_ranks([mean_step, mean_dec], dist, device)

    # end-to-end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(step, args, device, dist)

    cpu = None
    # the oracle baseline samples decode units: single-token steps only
    if rank == 0 and world == 1 and not args.no_cpu_baseline and step.new_tokens == 1:
        cpu = cpu_baseline_oracle(step)

    if rank != 0:
        return
    peak, peak_src = measured_peak()
    dbytes = step.decode_bytes()
    sbytes = dbytes + step.write_bytes()
    achieved = dbytes / (mean_dec * 1e-3) / 1e9
    if step.new_tokens >= PREFILL_TOKENS:
        # prefill chunks are a dense contraction: causal attention flops per
        # second against the measured bf16 tensor peak (burst: the call is
        # timed on its own)
        tpk, tsrc = measured_tensor_peak()
        if step.fp8:
            # e4m3 operands (kind::f8f6f4): the bf16 peak times the nominal
            # fp8 : bf16 dense ratio (4.5 : 2.25 PFLOP/s)
            tpk, tsrc = 2.0 * tpk, tsrc + " bf16 x 2 (nominal e4m3:bf16 ratio)"
        tf = step.decode_flops() / (mean_dec * 1e-3) / 1e12
        roofline = {"bound": "tensor", "kernel": "pa_varlen_attention alone (tensor-core "
                    "prefill tiles)", "achieved": round(tf, 2), "peak": tpk, "peak_source": tsrc,
                    "unit": "TFLOP/s", "frac": round(tf / tpk, 4), "traffic": None,
                    "algorithmic_flops": step.decode_flops()}
    else:
        roofline = {"bound": "hbm", "kernel": "pa_decode alone (tcgen05 paged decode; split "
                    "units merged in-kernel)", "achieved": round(achieved, 2), "peak": peak,
                    "peak_source": peak_src, "unit": "GB/s", "frac": round(achieved / peak, 4),
                    # the ncu record covers the headline decode (per-head kernel,
                    # block 16) only
                    "traffic": (recorded_traffic(dbytes, args.kv_dtype)
                                if args.workload == "llama8b" and args.block_size == 16
                                and args.kernel in (0, 2) and step.new_tokens == 1
                                and not step.group else None),
                    "algorithmic_bytes": dbytes}
    value = job_throughput(world, sbytes, mean_step * 1e-3) / 1e9
    w = step.w
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": max(args.warmup, 3), "ms_per_step": round(mean_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3" if step.fp8 else "bf16",
        "data": ("synthetic (seeded N(0,1) K/V quantised to e4m3 with scale amax/448, bf16 q; "
                 "lengths from the pages' seeded request mix)" if step.fp8 else
                 "synthetic (seeded N(0,1) bf16 K/V/q; lengths from the pages' seeded request mix)"),
        "config": step_config(args, w, step.unique_tokens, step.fp8, step.new_tokens,
                              step.group, sbytes, dbytes, world),
        "us_per_step": round(mean_step * 1e3, 2),
        "us_per_step_p50": round(statistics.median(step_ms) * 1e3, 2),
        "us_per_step_p90": round(float(np.percentile(step_ms, 90)) * 1e3, 2),
        "us_per_step_max": round(max(step_ms) * 1e3, 2),
        "us_decode_p50": round(statistics.median(dec_ms) * 1e3, 2),
        "us_decode": round(mean_dec * 1e3, 2),
        "us_write": round(sum(wr_ms) / K * 1e3, 2),
        "tokens_per_s": round(world * w.num_seqs * step.new_tokens / (mean_step * 1e-3), 1),
        "pct_of_nominal_8tbps": round(100 * achieved / 8000.0, 1),
        "roofline": roofline,
        "gpu_launches": K * 2 * step.launches_per_step,
        "clocks": clk.summary(),
    }
    if e2e is not None:
        line["e2e"] = e2e
    if cpu is not None:
        line["cpu_baseline"] = cpu
    print(json.dumps(line), flush=True)


def run_e2e(step, args, device, dist):
    """Same metric through the public API with pinned host buffers: per step,
    host slot mapping, host->device copies of the step's inputs, cache write,
    decode, and a device->host read of the output."""
    import torch
    w = step.w
    # The step's inputs travel as one packed pinned buffer (one host->device
    # copy per step); the device-side views point into one staging buffer.
    # With the captured single-token step the slots are derived in the graph
    # from the tables and lengths (pa_step_prepare); otherwise the host maps
    # them every step and they travel with the other inputs.
    device_slots = step.kernel == 0 and step.new_tokens == 1 and not step.group
    parts = [("q", step.q), ("k", step.k_new), ("v", step.v_new),
             ("bt", step.block_tables), ("cl", step.context_lens)]
    if not device_slots:
        parts.append(("slots", step.slots))
    offs, total = {}, 0
    for name, t in parts:
        offs[name] = total
        total += -(-(t.numel() * t.element_size()) // 256) * 256
    h_in = torch.empty(total, dtype=torch.uint8).pin_memory()
    d_in = torch.empty(total, dtype=torch.uint8, device=device)

    def view(buf, name, like):
        nbytes = like.numel() * like.element_size()
        return buf[offs[name]:offs[name] + nbytes].view(like.dtype).view(like.shape)

    h_v = {name: view(h_in, name, t) for name, t in parts}
    d_v = {name: view(d_in, name, t) for name, t in parts}
    for name, t in parts:
        if name != "slots":
            h_v[name].copy_(t.cpu())
    h_out = torch.empty(step.out.shape, dtype=torch.bfloat16).pin_memory()
    bi = total
    bo = h_out.numel() * h_out.element_size()

    graph = None
    if device_slots:
        # the step as one captured graph: packed inputs in, slots from the
        # tables and lengths, write + decode, output out
        d_slots = torch.empty(w.num_seqs, dtype=torch.int32, device=device)
        graph = step.ops.StepGraph(d_v["k"], d_v["v"], d_slots, step.out, d_v["q"],
                                   step.k_cache, step.v_cache, d_v["bt"], d_v["cl"], w.scale,
                                   step.k_scale, step.v_scale, step.ws,
                                   h2d=[(d_in, h_in)], d2h=[(h_out, step.out)],
                                   device_slots=True)
    else:
        h_v["slots"].numpy()[:] = step.pool.slot_mapping(w.block_tables, w.block_size,
                                                         step.positions, step.token_seq)

    def one():
        if graph is None:
            # host slot mapping of the step's new tokens into the pinned staging
            h_v["slots"].numpy()[:] = step.pool.slot_mapping(w.block_tables, w.block_size,
                                                             step.positions, step.token_seq)
        if graph is not None:
            graph.replay()
        else:
            d_in.copy_(h_in, non_blocking=True)
            step.run_write(d_v["slots"], d_v["k"], d_v["v"])
            step.run_decode(d_v["q"], d_v["bt"], d_v["cl"])
            h_out.copy_(step.out, non_blocking=True)
        torch.cuda.current_stream().synchronize()  # the host reads the result

    for _ in range(max(args.warmup, 3)):
        one()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one()
    torch.cuda.synchronize()
    dt = (time.perf_counter() - t0) / args.steps
    dt = slowest_over_ranks([dt], dist, device)[0]
    world = dist.get_world_size() if dist else 1
    sbytes = step.decode_bytes() + step.write_bytes()
    return {"value": round(job_throughput(world, sbytes, dt) / 1e9, 2), "unit": "GB/s",
            "us_per_step": round(dt * 1e6, 2), "h2d_bytes_per_step": bi,
            "d2h_bytes_per_step": bo,
            "path": ("one replay of the captured step (H2D of the packed inputs: q, new K/V, "
                     "tables, lengths; slots from tables and lengths on the device "
                     "(pa_step_prepare); pa_write_and_decode; D2H of the output), then a "
                     "stream synchronise" if graph is not None else
                     "host slot mapping, H2D, the library calls, D2H, stream synchronise")}


def run_reference(args, rank, world):
    """The oracle as the reference arm: every step is the whole step of the
    same workload -- the cache write of the new tokens, then the decode of
    every (sequence, KV head) unit -- by the fp64 CPU oracle on all host
    cores, on a seeded N(0,1) pool of the same shape."""
    if rank != 0:
        return
    from oracle import core as ocore
    from paged_kv_cache_108_gb300 import pool, synth
    if args.new_tokens != 1 or args.shared_prefix_group:
        print(json.dumps({"impl": "reference", "unavailable": "the oracle arm times single-token "
                          "decode steps through pa_decode only"}), flush=True)
        return
    w, unique = build_workload(args.workload, args.block_size, args.kv_dtype)
    fp8 = args.kv_dtype == "fp8"
    rng = np.random.default_rng(w.seed)
    shape = (w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim)
    ks = vs = 1.0
    if fp8:
        caches = []
        for _ in range(2):
            x = synth.normal_bf16(rng, shape)
            sc = synth.per_tensor_scale(x)
            codes = np.zeros(shape, dtype=np.uint8)
            ocore.reshape_and_cache(x.reshape(-1, w.num_kv_heads, w.head_dim), x.reshape(
                -1, w.num_kv_heads, w.head_dim), codes, codes.copy(),
                np.arange(w.num_blocks * w.block_size, dtype=np.int32), sc, sc)
            caches.append((codes, sc))
            del x
        (kc, ks), (vc, vs) = caches
    else:
        kc = synth.normal_bf16(rng, shape)
        vc = synth.normal_bf16(rng, shape)
    q = synth.normal_bf16(rng, (w.num_seqs, w.num_heads, w.head_dim))
    k_new = synth.normal_bf16(rng, (w.num_seqs, w.num_kv_heads, w.head_dim))
    v_new = synth.normal_bf16(rng, (w.num_seqs, w.num_kv_heads, w.head_dim))
    seqs = np.arange(w.num_seqs, dtype=np.int32)
    threads = os.cpu_count() or 1
    kv_bytes = 1 if fp8 else 2
    dbytes = decode_bytes_of(w, kv_bytes, 1, unique)
    sbytes = dbytes + write_bytes_of(w, kv_bytes, 1)

    def one_step():
        slots = pool.slot_mapping(w.block_tables, w.block_size, w.context_lens - 1, seqs)
        ocore.reshape_and_cache(k_new, v_new, kc, vc, slots, ks, vs)
        ocore.decode(q, kc, vc, w.block_tables, w.context_lens, w.scale, ks, vs,
                     nthreads=threads)

    for _ in range(max(args.warmup, 3)):
        one_step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one_step()
    dt = (time.perf_counter() - t0) / args.steps
    value = sbytes / dt / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": max(args.warmup, 3),
            "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1) pool of the same shape)",
            "config": step_config(args, w, unique, fp8, 1, 0, sbytes, dbytes, world),
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads,
                             "kind": "oracle",
                             "sample": f"the whole {args.workload} step per step: host slot "
                                       f"mapping and cache write of {w.num_seqs} tokens, then "
                                       f"all {w.num_seqs * w.num_kv_heads} (sequence, kv-head) "
                                       f"decode units, fp64, {threads} threads"},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
