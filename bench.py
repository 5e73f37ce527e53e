"""Benchmark of one flat ragged paged-attention step on GB300 (one JSON line on stdout).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload decode|mixed|longtail|prefix|prefill|long16k]
                    [--kv bf16|fp8] [--no-mixed] [--no-extras]

A step is the whole hot path over one batch of synthetic input: the KV-write scatter of the
step's new K/V rows, then paged attention for every query row (plus the fixed-order split
combine). The timed workload is the decode batch (Hq 32, Hkv 8, D 128, block 16, 64 decode
rows, ctx ~ lognormal(median 2048, sigma 1) clipped to [16, 16384]); the metric is decode KV
GB/s: algorithmic K/V bytes read per step (sum ctx * 2 * Hkv * D * 2 B) / step time. The
mixed ragged step (48 decode rows + 4 x 512 prefill rows) is reported alongside as tokens/s.

Inputs are resident in HBM before timing. The decode K/V pools (0.84 GB) exceed the 129 MB L2,
so no flush runs between timed steps; a workload whose K/V fit in L2 twice over (prefill
segments) is flushed by a 256 MiB write between timed steps. Timing: CUDA events on the
launching stream around each step, W untimed warm-up steps, max over ranks. The timed steps
replay CUDA graphs captured from the same library calls, so no host launch overhead sits
inside the timed region: the step is one graph (the KV write, then attention + combine as its
programmatic dependents, as the library's pipeline runs a step); the attention kernels alone
(the roofline) are timed in a second pass, their graph between the events and the write's
outside. The e2e leg runs steps through the public pipeline from host buffers, planning
included.

The default run also reports, each under its own key with its own roofline, clocks and
launch count: decode_16k (32 decode rows at ctx 16,384), prefill_segments (the mixed step's
four 512-row prefill segments, tensor roofline), longtail (the long-tail rollout decode) and
prefix_shared (samples sharing their prompts' blocks; roofline on the unique K/V bytes).

The CPU baseline (and --impl reference) times the oracle (fp64 numpy, as it stands) on every
host core: a spawn-started process pool over shared memory, whole passes over the same
workload for about --cpu-budget seconds, with the same metric and unit.

Under torchrun (N > 1) every rank runs its own decode batch (seed + rank) with no data-path
collective: the path shards by sequence, so scaling is weak.

--workload selects another of the synthetic workloads for the same JSON line (the default,
decode, is the headline): longtail (Hq 64, bs 32, 115 rows of 1k-4k and 13 of 16k-40k
context), prefix (16 prompts x 8 samples sharing 64 read-only blocks; the roofline counts the
unique K/V bytes), mixed (value in tokens/s) and prefill (the mixed step's four 512-row
prefill segments alone, tokens/s, tensor roofline).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from continuous_batching_gb300 import workloads as wl  # noqa: E402

METRIC = "paged-attn decode KV GB/s (% of HBM peak) and ragged-step tokens/s, 1×GB300"
UNIT = "GB/s"
WORKLOAD = ("decode batch: Hq=32, Hkv=8, D=128, block_size=16, 64 decode rows, ctx lognormal "
            "(median 2048, sigma 1.0) clipped to [16,16384], pool = sum(ceil(ctx/16)) blocks, "
            "permuted tables, bf16 ~N(0,1), seed 1")
MIXED = ("mixed ragged step: 48 decode rows (ctx lognormal median 3000, cap 16384) + 4 chunked-"
         "prefill segments of 512 rows at prior offsets {0,512,4096,9000}, T=2096, seed 2")


L2_BYTES = 129 << 20


def kv_bytes(st: wl.Step, elem_bytes: int = 2) -> int:
    return int(st.ctx_lens.astype(np.int64).sum()) * 2 * st.Hkv * st.D * elem_bytes


def prefill_flops(st: wl.Step) -> float:
    f = 0.0
    for s in range(st.B):
        n = int(st.n_q[s])
        if n > 1:
            o = int(st.ctx_lens[s]) - n
            f += 4.0 * st.D * st.Hq * (n * o + n * (n + 1) / 2)
    return f


WORKLOADS = {
    "decode": WORKLOAD,
    "mixed": MIXED,
    "longtail": ("long-tail rollout decode: Hq=64, Hkv=8, D=128, block_size=32, 128 decode rows, "
                 "115 ctx U[1k,4k] + 13 ctx U[16k,40k] at seeded positions, permuted tables, "
                 "bf16 ~N(0,1), seed 3"),
    "prefix": ("prefix-shared GRPO decode: Hq=32, Hkv=8, D=128, block_size=16, 16 prompts of 1024 "
               "tokens x 8 samples sharing the prompt's 64 read-only blocks + own U[1,3000] "
               "continuation, 128 decode rows, bf16 ~N(0,1), seed 4"),
    "prefill": ("prefill segments: the mixed step's 4 chunked-prefill segments of 512 rows at "
                "prior offsets {0,512,4096,9000} alone, Hq=32, Hkv=8, D=128, block_size=16, causal, "
                "T=2048, seed 2"),
    "long16k": ("16k-context decode: Hq=32, Hkv=8, D=128, block_size=16, 32 decode rows all at ctx "
                "16384, pool = 32*1024 blocks, permuted tables, bf16 ~N(0,1), seed 5"),
}
# reported beside the headline in the default run, each with its own roofline: the 16k-context
# decode and the prefill segments (the two targets of the path), the long-tail rollout and the
# prefix-shared decode
EXTRAS = (("decode_16k", "long16k"), ("prefill_segments", "prefill"), ("longtail", "longtail"),
          ("prefix_shared", "prefix"))
# the value of these workloads is tokens/s (ragged steps); the others report KV GB/s
TOKEN_WORKLOADS = ("mixed", "prefill")


def unique_kv_bytes(st: wl.Step) -> int:
    """K/V bytes that must leave HBM once: token rows of distinct blocks (shared blocks once)."""
    used = {}
    bs = st.block_size
    for s in range(st.B):
        L = int(st.ctx_lens[s])
        for j in range((L + bs - 1) // bs):
            b = int(st.block_table[s, j])
            used[b] = max(used.get(b, 0), min(bs, L - j * bs))
    return sum(used.values()) * 2 * st.Hkv * st.D * 2


def make_workload(name: str, rank: int) -> wl.Step:
    if name == "prefill":
        m = wl.make_config("mixed", seed=rank_seed("mixed", rank))
        st, _ = wl.subset(m, range(48, 52), name="prefill")
        return st
    return wl.make_config(name, seed=rank_seed(name, rank))


def load_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "src": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "src": "fallback"}


def kernel_source_hash() -> str:
    """Hash of the attention kernel's code (its sources and the ABI header it includes) with
    comments and blank space removed, so that a comment edit does not void the traffic records
    taken on the same code."""
    h = hashlib.sha256()
    csrc = "continuous_batching_gb300/csrc/"
    for f in (csrc + "attention.cu", csrc + "tmem_ldst.h", csrc + "common.h",
              "include/pagedattn.h"):
        src = open(os.path.join(ROOT, f)).read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        src = re.sub(r"//[^\n]*", " ", src)
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()[:16]


def measured_traffic(workload: str = "decode"):
    """DRAM bytes per attention launch from the committed ncu summary, if it was taken on the
    current kernel source (else None)."""
    p = os.path.join(ROOT, "profiles", f"attention_{workload}_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    if d.get("kernel_source_sha256_16") != kernel_source_hash():
        return None
    return d.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock / throttle samples taken while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self) -> dict:
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------------------ GPU arm

class GpuStep:
    """Device-resident inputs for one workload plus the public-API runner."""

    def __init__(self, st: wl.Step, torch, bd, kv: str = "bf16"):
        self.st, self.torch, self.bd = st, torch, bd
        dev = lambda a: torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16)
        self.shape = bd.Shape.make(st.Hq, st.Hkv, st.D, st.block_size, st.num_blocks)
        self.kp, self.vp = dev(st.k_pool), dev(st.v_pool)
        self.kv_scales = None
        if kv == "fp8":
            # the cache holds float8_e4m3fn codes with per-tensor scales (amax / 448); the
            # synthetic bf16 pool is quantised once, before timing, by the library's own write
            ks = float(self.kp.abs().max().float().item()) / 448.0
            vs = float(self.vp.abs().max().float().item()) / 448.0
            self.kv_scales = (float(np.float32(ks)), float(np.float32(vs)))
            n = st.num_blocks * st.block_size
            kp8 = torch.empty(self.kp.shape, dtype=torch.uint8, device="cuda")
            vp8 = torch.empty(self.vp.shape, dtype=torch.uint8, device="cuda")
            all_slots = torch.arange(n, dtype=torch.int32, device="cuda")
            bd.paged_kv_write_fp8(self.kp.view(n, st.Hkv, st.D), self.vp.view(n, st.Hkv, st.D),
                                  all_slots, kp8, vp8, *self.kv_scales, self.shape)
            torch.cuda.synchronize()
            self.kp, self.vp = kp8, vp8
        self.q, self.kn, self.vn = dev(st.q), dev(st.k_new), dev(st.v_new)
        self.out = torch.empty((st.T, st.Hq, st.D), dtype=torch.bfloat16, device="cuda")
        self.runner = bd.StepRunner(self.shape, kv_scales=self.kv_scales).prepare(
            st.cu_seqlens_q, st.ctx_lens, st.block_table)
        # the timed steps replay CUDA graphs of the same calls (fixed buffers, padded plan):
        # one graph for the KV write, one for the attention kernels
        lim = bd.StepLimits(B=st.B, T=st.T, max_blocks=st.block_table.shape[1],
                            max_ctx=int(st.ctx_lens.max()))
        self.graph_runner = bd.StepRunner(self.shape, limits=lim,
                                          kv_scales=self.kv_scales).prepare(
            st.cu_seqlens_q, st.ctx_lens, st.block_table)
        self.g_write = self.graph_runner.capture(self.q, self.kn, self.vn, self.kp, self.vp,
                                                 self.out, attend=False)
        self.g_attend = self.graph_runner.capture(self.q, self.kn, self.vn, self.kp, self.vp,
                                                  self.out, write=False)
        # and the whole step in one graph, as the library's pipeline runs it: the attention is
        # launched as a programmatic dependent of the KV write, so its start overlaps the write
        self.g_step = self.graph_runner.capture(self.q, self.kn, self.vn, self.kp, self.vp,
                                                self.out)
        # pinned host copies for the end-to-end measurement, and the public pipeline that runs
        # steps from them (two buffer sets, so that one step's host work and copies overlap the
        # kernels of the step before it)
        pin = lambda a: torch.from_numpy(a.view(np.int16).copy()).pin_memory()
        self.h_q, self.h_kn, self.h_vn = pin(st.q), pin(st.k_new), pin(st.v_new)
        self.h_out = [torch.empty((st.T, st.Hq, st.D), dtype=torch.int16).pin_memory()
                      for _ in range(2)]
        self.pipe = bd.StepPipeline(self.shape, lim, self.kp, self.vp, kv_scales=self.kv_scales)

    def launches_per_step(self) -> int:
        """kv_write_kernel, paged_attn_kernel, and the split combine when a context spans more
        than one split (the rule paged_attention_step applies)."""
        comb = 1 if int(self.st.ctx_lens.max()) > self.bd.PA_SPLIT_TOKENS else 0
        return 2 + comb

    def step(self):
        self.runner.run(self.q, self.kn, self.vn, self.kp, self.vp, self.out)

    def submit_e2e(self, i: int):
        """Step i through the public pipeline from host buffers: plan and slots on the host, one
        pinned metadata upload, pinned H2D of the new tokens' q / k / v, the captured KV write
        and attention, D2H of the output. Returns the event after which its output is on the
        host."""
        st = self.st
        return self.pipe.submit(st.cu_seqlens_q, st.ctx_lens, st.block_table, self.h_q,
                                self.h_kn, self.h_vn, self.h_out[i % 2])

    def run_e2e(self, n: int) -> float:
        """n steps end to end, each step's output read back before its host buffer is reused;
        returns seconds per step (wall clock from the first submission to the last output)."""
        pending = []
        t0 = time.perf_counter()
        for i in range(n):
            pending.append(self.submit_e2e(i))
            if len(pending) > 1:
                pending.pop(0).synchronize()          # the previous step's output is on the host
        while pending:
            pending.pop(0).synchronize()
        return (time.perf_counter() - t0) / n

    def e2e_bytes(self):
        st = self.st
        h2d = st.q.nbytes + st.k_new.nbytes + st.v_new.nbytes + self.pipe.meta_bytes
        return h2d, st.T * st.Hq * st.D * 2


def hold_gpu(torch, seconds: float) -> None:
    """Keeps the current stream busy for about `seconds` (a spin kernel; 2.1 GHz assumed)."""
    torch.cuda._sleep(int(seconds * 2.1e9))


def time_steps(g: GpuStep, torch, steps: int, warmup: int, flush, attn_only=False):
    """Per-step CUDA events around replays of the captured graphs, L2 flushed before each step
    when `flush` is given (outside the events). First the whole step as one graph (the KV write,
    then the attention as its programmatic dependent, as the library's pipeline runs a step),
    then the attention kernels alone: the write graph outside the events, the attention graph
    between them. Returns (per-step ms list, per-attention-call ms list)."""
    s = torch.cuda.current_stream()
    for _ in range(warmup):
        g.g_step.replay()
        g.g_write.replay()
        g.g_attend.replay()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(2 * steps)]
    # hold the GPU (outside every timed interval) while the host queues all timed steps, so
    # that no interval includes the GPU waiting for the host to enqueue the next graph
    hold_gpu(torch, 1e-3 + 6e-4 * steps)
    for i in range(steps):
        if flush is not None:
            flush.zero_()
        a, c = ev[i]
        a.record(s)
        g.g_step.replay()
        c.record(s)
    for i in range(steps):
        if flush is not None:
            flush.zero_()
        g.g_write.replay()
        b, c = ev[steps + i]
        b.record(s)
        g.g_attend.replay()
        c.record(s)
    torch.cuda.synchronize()
    step_ms = [a.elapsed_time(c) for a, c in ev[:steps]]
    attn_ms = [b.elapsed_time(c) for b, c in ev[steps:]]
    return step_ms, attn_ms


def rank_seed(name: str, rank: int) -> int:
    """Each rank of a multi-GPU run draws its own batch of the same workload."""
    base = {"decode": 1, "mixed": 2, "longtail": 3, "prefix": 4, "long16k": 5}[name]
    return base + rank


def combine_ranks(total_ms: float, units: float, dist=None, device="cpu"):
    """Whole-job timing over ranks: (max of the ranks' timed totals, sum of their work units).
    Ranks share nothing on the data path; this is the only cross-rank step."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return total_ms, units
    import torch
    t = torch.tensor([total_ms], dtype=torch.float64, device=device)
    u = torch.tensor([units], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def roofline_for(name: str, st: wl.Step, attn_ms: float, peaks: dict, fp8_kv: bool) -> dict:
    """Roofline of the attention launches (attention kernel + split combine) of one step:
    algorithmic bytes (K/V read once; unique bytes for the prefix-shared workload) against
    the measured copy bandwidth, or, for the prefill segments, causal algorithmic FLOPs
    against the measured bf16 tensor peak (burst: the kernel is timed by itself)."""
    traffic = measured_traffic(name + ("_fp8" if fp8_kv else ""))
    if name == "prefill":
        achieved = prefill_flops(st) / (attn_ms * 1e-3) / 1e12
        return {"bound": "tensor", "achieved": round(achieved, 1), "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_tflops"], 4),
                "traffic": traffic,
                "kernel": "paged_attention_step (tile routine), causal algorithmic FLOPs "
                          "4*D*Hq*(n*o + n(n+1)/2)",
                "peak_src": peaks["src"] + " (burst)"}
    bytes_step = kv_bytes(st, 1 if fp8_kv else 2)
    roof_bytes = (unique_kv_bytes(st) // (2 if fp8_kv else 1) if name == "prefix"
                  else bytes_step)
    achieved = roof_bytes / (attn_ms * 1e-3) / 1e9
    roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
            "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
            "traffic": traffic,
            "kernel": "paged_attention_step (attention kernels + split combine)",
            "peak_src": peaks["src"]}
    if name == "prefix":
        roof["bytes"] = "unique K/V bytes (shared prompt blocks counted once)"
        roof["logical_gbs"] = round(bytes_step / (attn_ms * 1e-3) / 1e9, 1)
    return roof


def measure_extra(name: str, rank: int, torch, bd, args, peaks: dict, flush) -> dict:
    """One more workload, timed like the headline (graph replays, CUDA events, the same L2
    rule), with the clocks sampled over its own loaded window."""
    st = make_workload(name, rank)
    fp8_kv = args.kv == "fp8"
    g = GpuStep(st, torch, bd, args.kv)
    bytes_step = kv_bytes(st, 1 if fp8_kv else 2)
    needs_flush = bytes_step < 2 * L2_BYTES
    torch.cuda.synchronize()
    with ClockSampler(int(os.environ.get("LOCAL_RANK", "0"))) as clk:
        if not args.no_clocks:
            load_for(g, torch, 0.6)
        step_ms, attn_ms = time_steps(g, torch, args.steps, args.warmup,
                                      flush if needs_flush else None)
        if not args.no_clocks:
            load_for(g, torch, 0.6)
    ms = statistics.mean(step_ms)
    tokens = name in TOKEN_WORKLOADS
    out = {"workload": WORKLOADS[name],
           "value": round(st.T / (ms * 1e-3), 1) if tokens else round(bytes_step / (ms * 1e-3) / 1e9, 2),
           "unit": "tokens/s" if tokens else UNIT, "ms_per_step": round(ms, 5),
           "attention_ms": round(statistics.mean(attn_ms), 5),
           "roofline": roofline_for(name, st, statistics.mean(attn_ms), peaks, fp8_kv),
           "l2": "flushed by a 256 MiB write between timed steps" if needs_flush else
                 "inputs larger than L2, no flush",
           "gpu_launches": g.launches_per_step() * args.steps, "clocks": clk.summary()}
    del g
    torch.cuda.empty_cache()
    return out


def load_for(g: GpuStep, torch, seconds: float) -> None:
    t = time.perf_counter()
    while time.perf_counter() - t < seconds:
        for _ in range(20):
            g.step()
        torch.cuda.synchronize()


def run_ours(args) -> dict:
    import torch

    from continuous_batching_gb300 import binding as bd
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    bd.load()
    peaks = load_peaks()

    name = args.workload
    st = make_workload(name, rank)
    fp8_kv = args.kv == "fp8"
    g = GpuStep(st, torch, bd, args.kv)
    # Between timed steps L2 is flushed by a 256 MiB write only when the step's K/V fit in L2
    # twice over (the prefill workload); the other workloads read 0.36-2.7 GB of K/V per step,
    # far more than the 129 MB L2 holds, and are timed without a flush (a write flush leaves
    # about 126 MB of dirty lines whose write-back would land inside the timed step)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    barrier()
    with ClockSampler(local) as clk:
        # keep the GPU under the same load for about a second on both sides of the timed
        # region so that the 200 ms clock samples cover it
        if not args.no_clocks:
            load_for(g, torch, 1.0)
        barrier()
        t0 = time.perf_counter()
        needs_flush = kv_bytes(st, 1 if fp8_kv else 2) < 2 * L2_BYTES
        step_ms, attn_ms = time_steps(g, torch, args.steps, args.warmup,
                                      flush if needs_flush else None)
        barrier()
        wall = time.perf_counter() - t0
        if not args.no_clocks:
            load_for(g, torch, 1.0)
    tokens = name in TOKEN_WORKLOADS
    bytes_step = kv_bytes(st, 1 if fp8_kv else 2)
    units_step = float(st.T) if tokens else float(bytes_step)
    unit = "tokens/s" if tokens else UNIT
    scale = 1.0 if tokens else 1e-9
    dist_mod = None
    if world > 1:
        import torch.distributed as dist_mod
    total_ms, all_units = combine_ranks(sum(step_ms), units_step, dist_mod, "cuda")
    ms_per_step = total_ms / args.steps
    value = all_units / (ms_per_step * 1e-3) * scale

    # end to end through the public API with host buffers (StepPipeline)
    g.run_e2e(4)
    e2e_s = g.run_e2e(max(8, args.steps))
    h2d, d2h = g.e2e_bytes()

    attn_avg = statistics.mean(attn_ms)
    roof = roofline_for(name, st, attn_avg, peaks, fp8_kv)

    # the mixed ragged step (tokens/s) alongside the decode headline
    mixed = None
    if name == "decode" and not args.no_mixed:
        sm = wl.make_config("mixed", seed=rank_seed("mixed", rank))
        gm = GpuStep(sm, torch, bd, args.kv)
        m_step, m_attn = time_steps(gm, torch, args.steps, args.warmup,
                                    flush if kv_bytes(sm, 1 if fp8_kv else 2) < 2 * L2_BYTES
                                    else None)
        mm = statistics.mean(m_step)
        pf = prefill_flops(sm)
        mixed = {"workload": MIXED, "tokens_per_s": round(sm.T / (mm * 1e-3), 1),
                 "ms_per_step": round(mm, 4),
                 "prefill_algorithmic_tflop_per_s_over_whole_step": round(pf / (mm * 1e-3) / 1e12, 2),
                 "tensor_peak_tflops": peaks["bf16_tflops"]}
        del gm

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": unit, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 (K/V as fp8 e4m3 codes, f16 MMA operands)" if fp8_kv else "bf16",
        "data": "synthetic",
        "config": {"workload": WORKLOADS[name], "kv_bytes_per_step": bytes_step, "T": st.T,
                   "kv_cache": ("float8_e4m3fn codes, per-tensor scales "
                                f"{g.kv_scales[0]:.6g} / {g.kv_scales[1]:.6g}") if fp8_kv else "bf16",
                   "l2": (f"inputs fit L2 ({bytes_step / 1e9:.3f} GB K/V): L2 flushed by a 256 MiB "
                          "write between timed steps") if needs_flush else
                         (f"inputs larger than L2 ({bytes_step / 1e9:.2f} GB K/V per step, L2 "
                          "129 MB), no flush between timed steps"),
                   "parallelism": f"replicas{world}"},
        "e2e": {"value": round(units_step / e2e_s * scale, 2), "unit": unit,
                "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "ms_per_step": round(e2e_s * 1e3, 4)},
        "roofline": roof,
        "gpu_launches": g.launches_per_step() * args.steps,
        "clocks": clk.summary(),
        "wall_s_timed_region": round(wall, 3),
    }
    if mixed:
        line["ragged_step"] = mixed
    if name == "decode" and not args.no_extras:
        for key, ex in EXTRAS:
            line[key] = measure_extra(ex, rank, torch, bd, args, peaks, flush)
    if rank == 0 and not args.no_cpu_baseline and not fp8_kv:
        line["cpu_baseline"] = cpu_baseline(st, budget_s=args.cpu_budget, tokens=tokens)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return line if rank == 0 else None


# ---------------------------------------------------------------------- CPU oracle arm

_CPU = {}


def _cpu_worker_init(specs: dict, Hq: int) -> None:
    """Worker of the CPU baseline: attaches to the step's arrays in shared memory (no copy)."""
    from multiprocessing import shared_memory
    for name, (shm_name, shape, dtype) in specs.items():
        shm = shared_memory.SharedMemory(name=shm_name)
        _CPU[name + "_shm"] = shm
        _CPU[name] = np.ndarray(shape, np.dtype(dtype), buffer=shm.buf)
    _CPU["Hq"] = Hq


def _cpu_worker_run(rows) -> int:
    import oracle.paged_attention as pa
    c = _CPU
    pa.attention_rows(c["q"], c["k_pool"], c["v_pool"], c["block_table"], c["cu_seqlens_q"],
                      c["ctx_lens"], c["Hq"], rows)
    return len(rows)


class OraclePool:
    """The oracle (fp64 numpy, as it stands) on every host core: a pool of `workers` processes
    (default os.cpu_count()), started with spawn, shares the step's arrays through shared
    memory and computes whole query groups (KV workloads: one sequence per task, longest
    first; token workloads: 8 query rows per task)."""

    def __init__(self, st: wl.Step, tokens: bool = False, workers: int = 0):
        import multiprocessing as mp
        from multiprocessing import shared_memory
        self.st, self.tokens = st, tokens
        self.n_workers = workers or os.cpu_count() or 1
        if tokens:
            self.groups = [np.arange(i, min(i + 8, st.T)) for i in range(0, st.T, 8)]
        else:
            order = np.argsort(-st.ctx_lens, kind="stable")
            self.groups = [np.arange(st.cu_seqlens_q[s], st.cu_seqlens_q[s + 1]) for s in order]
        seq_of = np.searchsorted(st.cu_seqlens_q, np.arange(st.T), side="right") - 1
        self.pass_bytes = sum(int(st.ctx_lens[seq_of[r[0]]]) * 2 * st.Hkv * st.D * 2 * len(r)
                              for r in self.groups if len(r))
        self.shms, specs = [], {}
        # one BLAS / OpenMP thread per worker process (the oracle's einsums run in numpy's
        # own loops; the pool supplies the parallelism)
        saved = {k: os.environ.get(k) for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS",
                                                "MKL_NUM_THREADS")}
        try:
            for name in ("q", "k_pool", "v_pool", "block_table", "cu_seqlens_q", "ctx_lens"):
                a = np.ascontiguousarray(getattr(st, name))
                shm = shared_memory.SharedMemory(create=True, size=max(a.nbytes, 1))
                np.ndarray(a.shape, a.dtype, buffer=shm.buf)[...] = a
                self.shms.append(shm)
                specs[name] = (shm.name, a.shape, a.dtype.str)
            for k in saved:
                os.environ[k] = "1"
            self.pool = mp.get_context("spawn").Pool(
                self.n_workers, initializer=_cpu_worker_init, initargs=(specs, st.Hq))
            # every worker started and attached before anything is timed
            self.pool.map(_cpu_worker_run, [np.zeros(0, np.int64)] * self.n_workers)
        except BaseException:
            self.close()
            raise
        finally:
            for k, v in saved.items():
                if v is None:
                    os.environ.pop(k, None)
                else:
                    os.environ[k] = v

    def run(self, budget_s: float) -> dict:
        """Full passes over the workload until about budget_s of wall time has gone by (at
        least one); the value is their K/V bytes (or query rows) over that wall time."""
        st = self.st
        passes, rows_done = 0, 0
        t0 = time.perf_counter()
        while True:
            rows_done += sum(self.pool.imap_unordered(_cpu_worker_run, self.groups, chunksize=1))
            passes += 1
            if time.perf_counter() - t0 > budget_s:
                break
        dt = time.perf_counter() - t0
        where = (f"numpy fp64 oracle in {self.n_workers} spawned worker processes (host has "
                 f"{os.cpu_count()} cores), one BLAS/OpenMP thread each")
        if self.tokens:
            return {"value": round(rows_done / dt, 2), "unit": "tokens/s", "cores": self.n_workers,
                    "kind": "oracle", "blas_threads_per_worker": 1,
                    "sample": f"{passes} full pass(es) over all {st.T} query rows (tasks of 8 rows, "
                              f"all {st.Hq} heads) in {dt:.1f} s; {where}"}
        return {"value": round(passes * self.pass_bytes / dt / 1e9, 4), "unit": UNIT,
                "cores": self.n_workers, "kind": "oracle", "blas_threads_per_worker": 1,
                "sample": f"{passes} full pass(es) over all {st.B} decode rows (one sequence per "
                          f"task, all {st.Hq} heads), {passes * self.pass_bytes / 1e9:.3f} GB of K/V "
                          f"in {dt:.1f} s; {where}"}

    def close(self):
        pool = getattr(self, "pool", None)
        if pool is not None:
            pool.terminate()
            pool.join()
            self.pool = None
        for shm in getattr(self, "shms", []):
            shm.close()
            shm.unlink()
        self.shms = []

    def __enter__(self):
        return self

    def __exit__(self, *a):
        self.close()


def cpu_baseline(st: wl.Step, budget_s: float = 10.0, tokens: bool = False,
                 workers: int = 0) -> dict:
    """The oracle timed on every host core (OraclePool) for about budget_s of wall time."""
    with OraclePool(st, tokens, workers) as op:
        return op.run(budget_s)


def run_reference(args) -> dict:
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return None
    name = args.workload
    st = make_workload(name, 0)
    tokens = name in TOKEN_WORKLOADS
    per = max(1.0, min(20.0, 90.0 / max(args.steps, 1)))
    vals = []
    with OraclePool(st, tokens) as op:
        for _ in range(args.warmup):
            op.run(0.0)                                  # one pass each
        t0 = time.perf_counter()
        for _ in range(args.steps):
            vals.append(op.run(per))
        wall = time.perf_counter() - t0
    v = statistics.mean(x["value"] for x in vals)
    base = vals[0]
    base["value"] = round(v, 4)
    unit = base["unit"]
    return {"impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": unit,
            "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(wall / args.steps * 1e3, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": WORKLOADS[name]},
            "cpu_baseline": base,
            "e2e": {"value": round(v, 4), "unit": unit, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="decode", choices=sorted(WORKLOADS),
                    help="synthetic workload of the timed step (decode is the headline)")
    ap.add_argument("--no-mixed", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the 16k-decode, prefill-segment and long-tail lines that the "
                         "default (decode) run reports beside the headline")
    ap.add_argument("--kv", default="bf16", choices=["bf16", "fp8"],
                    help="KV cache type: bf16, or float8_e4m3fn codes with per-tensor scales "
                         "(head_dim 128 workloads)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--no-clocks", action="store_true",
                    help="skip the loaded windows around the timed region that the clock "
                         "samples need (for profiler runs)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    line = run_reference(args) if args.impl == "reference" else run_ours(args)
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
