#!/usr/bin/env python
"""Benchmark of the chunked-prefill causal attention hot path on one GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                    [--workload gqa_prefill|decode|mixed|rolling|fp32] [--no-pad]

Default workload (the one the headline metric is quoted on): one GQA layer,
32 query / 8 KV heads, head_dim 128, bf16, a 4000-token prompt prefilled in
chunks of 512 (7 x 512 + 416) into a KV cache of physical capacity 8192.  One
step is the whole path for one prompt: chunk plan, query-width ladder (the
416-row tail is widened to 512 by repeating its last row), and per chunk the
KV append, the chunk attention and the commit of seqlens_k to past + real
rows, made as one cp_prefill_chunk call (two kernels: the append, then the
attention, which also advances seqlens_k).  Each step is one replay of a CUDA
graph captured from the library's public calls; L2 is flushed (512 MiB write)
between timed steps.

Prints one JSON line (rank 0).  ``--impl reference`` times the CPU oracle
(test infrastructure, float64 numpy) on a bounded sample of the same
workload instead.  Other workloads (decode rows, mixed step) print the same
kind of line with their own metric.
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
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "chunked-prefill attn tokens/s & effective TFLOP/s; % of GB300 BF16/HBM roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=3000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", default="native", choices=["native", "reference"])
    p.add_argument("--workload", default="gqa_prefill", choices=["gqa_prefill", "decode", "mixed", "rolling", "fp32"])
    p.add_argument("--no-pad", action="store_true", help="do not widen chunks to the query-width ladder")
    p.add_argument("--cpu-seconds", type=float, default=12.0, help="CPU-baseline sample budget")
    p.add_argument("--skip-cpu", action="store_true")
    return p.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# --------------------------------------------------------------------------- distributed

def dist_init(n_gpus):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    """The largest value of x over all ranks (the slowest rank's time)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(local_ms, units_per_step, steps, world):
    """Whole-job throughput of `world` replicas: every rank processes
    `units_per_step` units per step, the job takes as long as the slowest rank.
    Returns (max_ms_over_ranks, units per second over all ranks)."""
    total_ms = max_over_ranks(local_ms, world)
    return total_ms, world * units_per_step * steps / (total_ms / 1e3)


# --------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id=None):
        self.proc = None
        self.bus_id = bus_id
        self.path = tempfile.mktemp(prefix="clocks_", suffix=".csv")

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
        if self.bus_id:
            cmd += ["-i", self.bus_id]
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(cmd, stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9 and parts[1].replace(".", "").isdigit():
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for name, val in zip(names, r[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": float(rows[0][2]),
                "power_w_max": max(float(r[3]) for r in rows if r[3].replace(".", "").isdigit()),
                "samples": len(rows), "reasons": sorted(reasons)}


# --------------------------------------------------------------------------- helpers

def kernel_traffic(kernel_file, profile_name):
    """DRAM bytes per launch recorded in profiles/<profile_name> for the kernel
    source it was measured on; None when the source has changed since."""
    prof = os.path.join(ROOT, "profiles", profile_name)
    if not os.path.exists(prof):
        return None
    text = open(prof).read()
    m_sha = re.search(r"source_sha256:\s*([0-9a-f]{64})", text)
    m_b = re.search(r"dram_bytes_per_launch:\s*([0-9.e+]+)", text)
    if not (m_sha and m_b):
        return None
    src = os.path.join(ROOT, "chunked_prefill_causal_cp_gb300", "csrc", kernel_file)
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()
    return float(m_b.group(1)) if sha == m_sha.group(1) else None


def cpu_cores():
    return os.cpu_count() or 1


def visible_pairs(past, rows):
    """Visible (query, key) pairs of `rows` causal rows after `past` cached keys."""
    return rows * past + rows * (rows + 1) // 2


# --------------------------------------------------------------------------- workloads

class GqaPrefill:
    """The 4000-token GQA prompt, chunk 512, capacity 8192 (see module doc)."""

    N, W, HQ, HKV, D, CAP = 4000, 512, 32, 8, 128, 8192

    def __init__(self, dev, pad=True):
        import torch
        import chunked_prefill_causal_cp_gb300 as cp
        import synth_inputs as SI

        self.cp, self.torch, self.dev, self.pad = cp, torch, dev, pad
        self.sizes = cp.cp_chunk_plan(self.N, self.W)
        self.widths = [cp.cp_query_width(r, self.W) if pad else r for r in self.sizes]
        self.rows_alloc = sum(self.sizes[:-1]) + self.widths[-1]
        q, k, v = SI.gqa_prompt(self.N, seed=1)
        self.host_q, self.host_k, self.host_v = q, k, v
        bf = torch.bfloat16
        self.q = torch.zeros(self.rows_alloc, self.HQ, self.D, dtype=bf, device=dev)
        self.k = torch.zeros(self.rows_alloc, self.HKV, self.D, dtype=bf, device=dev)
        self.v = torch.zeros(self.rows_alloc, self.HKV, self.D, dtype=bf, device=dev)
        self.q[:self.N].copy_(q)
        self.k[:self.N].copy_(k)
        self.v[:self.N].copy_(v)
        self.out = torch.zeros(self.rows_alloc, self.HQ, self.D, dtype=bf, device=dev)
        self.desc = cp.layer_desc(bf, 1, self.HQ, self.HKV, self.D, cp.CP_CACHE_CONTIG, capacity=self.CAP)
        self.kc = torch.zeros(1, self.HKV, self.CAP, self.D, dtype=bf, device=dev)
        self.vc = torch.zeros_like(self.kc)
        self.lens = torch.zeros(1, dtype=torch.int32, device=dev)
        self.pasts = torch.tensor([0] + list(torch.tensor(self.sizes).cumsum(0)[:-1].tolist()),
                                  dtype=torch.int32, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.ws = torch.zeros(max(16, cp.cp_workspace_size(self.desc, self.W, self.CAP, 1)),
                              dtype=torch.uint8, device=dev)
        self.flops_chunk = []
        past = 0
        for r in self.sizes:
            self.flops_chunk.append(4 * self.D * self.HQ * visible_pairs(past, r))
            past += r
        self.flops = sum(self.flops_chunk)
        self.tokens = self.N
        # launches of this library per step: one pad launch (q, k and v) per widened chunk + per chunk
        # the append and the attention (which advances seqlens_k itself)
        self.launches = sum(1 for r, w in zip(self.sizes, self.widths) if w > r) + 2 * len(self.sizes)

    def _chunk(self, i, attn=True, append=True, commit=True):
        cp = self.cp
        r, w = self.sizes[i], self.widths[i]
        past = sum(self.sizes[:i])
        sl = slice(past, past + w)
        q, k, v = self.q[None, sl], self.k[None, sl], self.v[None, sl]
        if append and w > r:
            cp.cp_pad_chunk(self.desc, q, k, v, r, w)
        if append and attn and commit:  # the whole chunk in one call
            cp.cp_prefill_chunk(self.desc, q, k, v, self.kc, self.vc, self.lens, w, r, past, self.out[None, sl],
                                self.ws, dev_status=self.status)
            return
        if append:
            cp.cp_kv_append(self.desc, k, v, w, self.kc, self.vc, self.lens, past, dev_status=self.status)
        if attn:
            cp.cp_prefill_chunk_attn(self.desc, q, self.kc, self.vc, self.lens, w, r, past, self.out[None, sl],
                                     self.ws, commit=commit, dev_status=self.status)

    def step(self):
        self.lens.zero_()
        for i in range(len(self.sizes)):
            self._chunk(i)

    def capture(self):
        torch = self.torch
        s = torch.cuda.Stream(self.dev)
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            for _ in range(2):
                self.step()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.step()
        # per-chunk graphs for the kernel-level timing: state set-up, then attention alone
        self.setup_graphs, self.attn_graphs = [], []
        for i in range(len(self.sizes)):
            gs, ga = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
            with torch.cuda.graph(gs):
                self.lens.copy_(self.pasts[i:i + 1])
                self._chunk(i, attn=False)
            with torch.cuda.graph(ga):
                self._chunk(i, append=False, commit=False)
            self.setup_graphs.append(gs)
            self.attn_graphs.append(ga)
        self.graph = g
        return g

    def capture_e2e(self):
        """One CUDA graph of a whole step with its host traffic, pipelined the way
        a serving loop runs chunked prefill: chunk i's q/k/v rows go host ->
        device on one copy stream while chunk i-1 is computed, and chunk i's
        output rows go device -> host on another as soon as chunk i is done.
        Every input byte and every output byte of the step crosses the bus inside
        the graph; the step ends when the last output row is on the host."""
        torch = self.torch
        main = torch.cuda.Stream(self.dev)
        up, down = torch.cuda.Stream(self.dev), torch.cuda.Stream(self.dev)
        n = len(self.sizes)
        ev_in = [torch.cuda.Event() for _ in range(n)]
        ev_done = [torch.cuda.Event() for _ in range(n)]

        def body():
            self.lens.zero_()
            up.wait_stream(main)
            down.wait_stream(main)
            past = 0
            for i, r in enumerate(self.sizes):
                sl = slice(past, past + r)
                with torch.cuda.stream(up):
                    self.q[sl].copy_(self.hq[sl], non_blocking=True)
                    self.k[sl].copy_(self.hk[sl], non_blocking=True)
                    self.v[sl].copy_(self.hv[sl], non_blocking=True)
                    ev_in[i].record(up)
                main.wait_event(ev_in[i])
                self._chunk(i)
                ev_done[i].record(main)
                with torch.cuda.stream(down):
                    down.wait_event(ev_done[i])
                    self.ho[sl].copy_(self.out[sl], non_blocking=True)
                past += r
            main.wait_stream(up)
            main.wait_stream(down)

        main.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(main):
            for _ in range(2):
                body()
        torch.cuda.current_stream().wait_stream(main)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=main):
            body()
        self.e2e_graph = g
        return g

    def pin(self):
        self.hq = self.host_q.pin_memory()
        self.hk = self.host_k.pin_memory()
        self.hv = self.host_v.pin_memory()
        self.ho = self.torch.empty(self.N, self.HQ, self.D, dtype=self.torch.bfloat16).pin_memory()
        self.h2d = (self.hq.numel() + self.hk.numel() + self.hv.numel()) * 2
        self.d2h = self.ho.numel() * 2

    def config(self):
        return {"workload": "gqa32x8_d128_bf16_prompt4000_chunk512_cap8192",
                "model": "single GQA attention layer (synthetic N(0,1) q/k/v)",
                "prompt_tokens": self.N, "chunk": self.W, "chunks": self.sizes,
                "query_widths": self.widths, "kv_capacity": self.CAP, "heads_q": self.HQ,
                "heads_kv": self.HKV, "head_dim": self.D, "global_batch": 1, "seq_len": self.N,
                "padding": "ladder" if self.pad else "none", "parallelism": "replica per GPU",
                "l2": "flushed between timed steps (512 MiB write)", "cuda_graph": True}

    def cpu_sample(self, budget_s):
        """Oracle (as it stands) on whole KV-head groups of the same prompt until
        the time budget is spent; returns (tokens/s scaled to all heads, sample)."""
        import numpy as np
        import oracle
        q = self.host_q.double().numpy()
        k = self.host_k.double().numpy()
        v = self.host_v.double().numpy()
        G = self.HQ // self.HKV
        t0 = time.perf_counter()
        groups = 0
        while groups < self.HKV:
            g = groups
            oracle.chunked_prefill(q[:, g * G:(g + 1) * G], k[:, g:g + 1], v[:, g:g + 1], self.W)
            groups += 1
            if time.perf_counter() - t0 > budget_s:
                break
        t = time.perf_counter() - t0
        full = t * self.HKV / groups
        sample = (f"oracle.chunked_prefill of the 4000-token prompt (chunks {self.sizes[0]}x"
                  f"{len(self.sizes) - 1}+{self.sizes[-1]}, unpadded) for {groups} of {self.HKV} KV-head "
                  f"groups ({groups * G} of {self.HQ} query heads), {t:.1f} s, scaled to all heads")
        return self.N / full, sample, t


def time_steps(run_step, flush, steps, torch):
    """Per-step CUDA-event times (ms) on the current stream, L2 flushed between."""
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        flush.zero_()
        starts[i].record()
        run_step()
        ends[i].record()
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in zip(starts, ends)]


def run_native(args):
    import torch
    rank, world, local = dist_init(args.gpus)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    from chunked_prefill_causal_cp_gb300 import _build
    if rank == 0 or world == 1:
        _build.build()
    barrier(world)
    import chunked_prefill_causal_cp_gb300 as cp
    cp.lib()
    pk, pk_src = peaks()
    if args.workload in ("rolling", "fp32"):
        return run_chunk_loop(args, rank, world, dev, pk, pk_src)
    if args.workload != "gqa_prefill":
        return run_paged(args, rank, world, dev, pk, pk_src)

    wl = GqaPrefill(dev, pad=not args.no_pad)
    wl.capture()
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    for _ in range(max(args.warmup, 3)):
        wl.graph.replay()
    torch.cuda.synchronize()
    if int(wl.status.item()) != 0:
        raise RuntimeError(f"device status {int(wl.status.item())}")

    bus = None
    try:
        bus = torch.cuda.get_device_properties(dev).pci_bus_id
    except AttributeError:
        pass
    clocks = ClockSampler(bus)
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    times = time_steps(wl.graph.replay, flush, args.steps, torch)
    clk = clocks.stop()
    torch.cuda.synchronize()
    barrier(world)
    total_ms, value = job_throughput(sum(times), wl.tokens, args.steps, world)
    ms_per_step = total_ms / args.steps

    # ---- kernel-level timing of the attention kernel (per chunk, same state as in the step).
    # A short spin kernel (no memory traffic) keeps the GPU busy while the start
    # event, the one-kernel graph and the end event are enqueued, so the events
    # bracket the kernel's execution and not the host's launch latency.
    reps = 20
    spin_cycles = int(30e-6 * float(pk.get("sm_max_mhz", 2070.0)) * 1e6)
    attn_ms = [0.0] * len(wl.sizes)
    for _ in range(reps):
        for i in range(len(wl.sizes)):
            wl.setup_graphs[i].replay()
            torch.cuda._sleep(spin_cycles)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            wl.attn_graphs[i].replay()
            e1.record()
            e1.synchronize()
            attn_ms[i] += e0.elapsed_time(e1) / reps
    attn_tflops = wl.flops / (sum(attn_ms) / 1e3) / 1e12
    peak = float(pk["bf16_tflops"])
    traffic = kernel_traffic("attn_tc.cu", "attn_tc_gqa_prefill.md")

    # ---- end to end: host buffers in, result out, through the captured public calls
    wl.pin()
    e2e_steps = max(20, min(args.steps // 10, 300))

    wl.capture_e2e()

    def e2e_step():
        wl.e2e_graph.replay()

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    e2e_times = time_steps(e2e_step, flush, e2e_steps, torch)
    _, e2e_value = job_throughput(sum(e2e_times), wl.tokens, e2e_steps, world)
    if int(wl.status.item()) != 0:
        raise RuntimeError(f"device status {int(wl.status.item())}")

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) q/k/v)",
        "config": wl.config(),
        "effective_tflops": wl.flops * args.steps * world / (total_ms / 1e3) / 1e12,
        "flops_per_step": wl.flops,
        "roofline": {"bound": "tensor", "achieved": attn_tflops, "peak": peak, "unit": "TFLOP/s",
                     "frac": attn_tflops / peak, "traffic": traffic, "kernel": "attn_tc_kernel",
                     "peak_source": f"{pk_src} bf16_tflops (burst; kernel timed alone)",
                     "frac_of_sustained": attn_tflops / float(pk.get("bf16_tflops_sustained", peak)),
                     "per_chunk_us": [round(t * 1e3, 2) for t in attn_ms],
                     "kernel_timing": ("CUDA events around a one-kernel graph of each chunk's attention, "
                                       "enqueued behind a 30 us spin kernel so launch latency is excluded; "
                                       "same cache state as in the step, mean of 20"),
                     "per_chunk_tflops": [round(f / (t / 1e3) / 1e12, 1) for f, t in zip(wl.flops_chunk, attn_ms)]},
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": wl.h2d,
                "d2h_bytes_per_step": wl.d2h,
                "path": ("one captured graph per step of the public calls with its host traffic: chunk i's "
                         "q/k/v rows pinned host -> device on a copy stream while chunk i-1 computes, chunk i's "
                         "output rows device -> pinned host on a second copy stream once chunk i is done")},
        "gpu_launches": wl.launches * args.steps,
        "clocks": clk,
    }
    if rank == 0 and world == 1 and not args.skip_cpu:
        v_cpu, sample, _ = wl.cpu_sample(args.cpu_seconds)
        line["cpu_baseline"] = {"value": v_cpu, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
                                "sample": sample}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


class PagedStep:
    """The mixed-step workload: 64 running decodes with contexts U{512..8192} in
    16-token pages (seeded page permutation), GQA 32/8 x 128 bf16.  ``decode``:
    the 64 decode rows alone.  ``mixed``: the first step of the 8192-token
    budget (64 decode rows + the first 8128 rows of a 20000-token prompt)."""

    HQ, HKV, D = 32, 8, 128

    def __init__(self, dev, mode):
        import torch
        import chunked_prefill_causal_cp_gb300 as cp
        import synth_inputs as SI

        self.cp, self.torch, self.mode = cp, torch, mode
        mb = SI.mixed_batch()
        self.mb = mb
        bf = torch.bfloat16
        self.desc = cp.layer_desc(bf, 0, self.HQ, self.HKV, self.D, cp.CP_CACHE_PAGED, page_size=mb.page_size,
                                  num_pages=mb.num_pages, max_blocks=mb.max_blocks)
        g = torch.Generator(device=dev).manual_seed(mb.seed)
        self.kp = torch.randn(mb.num_pages, self.HKV, mb.page_size, self.D, generator=g, device=dev).to(bf)
        self.vp = torch.randn(mb.num_pages, self.HKV, mb.page_size, self.D, generator=g, device=dev).to(bf)
        nd = len(mb.decode_ctx)
        rows = [1] * nd
        if mode == "mixed":
            entries = [e for e in cp.cp_schedule(8192, nd, mb.prompt_lens) if e[0] == 0]
            rows = [e[3] for e in entries]
            seqs = [e[1] for e in entries]
        else:
            seqs = list(range(nd))
        past = [c - 1 for c in mb.decode_ctx] + [0] * (len(seqs) - nd)
        self.rows, self.seqs, self.past_host = rows, seqs, past
        self.T = sum(rows)
        self.S = len(seqs)
        self.max_ctx = max(p + r for p, r in zip(past, rows))
        self.q = torch.randn(self.T, self.HQ, self.D, generator=g, device=dev).to(bf)
        self.kn = torch.randn(self.T, self.HKV, self.D, generator=g, device=dev).to(bf)
        self.vn = torch.randn(self.T, self.HKV, self.D, generator=g, device=dev).to(bf)
        self.out = torch.empty(self.T, self.HQ, self.D, dtype=bf, device=dev)
        self.bt = mb.block_table[seqs].contiguous().to(dev)
        cu = [0]
        for r in rows:
            cu.append(cu[-1] + r)
        self.cu = torch.tensor(cu, dtype=torch.int32, device=dev)
        self.past0 = torch.tensor(past, dtype=torch.int32, device=dev)
        self.past = self.past0.clone()
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.ws = torch.zeros(cp.cp_workspace_size(self.desc, self.T, self.max_ctx, self.S), dtype=torch.uint8,
                              device=dev)
        # algorithmic work
        kv_row = self.HKV * self.D * 2
        self.decode_bytes = sum((p + 1) * kv_row * 2 for p, r in zip(past, rows) if r == 1) \
            + sum(self.HQ * self.D * 2 * 2 + kv_row * 2 for r in rows if r == 1)
        self.flops = sum(4 * self.D * self.HQ * visible_pairs(p, r) for p, r in zip(past, rows))
        self.launches = 5 if mode == "mixed" else 4  # append, decode split, combine, [prefill], commit

    def step(self):
        self.past.copy_(self.past0)
        self.cp.cp_mixed_step(self.desc, self.q, self.kn, self.vn, self.kp, self.vp, self.bt, self.cu, self.past,
                              self.S, self.T, self.max_ctx, self.out, self.ws, dev_status=self.status)


def rolling_visible_pairs(L, c, C, left_pad):
    """Visible (query, key) pairs of the rolling workload, real query rows only:
    chunk k row i is position p = k*c + i; logical slot j holds position
    a = (k+1)*c - C + j, visible iff a >= 0, a >= left_pad and a <= p."""
    total = 0
    for k in range(L // c):
        lo = max(0, (k + 1) * c - C, left_pad)
        for i in range(c):
            p = k * c + i
            if p >= left_pad:
                total += max(0, p - lo + 1)
    return total


class ChunkLoop:
    """Chunk-by-chunk prefill of one prompt through the public calls, for the
    rolling-cache workload (fp16 MHA 16 x 128, window 1024, chunk 256, aligned
    lengths 2048 and 768 with 48 and 68 left-pad rows) and the fp32 example
    (1000 tokens, 8 heads x 64, chunk 256)."""

    def __init__(self, dev, mode):
        import torch
        import chunked_prefill_causal_cp_gb300 as cp
        import synth_inputs as SI

        self.cp, self.torch, self.mode = cp, torch, mode
        self.runs = []
        if mode == "rolling":
            H, d, c, C = 16, 128, 256, 1024
            for n_real in (2000, 700):
                L = cp.cp_aligned_length(n_real, c)
                q, k, v = SI.rolling_prompt(L, seed=3, heads=H, dim=d)
                self.runs.append(dict(kind=cp.CP_CACHE_ROLLING, H=H, Hkv=H, d=d, W=c, cap=C, L=L, lp=L - n_real,
                                      q=q, k=k, v=v, dtype=torch.float16,
                                      pairs=rolling_visible_pairs(L, c, C, L - n_real)))
        else:
            q, k, v = SI.fp32_sdpa_example()
            N, W = q.shape[0], 256
            self.runs.append(dict(kind=cp.CP_CACHE_CONTIG, H=q.shape[1], Hkv=k.shape[1], d=q.shape[2], W=W,
                                  cap=N, L=N, lp=0, q=q, k=k, v=v, dtype=torch.float32,
                                  pairs=visible_pairs(0, N)))
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        for r in self.runs:
            r["desc"] = cp.layer_desc(r["dtype"], 1, r["H"], r["Hkv"], r["d"], r["kind"], capacity=r["cap"])
            r["qd"], r["kd"], r["vd"] = (t.to(dev, r["dtype"]) for t in (r["q"], r["k"], r["v"]))
            r["kc"] = torch.zeros(1, r["Hkv"], r["cap"], r["d"], dtype=r["dtype"], device=dev)
            r["vc"] = torch.zeros_like(r["kc"])
            r["lens"] = torch.zeros(1, dtype=torch.int32, device=dev)
            r["left"] = torch.tensor([r["lp"]], dtype=torch.int32, device=dev)
            r["out"] = torch.empty(r["L"], r["H"], r["d"], dtype=r["dtype"], device=dev)
            r["sizes"] = cp.cp_chunk_plan(r["L"], r["W"])
            r["ws"] = torch.zeros(cp.cp_workspace_size(r["desc"], r["W"], r["cap"], 1), dtype=torch.uint8,
                                  device=dev)
        self.tokens = sum(r["L"] - r["lp"] for r in self.runs)
        self.flops = sum(4 * r["d"] * r["H"] * r["pairs"] for r in self.runs)
        # one cp_prefill_chunk call per chunk: the append and the attention (the tensor-core kernel
        # advances seqlens_k itself; the fp32 path takes a separate advance)
        self.launches = sum((2 if r["dtype"] != torch.float32 else 3) * len(r["sizes"]) for r in self.runs)

    def step(self):
        cp = self.cp
        for r in self.runs:
            r["lens"].zero_()
            rolling = r["kind"] == cp.CP_CACHE_ROLLING
            past = 0
            for w in r["sizes"]:
                sl = slice(past, past + w)
                cp.cp_prefill_chunk(r["desc"], r["qd"][None, sl], r["kd"][None, sl], r["vd"][None, sl], r["kc"],
                                    r["vc"], r["lens"], w, w, past, r["out"][None, sl], r["ws"],
                                    left_pad=r["left"] if rolling else None, dev_status=self.status)
                past += w

    def config(self):
        if self.mode == "rolling":
            return {"workload": "rolling_fp16_mha16_d128_window1024_chunk256_len2048+768",
                    "aligned_lengths": [r["L"] for r in self.runs], "left_pad": [r["lp"] for r in self.runs],
                    "visible_pairs": [r["pairs"] for r in self.runs],
                    "l2": "flushed between timed steps (512 MiB write)", "cuda_graph": True}
        return {"workload": "fp32_mha8_d64_prompt1000_chunk256", "visible_pairs": self.runs[0]["pairs"],
                "l2": "flushed between timed steps (512 MiB write)", "cuda_graph": True}


def run_chunk_loop(args, rank, world, dev, pk, pk_src):
    import torch
    wl = ChunkLoop(dev, args.workload)
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(2):
            wl.step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        wl.step()
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    for _ in range(max(args.warmup, 3)):
        g.replay()
    torch.cuda.synchronize()
    clocks = ClockSampler()
    clocks.start()
    times = time_steps(g.replay, flush, args.steps, torch)
    clk = clocks.stop()
    total_ms, value = job_throughput(sum(times), wl.tokens, args.steps, world)
    ms = total_ms / args.steps
    if int(wl.status.item()) != 0:
        raise RuntimeError(f"device status {int(wl.status.item())}")
    tflops = wl.flops / (ms / 1e3) / 1e12
    fp32 = args.workload == "fp32"
    line = {"metric": f"{args.workload} chunked-prefill tokens/s (real rows)", "value": value, "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32" if fp32 else "f16",
            "data": "synthetic", "config": wl.config(), "flops_per_step": wl.flops, "tflops_whole_step": tflops,
            "tensor_frac_whole_step": None if fp32 else tflops / float(pk["bf16_tflops"]),
            "gpu_launches": wl.launches * args.steps, "clocks": clk, "peaks": pk_src}
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_paged(args, rank, world, dev, pk, pk_src):
    import torch
    wl = PagedStep(dev, args.workload)
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(2):
            wl.step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        wl.step()
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    for _ in range(max(args.warmup, 3)):
        g.replay()
    torch.cuda.synchronize()
    clocks = ClockSampler()
    clocks.start()
    times = time_steps(g.replay, flush, args.steps, torch)
    clk = clocks.stop()
    total_ms = max_over_ranks(sum(times), world)
    ms = total_ms / args.steps
    if int(wl.status.item()) != 0:
        raise RuntimeError(f"device status {int(wl.status.item())}")
    hbm = float(pk["hbm_gbs"])
    tc = float(pk["bf16_tflops"])
    line = {"metric": f"{args.workload} step rows/s (paged KV, 16-token pages)",
            "value": world * wl.T * args.steps / (total_ms / 1e3), "unit": "rows/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"paged_{args.workload}_gqa32x8_d128_bf16", "decode_rows": sum(
                1 for r in wl.rows if r == 1), "prefill_rows": sum(r for r in wl.rows if r > 1),
                "decode_ctx_mean": sum(wl.mb.decode_ctx) / len(wl.mb.decode_ctx), "page_size": wl.mb.page_size,
                "l2": "flushed between timed steps (512 MiB write)", "cuda_graph": True},
            "decode_bytes_per_step": wl.decode_bytes, "flops_per_step": wl.flops,
            "roofline": ({"bound": "hbm", "achieved": wl.decode_bytes / (ms / 1e3) / 1e9, "peak": hbm,
                          "unit": "GB/s", "frac": wl.decode_bytes / (ms / 1e3) / 1e9 / hbm,
                          "traffic": kernel_traffic("decode.cu", "decode_split_paged.md"),
                          "kernel": "decode_split_kernel",
                          "scope": "K/V bytes of the decode rows over the whole step (append, split-KV "
                                   "kernel, combine, commit): a lower bound on the kernel's own rate",
                          "peak_source": "measured hbm_gbs (copy)"}
                         if args.workload == "decode" else None),
            "decode_gbs_whole_step": wl.decode_bytes / (ms / 1e3) / 1e9,
            "hbm_frac_whole_step": wl.decode_bytes / (ms / 1e3) / 1e9 / hbm,
            "tflops_whole_step": wl.flops / (ms / 1e3) / 1e12,
            "roofline_time_us": max(wl.flops / (tc * 1e12), wl.decode_bytes / (hbm * 1e9)) * 1e6,
            "gpu_launches": wl.launches * args.steps, "clocks": clk, "peaks": pk_src}
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_reference(args):
    """The CPU oracle as the reference arm (rank 0 only)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import numpy as np
    import oracle
    import synth_inputs as SI
    wl = GqaPrefill.__new__(GqaPrefill)
    q, k, v = SI.gqa_prompt(GqaPrefill.N, seed=1)
    qn, kn, vn = (t.double().numpy() for t in (q, k, v))
    G = GqaPrefill.HQ // GqaPrefill.HKV
    sizes = oracle.chunk_plan(GqaPrefill.N, GqaPrefill.W)

    def one_group(g):
        oracle.chunked_prefill(qn[:, g * G:(g + 1) * G], kn[:, g:g + 1], vn[:, g:g + 1], GqaPrefill.W)

    for i in range(args.warmup):
        one_group(i % GqaPrefill.HKV)
    times = []
    t_budget = 150.0
    t_start = time.perf_counter()
    for i in range(args.steps):
        t0 = time.perf_counter()
        one_group(i % GqaPrefill.HKV)
        times.append(time.perf_counter() - t0)
        if time.perf_counter() - t_start > t_budget:
            break
    per_group = sum(times) / len(times)
    value = GqaPrefill.N / (per_group * GqaPrefill.HKV)
    sample = (f"each step: oracle.chunked_prefill of the 4000-token prompt (chunks {sizes}) for one KV-head "
              f"group ({G} of {GqaPrefill.HQ} query heads); tokens/s scaled to all {GqaPrefill.HKV} groups; "
              f"{len(times)} of {args.steps} requested steps timed within a {t_budget:.0f} s budget")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": len(times), "steps_requested": args.steps, "warmup": args.warmup,
            "ms_per_step": per_group * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic (seeded N(0,1) q/k/v)",
            "config": {"workload": "gqa32x8_d128_bf16_prompt4000_chunk512_cap8192", "prompt_tokens": 4000,
                       "chunk": 512, "kv_capacity": 8192, "heads_q": 32, "heads_kv": 8, "head_dim": 128},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_native(args)


if __name__ == "__main__":
    main()
