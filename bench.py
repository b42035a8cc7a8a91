#!/usr/bin/env python
"""Benchmark of the chunked-prefill causal attention hot path on one GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                    [--workload gqa_prefill|fp32|ladder|rolling|decode|mixed|verify|varlen|deep|append|append_paged]
                    [--chunk W] [--prompt N] [--budget B] [--overlap] [--no-pad] [--no-extras] [--sweep]

Default workload (the one the headline metric is quoted on): one GQA layer,
32 query / 8 KV heads, head_dim 128, bf16, a 4000-token prompt prefilled in
chunks of 512 (7 x 512 + 416) into a KV cache of physical capacity 8192.  One
step is the whole path for one prompt: chunk plan, query-width ladder (the
416-row tail is widened to 512 by repeating its last row, one cp_pad_chunk
launch), and per chunk one cp_prefill_chunk call, which is one kernel launch
on a contiguous cache: the chunk's K/V append, the chunk attention and the
advance of seqlens_k to past + real rows.  Each step is one replay of a CUDA
graph captured from the library's public calls; L2 is flushed (512 MiB write)
between timed steps.

Before anything is timed, each workload checks one replay of its own graph
(cache bytes, lengths, and sampled output rows against a float32 PyTorch
evaluation of the attention definition); a failed check ends the run without
a line.

The default line also carries, under "configs", one measurement of each of
the other workloads (fp32 example, padding ladder, rolling cache, decode
rows, k-row verify chunks at long lengths, ragged prompts in one call, one
8128-row chunk at 8128 cached positions (the attention kernel's steady state),
the KV append alone on a contiguous and a paged cache, and the whole mixed
token-budget schedule at budgets 8192 and 2048, serial and with the decode
rows on a side stream), each with its own check, and under "cpu_baseline" the
C++ oracle on bounded samples of the default and the other workloads.  ``--workload X`` prints X's
line alone; ``--chunk`` / ``--prompt`` / ``--budget`` set the chunk width, the
prompt length and the token budget, and ``--sweep`` prints one line per chunk
width and per token budget.  ``--impl reference`` times the C++ CPU oracle (test infrastructure,
float64, std::thread) on a bounded sample of the default workload instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "chunked-prefill attn tokens/s & effective TFLOP/s; % of GB300 BF16/HBM roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
HBM_NOMINAL_GBS = 7900.0  # the part's nominal HBM3e rate, reported beside the measured copy rate
BF16_TOL = 2e-2   # max-abs error bound for 16-bit inputs with fp32 accumulation
FP32_TOL = 1e-4   # max-abs error bound for the fp32 path
L2_NOTE = "flushed between timed steps (512 MiB write)"


def parse_args(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=3000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", default="native", choices=["native", "reference"])
    p.add_argument("--workload", default="gqa_prefill",
                   choices=["gqa_prefill", "fp32", "ladder", "rolling", "decode", "mixed", "verify", "varlen", "deep",
                            "append", "append_paged"])
    p.add_argument("--sweep", action="store_true",
                   help="one line per chunk width W (gqa_prefill) and per token budget (mixed schedule)")
    p.add_argument("--chunk", type=int, default=512, help="chunk width W of the gqa_prefill workload")
    p.add_argument("--prompt", type=int, default=4000, help="prompt tokens of the gqa_prefill workload")
    p.add_argument("--budget", type=int, default=8192, help="token budget of the mixed workload")
    p.add_argument("--no-pad", action="store_true", help="do not widen chunks to the query-width ladder")
    p.add_argument("--overlap", action="store_true",
                   help="mixed / varlen workloads: cp_mixed_step_overlap / cp_prefill_varlen_overlap "
                        "(split-KV kernels on a side stream)")
    p.add_argument("--no-extras", action="store_true", help="default line without the other workloads")
    p.add_argument("--cpu-seconds", type=float, default=12.0, help="CPU-baseline sample budget")
    p.add_argument("--skip-cpu", action="store_true")
    return p.parse_args(argv)


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
    """nvidia-smi sampling of SM clock and throttle reasons while the GPU is loaded."""

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

def kernel_traffic(profile_name):
    """DRAM bytes per launch recorded in profiles/<profile_name> (a JSON record
    written from an ncu capture), or None when the kernel source it names has
    changed since the capture."""
    import hashlib
    prof = os.path.join(ROOT, "profiles", profile_name)
    if not os.path.exists(prof):
        return None
    with open(prof) as f:
        rec = json.load(f)
    src = os.path.join(ROOT, "chunked_prefill_causal_cp_gb300", "csrc", rec.get("kernel_source", ""))
    if not os.path.isfile(src):
        return None
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()
    if sha != rec.get("source_sha256"):
        return None
    return float(rec["dram_bytes_per_launch"])


def mixed_rooflines(steps, tc, hbm):
    """Two roofline times of a mixed schedule, in ms: T* = sum over steps of
    max(FLOPs / tensor peak, decode bytes / copy rate), which assumes the decode
    rows' bytes stream entirely beside the tensor-core work, and the serial
    time = sum of the two, which holds when an SM's shared-memory intake is
    about its share of the HBM rate (so an SM cannot do both at once)."""
    t_star = sum(max(st["flops"] / (tc * 1e12), st["bytes"] / (hbm * 1e9)) for st in steps) * 1e3
    t_serial = sum(st["flops"] / (tc * 1e12) + st["bytes"] / (hbm * 1e9) for st in steps) * 1e3
    return t_star, t_serial


def fp32_alu_peak_tflops(dev):
    """FP32 FMA peak of the SIMT path: SMs x 128 FMA lanes x 2 FLOP x the part's
    maximum SM clock (2070 MHz)."""
    import torch
    return torch.cuda.get_device_properties(dev).multi_processor_count * 128 * 2 * 2.07e9 / 1e12


def cpu_cores():
    return os.cpu_count() or 1


def visible_pairs(past, rows):
    """Visible (query, key) pairs of `rows` causal rows after `past` cached keys."""
    return rows * past + rows * (rows + 1) // 2


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


def ref_rows(q_tok, keys, vals, scale):
    """float32 PyTorch evaluation of the attention definition for one token:
    q_tok [Hq, D] over visible keys / values [n, Hkv, D]; query head h reads
    KV head h // (Hq / Hkv).  Returns [Hq, D] (float32)."""
    import torch
    hq, d = q_tok.shape
    hkv = keys.shape[1]
    qf = q_tok.float().view(hkv, hq // hkv, d)
    s = torch.einsum("gjd,ngd->gjn", qf, keys.float()) * scale
    p = torch.softmax(s, dim=-1)
    return torch.einsum("gjn,ngd->gjd", p, vals.float()).reshape(hq, d)


def bits_equal(a, b):
    """Byte equality of two tensors of the same shape and dtype."""
    import torch
    if a.shape != b.shape or a.dtype != b.dtype:
        return False
    if a.element_size() == 2:
        return torch.equal(a.contiguous().view(torch.int16), b.contiguous().view(torch.int16))
    return torch.equal(a.contiguous().view(torch.int32), b.contiguous().view(torch.int32))


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


def capture(step, dev):
    """Two eager runs on a side stream, then one CUDA graph of `step`."""
    import torch
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(2):
            step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    return g


class CheckFailed(RuntimeError):
    pass


def require(check, what):
    """Ends the run (no line is printed) when a pre-timing check failed."""
    if not check.get("ok"):
        raise CheckFailed(f"{what}: check before timing failed: {json.dumps(check)}")
    return check


# --------------------------------------------------------------------------- workloads

class GqaPrefill:
    """The GQA prompt (default 4000 tokens, chunk 512, capacity 8192; see module doc)."""

    HQ, HKV, D, CAP = 32, 8, 128, 8192

    def __init__(self, dev, pad=True, N=4000, W=512):
        import torch
        import chunked_prefill_causal_cp_gb300 as cp
        import synth_inputs as SI

        self.cp, self.torch, self.dev, self.pad = cp, torch, dev, pad
        self.N, self.W = N, W
        self.sizes = cp.cp_chunk_plan(self.N, self.W)
        self.widths = [cp.cp_query_width(r, self.W) if pad else r for r in self.sizes]
        self.rows_alloc = sum(self.sizes[:-1]) + self.widths[-1]
        if self.rows_alloc > self.CAP:
            raise ValueError(f"prompt {N} with chunk {W} needs {self.rows_alloc} slots > capacity {self.CAP}")
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
        # launches of this library per step: one pad launch (q, k and v together) per widened
        # chunk, then one launch per chunk (append, attention and the advance of seqlens_k)
        self.launches = sum(1 for r, w in zip(self.sizes, self.widths) if w > r) + len(self.sizes)

    def _chunk(self, i, attn=True, append=True, commit=True, pad=True):
        cp = self.cp
        r, w = self.sizes[i], self.widths[i]
        past = sum(self.sizes[:i])
        sl = slice(past, past + w)
        q, k, v = self.q[None, sl], self.k[None, sl], self.v[None, sl]
        if append and pad and w > r:
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
        self.graph = capture(self.step, self.dev)
        return self.graph

    def capture_prefixes(self):
        """Graphs of the first k chunk calls (k = 0 .. n) without the pad launch
        (the widened rows are already in place after one step): graph k runs
        chunks 0 .. k-1 in the same launch chain as the step, so the attention
        launches' in-situ time is T(n) - T(0) and chunk k's is T(k+1) - T(k)."""
        torch = self.torch
        self.prefix_graphs = []
        for k in range(len(self.sizes) + 1):
            def body(k=k):
                self.lens.zero_()
                for i in range(k):
                    self._chunk(i, pad=False)
            self.prefix_graphs.append(capture(body, self.dev))
        torch.cuda.synchronize()

    def self_check(self, n_sample=26, seed=7):
        """One replayed step against what it must hold: the cache holds the
        prompt's K/V rows bit for bit and, in the slots of the widened tail,
        copies of the last real row; seqlens_k = N; the device status is clear;
        each chunk's first and last rows and random rows agree with ref_rows."""
        torch = self.torch
        torch.cuda.synchronize()
        N = self.N
        kc = self.kc[0].transpose(0, 1)
        vc = self.vc[0].transpose(0, 1)
        cache_ok = bits_equal(kc[:N], self.k[:N]) and bits_equal(vc[:N], self.v[:N])
        pad = self.widths[-1] - self.sizes[-1]
        if pad:
            cache_ok = cache_ok and bits_equal(kc[N:N + pad], self.k[N - 1:N].expand(pad, -1, -1)) \
                and bits_equal(vc[N:N + pad], self.v[N - 1:N].expand(pad, -1, -1))
        toks = set()
        past = 0
        for r in self.sizes:
            toks.update((past, past + r - 1))
            past += r
        g = torch.Generator().manual_seed(seed)
        while len(toks) < n_sample:
            toks.add(int(torch.randint(0, N, (1,), generator=g)))
        scale = self.D ** -0.5
        err = 0.0
        for t in sorted(toks):
            ref = ref_rows(self.q[t], self.k[:t + 1], self.v[:t + 1], scale)
            err = max(err, float((self.out[t].float() - ref).abs().max()))
        lens = int(self.lens.item())
        status = int(self.status.item())
        ok = cache_ok and lens == N and status == 0 and err < BF16_TOL
        return {"ok": ok, "rows_checked": len(toks), "max_abs_err": err, "tol": BF16_TOL,
                "cache_bit_exact": cache_ok, "seqlens_k": lens, "status": status,
                "reference": "float32 PyTorch evaluation of the definition on the GPU"}

    def config(self):
        return {"workload": f"gqa32x8_d128_bf16_prompt{self.N}_chunk{self.W}_cap{self.CAP}",
                "prompt_tokens": self.N, "chunk": self.W, "chunks": self.sizes,
                "query_widths": self.widths, "kv_capacity": self.CAP, "heads_q": self.HQ,
                "heads_kv": self.HKV, "head_dim": self.D, "global_batch": 1, "seq_len": self.N,
                "padding": "ladder" if self.pad else "none", "parallelism": "replica per GPU",
                "l2": L2_NOTE, "cuda_graph": True}

    # ---- end to end: host buffers in, result out, through the captured public calls
    def pin(self):
        """Pinned host staging in the layout a serving loop would fill: each
        chunk's q, k and v rows back to back, so one copy per chunk moves all
        three (each extra copy costs about 2 us of the host link on this part).
        The device side mirrors it: per chunk one buffer [q | k | v] whose three
        parts are the call's q, k_new and v_new."""
        torch = self.torch
        row = (self.HQ + 2 * self.HKV) * self.D  # elements per token in a packed chunk
        self.e2e_chunks = []
        past = 0
        for r, w in zip(self.sizes, self.widths):
            hbuf = torch.empty(w * row, dtype=torch.bfloat16).pin_memory()
            nq, nk = r * self.HQ * self.D, r * self.HKV * self.D
            dbuf = torch.zeros(w * row, dtype=torch.bfloat16, device=self.dev)
            qsz, ksz = w * self.HQ * self.D, w * self.HKV * self.D
            hq = hbuf[:qsz]
            hk = hbuf[qsz:qsz + ksz]
            hv = hbuf[qsz + ksz:]
            hq[:nq].copy_(self.host_q[past:past + r].reshape(-1))
            hk[:nk].copy_(self.host_k[past:past + r].reshape(-1))
            hv[:nk].copy_(self.host_v[past:past + r].reshape(-1))
            self.e2e_chunks.append(dict(
                h=hbuf, d=dbuf, bytes_in=(nq + 2 * nk) * 2, r=r, w=w, past=past,
                q=dbuf[:qsz].view(1, w, self.HQ, self.D), k=dbuf[qsz:qsz + ksz].view(1, w, self.HKV, self.D),
                v=dbuf[qsz + ksz:].view(1, w, self.HKV, self.D),
                h_in=(hq[:nq], hk[:nk], hv[:nk])))
            past += r
        self.ho = torch.empty(self.N, self.HQ, self.D, dtype=torch.bfloat16).pin_memory()
        self.h2d = sum(c["bytes_in"] for c in self.e2e_chunks)
        self.d2h = self.ho.numel() * 2

    def capture_e2e(self):
        """One CUDA graph of a whole step with its host traffic, pipelined the way
        a serving loop runs chunked prefill: each chunk's packed q/k/v rows go
        host -> device in one copy on a copy stream, all queued at once in chunk
        order; each chunk's call waits for its own rows; its output rows go
        device -> host on a second copy stream as soon as the chunk is done.
        Every input byte and every output byte of the step crosses the bus inside
        the graph; the step ends when the last output row is on the host."""
        torch = self.torch
        cp = self.cp
        main = torch.cuda.Stream(self.dev)
        up, down = torch.cuda.Stream(self.dev), torch.cuda.Stream(self.dev)
        n = len(self.sizes)
        ev_in = [torch.cuda.Event() for _ in range(n)]
        ev_done = [torch.cuda.Event() for _ in range(n)]

        def body():
            self.lens.zero_()
            up.wait_stream(main)
            down.wait_stream(main)
            with torch.cuda.stream(up):
                for i, c in enumerate(self.e2e_chunks):
                    if c["w"] == c["r"]:
                        c["d"].copy_(c["h"], non_blocking=True)
                    else:  # a short chunk: only its real rows cross the link
                        qsz, ksz = c["w"] * self.HQ * self.D, c["w"] * self.HKV * self.D
                        hq, hk, hv = c["h_in"]
                        c["d"][:hq.numel()].copy_(hq, non_blocking=True)
                        c["d"][qsz:qsz + hk.numel()].copy_(hk, non_blocking=True)
                        c["d"][qsz + ksz:qsz + ksz + hv.numel()].copy_(hv, non_blocking=True)
                    ev_in[i].record(up)
            for i, c in enumerate(self.e2e_chunks):
                main.wait_event(ev_in[i])
                r, w, past = c["r"], c["w"], c["past"]
                if w > r:
                    cp.cp_pad_chunk(self.desc, c["q"], c["k"], c["v"], r, w)
                cp.cp_prefill_chunk(self.desc, c["q"], c["k"], c["v"], self.kc, self.vc, self.lens, w, r, past,
                                    self.out[None, past:past + w], self.ws, dev_status=self.status)
                ev_done[i].record(main)
                with torch.cuda.stream(down):
                    down.wait_event(ev_done[i])
                    self.ho[past:past + r].copy_(self.out[past:past + r], non_blocking=True)
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

    def cpu_sample(self, budget_s):
        """The C++ oracle (as it stands, std::thread on every host core) on
        whole KV-head groups of the same prompt until the time budget is spent.
        Returns (tokens/s scaled to all heads, sample, seconds, max-abs
        difference between the oracle's rows and this workload's last GPU
        output for the groups it ran, query heads compared, threads)."""
        import numpy as np
        from oracle import cpp as oracle
        oracle.set_threads(0)
        q = self.host_q.double().numpy()
        k = self.host_k.double().numpy()
        v = self.host_v.double().numpy()
        gpu = self.out[:self.N].float().cpu().double().numpy()
        G = self.HQ // self.HKV
        t0 = time.perf_counter()
        groups = 0
        diff = 0.0
        while groups < self.HKV:
            g = groups
            o, _, _ = oracle.chunked_prefill(q[:, g * G:(g + 1) * G], k[:, g:g + 1], v[:, g:g + 1], self.W)
            diff = max(diff, float(np.abs(o - gpu[:, g * G:(g + 1) * G]).max()))
            groups += 1
            if time.perf_counter() - t0 > budget_s:
                break
        t = time.perf_counter() - t0
        full = t * self.HKV / groups
        sample = (f"C++ oracle chunked_prefill of the {self.N}-token prompt (chunks {self.sizes[0]}x"
                  f"{len(self.sizes) - 1}+{self.sizes[-1]}, unpadded) for {groups} of {self.HKV} KV-head "
                  f"groups ({groups * G} of {self.HQ} query heads), {t:.1f} s, scaled to all heads")
        return self.N / full, sample, t, diff, groups * G, oracle.threads()


def oracle_single_thread_fp32():
    """The C++ oracle on one thread over the fp32 example (1000 tokens, 8 heads
    x 64, chunks of 256): tokens/s and seconds."""
    from oracle import cpp as oracle
    import synth_inputs as SI
    q, k, v = (t.double().numpy() for t in SI.fp32_sdpa_example())
    oracle.set_threads(1)
    try:
        t0 = time.perf_counter()
        oracle.chunked_prefill(q, k, v, 256)
        t = time.perf_counter() - t0
    finally:
        oracle.set_threads(0)
    return q.shape[0] / t, t


def oracle_config_samples(budget_s=3.0, ladder_groups=8):
    """The C++ oracle (as it stands, std::thread on every host core) on bounded
    samples of the other workloads, each scaled to its workload's unit; every
    entry says what ran and how it was scaled.  `ladder_groups` KV-head groups
    of the ladder prompts run (8: all of them)."""
    import numpy as np
    import torch
    from oracle import cpp as oracle
    import synth_inputs as SI

    oracle.set_threads(0)
    res = {}
    # the fp32 example, whole
    q, k, v = (t.double().numpy() for t in SI.fp32_sdpa_example())
    t0 = time.perf_counter()
    oracle.chunked_prefill(q, k, v, 256)
    t = time.perf_counter() - t0
    res["fp32_example"] = {"tokens_per_s": q.shape[0] / t, "seconds": t,
                           "sample": "the whole example: 1000 tokens, 8 heads x 64, chunks of 256"}
    # the ladder prompts, all heads, until twice the budget is spent (about 4 s for all six)
    toks, t_sum, done = 0, 0.0, 0
    for idx in range(len(SI.LADDER_PROMPT_LENGTHS)):
        q, k, v = (t.double().numpy() for t in SI.ladder_prompt(idx))
        t0 = time.perf_counter()
        oracle.chunked_prefill(q[:, :4 * ladder_groups], k[:, :ladder_groups], v[:, :ladder_groups], 512)
        t_sum += time.perf_counter() - t0
        toks += q.shape[0]
        done += 1
        if t_sum > 2 * budget_s:
            break
    heads = "all 32 query heads" if ladder_groups == 8 else f"{4 * ladder_groups} of 32 query heads, scaled to 32"
    res["padding_ladder"] = {"tokens_per_s": toks / (t_sum * 8 / ladder_groups), "seconds": t_sum,
                             "sample": f"{done} of the 6 prompts, {heads}, chunks of 512 (the real rows, "
                                       "which padding leaves unchanged)"}
    # the rolling runs, whole, the shorter first
    toks, t_sum, runs = 0, 0.0, []
    for L, n_real in ((768, 700), (2048, 2000)):
        q, k, v = (t.double().numpy() for t in SI.rolling_prompt(L))
        t0 = time.perf_counter()
        oracle.rolling_prefill(q, k, v, 256, 1024, L - n_real)
        t_sum += time.perf_counter() - t0
        toks += n_real
        runs.append(L)
        if t_sum > budget_s:
            break
    res["rolling"] = {"tokens_per_s": toks / t_sum, "seconds": t_sum,
                      "sample": f"the whole rolling run(s) of aligned length {runs}, 16 heads x 128, C = 1024, c = 256"}
    # the mixed schedule's step 1 at budget 8192 (64 decode rows, then the first 8128 rows of a prompt), sampled
    mb = SI.mixed_batch()
    ctx = mb.decode_ctx
    g = torch.Generator().manual_seed(29)
    t_dec, keys_dec = 0.0, 0
    for i in range(8):
        c = ctx[i]
        kk = torch.randn(c, 8, 128, generator=g, dtype=torch.float64).numpy()
        vv = torch.randn(c, 8, 128, generator=g, dtype=torch.float64).numpy()
        qq = torch.randn(32, 128, generator=g, dtype=torch.float64).numpy()
        t0 = time.perf_counter()
        oracle.attention_row(qq, kk, vv, c - 1)
        t_dec += time.perf_counter() - t0
        keys_dec += c
    dec_all = t_dec * sum(ctx) / keys_dec
    n_pre = 8128
    kk = torch.randn(n_pre, 8, 128, generator=g, dtype=torch.float64).numpy()
    vv = torch.randn(n_pre, 8, 128, generator=g, dtype=torch.float64).numpy()
    t_pre, pairs = 0.0, 0
    for p in np.linspace(0, n_pre - 1, 16).astype(int):
        qq = torch.randn(32, 128, generator=g, dtype=torch.float64).numpy()
        t0 = time.perf_counter()
        oracle.attention_row(qq, kk, vv, int(p))
        t_pre += time.perf_counter() - t0
        pairs += int(p) + 1
    pre_all = t_pre * (n_pre * (n_pre + 1) // 2) / pairs
    res["mixed_budget8192_step1"] = {
        "rows_per_s": (64 + n_pre) / (dec_all + pre_all), "seconds_estimated": dec_all + pre_all,
        "seconds_run": t_dec + t_pre,
        "sample": "8 of the 64 decode rows over their whole contexts, scaled by context length to all 64; "
                  "16 of the 8128 prompt rows at evenly spread positions, scaled by visible keys to the chunk"}
    res["threads"] = oracle.threads()
    return res


class ChunkLoop:
    """Chunk-by-chunk prefill of one prompt through the public calls, for the
    rolling-cache workload (fp16 MHA 16 x 128, window 1024, chunk 256, aligned
    lengths 2048 and 768 with 48 and 68 left-pad rows) and the fp32 example
    (1000 tokens, 8 heads x 64, chunk 256)."""

    def __init__(self, dev, mode):
        import torch
        import chunked_prefill_causal_cp_gb300 as cp
        import synth_inputs as SI

        self.cp, self.torch, self.mode, self.dev = cp, torch, mode, dev
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
        # one cp_prefill_chunk call per chunk, one launch each: the fp32 kernel on the contiguous
        # cache, the tensor-core kernel on the ring (256-row chunks on a 1024-slot ring), each
        # appending the chunk, attending and advancing seqlens_k
        self.launches = sum(len(r["sizes"]) for r in self.runs)

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

    def self_check(self, n_sample=24, seed=11):
        """fp32: every row against a float64 evaluation of causal attention on
        the GPU (1e-4).  Rolling: the ring holds position p in slot p mod C bit
        for bit for the last C positions; sampled real rows agree with ref_rows
        over the window the chunk sees, positions [max(0, (k+1)c - C, left_pad), p]."""
        torch = self.torch
        torch.cuda.synchronize()
        status = int(self.status.item())
        if self.mode == "fp32":
            r = self.runs[0]
            q, k, v = (t.double() for t in (r["qd"], r["kd"], r["vd"]))
            s = torch.einsum("thd,shd->hts", q, k) * r["d"] ** -0.5
            n = q.shape[0]
            s.masked_fill_(torch.ones(n, n, dtype=torch.bool, device=s.device).triu(1), float("-inf"))
            ref = torch.einsum("hts,shd->thd", torch.softmax(s, dim=-1), v)
            err = float((r["out"].double() - ref).abs().max())
            lens = int(r["lens"].item())
            ok = err < FP32_TOL and lens == n and status == 0
            return {"ok": ok, "rows_checked": n, "max_abs_err": err, "tol": FP32_TOL, "seqlens_k": lens,
                    "status": status, "reference": "float64 PyTorch causal attention on the GPU, every row"}
        err, rows, ring_ok, lens_ok = 0.0, 0, True, True
        g = torch.Generator().manual_seed(seed)
        for r in self.runs:
            L, lp, c, C = r["L"], r["lp"], r["W"], r["cap"]
            lens_ok = lens_ok and int(r["lens"].item()) == L
            for p in range(max(0, L - C), L):
                ring_ok = ring_ok and bits_equal(r["kc"][0, :, p % C], r["kd"][p]) \
                    and bits_equal(r["vc"][0, :, p % C], r["vd"][p])
                if not ring_ok:
                    break
            picks = {lp, L - 1}
            while len(picks) < n_sample // len(self.runs):
                picks.add(int(torch.randint(lp, L, (1,), generator=g)))
            for p in sorted(picks):
                k_ = p // c
                lo = max(0, (k_ + 1) * c - C, lp)
                ref = ref_rows(r["qd"][p], r["kd"][lo:p + 1], r["vd"][lo:p + 1], r["d"] ** -0.5)
                err = max(err, float((r["out"][p].float() - ref).abs().max()))
                rows += 1
        ok = ring_ok and lens_ok and status == 0 and err < BF16_TOL
        return {"ok": ok, "rows_checked": rows, "max_abs_err": err, "tol": BF16_TOL, "ring_bit_exact": ring_ok,
                "seqlens_k_ok": lens_ok, "status": status,
                "reference": "float32 PyTorch evaluation of the windowed definition on the GPU"}

    def config(self):
        if self.mode == "rolling":
            return {"workload": "rolling_fp16_mha16_d128_window1024_chunk256_len2048+768",
                    "aligned_lengths": [r["L"] for r in self.runs], "left_pad": [r["lp"] for r in self.runs],
                    "visible_pairs": [r["pairs"] for r in self.runs], "l2": L2_NOTE, "cuda_graph": True}
        return {"workload": "fp32_mha8_d64_prompt1000_chunk256", "visible_pairs": self.runs[0]["pairs"],
                "l2": L2_NOTE, "cuda_graph": True}


class LadderRuns:
    """The query-padding workload: the GQA layer with chunk 512 and prompts
    {1041, 1468, 3118, 3788, 1137, 1200} (seeds 10 + idx), each prefilled
    twice; the last chunk of each is widened to its ladder tier {171, 342, 512}
    by repeating its last real row.  Contiguous cache of capacity 4096."""

    HQ, HKV, D, W, CAP = 32, 8, 128, 512, 4096

    def __init__(self, dev, pad=True):
        import torch
        import chunked_prefill_causal_cp_gb300 as cp
        import synth_inputs as SI

        self.cp, self.torch, self.dev, self.pad = cp, torch, dev, pad
        bf = torch.bfloat16
        self.desc = cp.layer_desc(bf, 1, self.HQ, self.HKV, self.D, cp.CP_CACHE_CONTIG, capacity=self.CAP)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.ws = torch.zeros(cp.cp_workspace_size(self.desc, self.W, self.CAP, 1), dtype=torch.uint8, device=dev)
        self.runs = []
        for idx, n in enumerate(SI.LADDER_PROMPT_LENGTHS):
            q, k, v = SI.ladder_prompt(idx)
            sizes = cp.cp_chunk_plan(n, self.W)
            widths = [cp.cp_query_width(r, self.W) if pad else r for r in sizes]
            alloc = sum(sizes[:-1]) + widths[-1]
            r = dict(n=n, sizes=sizes, widths=widths)
            for name, t, h in (("q", q, self.HQ), ("k", k, self.HKV), ("v", v, self.HKV)):
                buf = torch.zeros(alloc, h, self.D, dtype=bf, device=dev)
                buf[:n].copy_(t)
                r[name] = buf
            r["out"] = torch.zeros(alloc, self.HQ, self.D, dtype=bf, device=dev)
            r["kc"] = torch.zeros(1, self.HKV, self.CAP, self.D, dtype=bf, device=dev)
            r["vc"] = torch.zeros_like(r["kc"])
            r["lens"] = torch.zeros(1, dtype=torch.int32, device=dev)
            self.runs.append(r)
        self.tokens = 2 * sum(r["n"] for r in self.runs)
        self.flops = 2 * sum(4 * self.D * self.HQ * visible_pairs(0, r["n"]) for r in self.runs)
        self.padded_rows = 2 * sum(r["widths"][-1] - r["sizes"][-1] for r in self.runs)
        self.launches = 2 * sum(len(r["sizes"]) + (r["widths"][-1] > r["sizes"][-1]) for r in self.runs)

    def run_once(self, r):
        cp = self.cp
        r["lens"].zero_()
        past = 0
        for rr, w in zip(r["sizes"], r["widths"]):
            sl = slice(past, past + w)
            q, k, v = r["q"][None, sl], r["k"][None, sl], r["v"][None, sl]
            if w > rr:
                cp.cp_pad_chunk(self.desc, q, k, v, rr, w)
            cp.cp_prefill_chunk(self.desc, q, k, v, r["kc"], r["vc"], r["lens"], w, rr, past, r["out"][None, sl],
                                self.ws, dev_status=self.status)
            past += rr

    def step(self):
        for _ in range(2):
            for r in self.runs:
                self.run_once(r)

    def self_check(self, unpadded=None, n_sample=4, seed=13):
        """Real rows bit-identical to an unpadded run of the same prompts; the
        cache holds the prompt rows bit for bit and, after them, the pad rows
        (copies of the last real row); seqlens_k = the real length; sampled rows
        agree with ref_rows."""
        torch = self.torch
        torch.cuda.synchronize()
        same, cache_ok, lens_ok, err, rows = True, True, True, 0.0, 0
        g = torch.Generator().manual_seed(seed)
        for i, r in enumerate(self.runs):
            n = r["n"]
            if unpadded is not None:
                same = same and bits_equal(r["out"][:n], unpadded.runs[i]["out"][:n])
            kc = r["kc"][0].transpose(0, 1)
            cache_ok = cache_ok and bits_equal(kc[:n], r["k"][:n])
            pad = r["widths"][-1] - r["sizes"][-1]
            if pad:
                cache_ok = cache_ok and bits_equal(kc[n:n + pad], r["k"][n - 1:n].expand(pad, -1, -1))
            lens_ok = lens_ok and int(r["lens"].item()) == n
            picks = {n - 1}
            while len(picks) < n_sample:
                picks.add(int(torch.randint(0, n, (1,), generator=g)))
            for t in sorted(picks):
                ref = ref_rows(r["q"][t], r["k"][:t + 1], r["v"][:t + 1], self.D ** -0.5)
                err = max(err, float((r["out"][t].float() - ref).abs().max()))
                rows += 1
        status = int(self.status.item())
        ok = same and cache_ok and lens_ok and status == 0 and err < BF16_TOL
        return {"ok": ok, "real_rows_bit_identical_to_unpadded": same, "cache_bit_exact": cache_ok,
                "seqlens_k_ok": lens_ok, "rows_checked": rows, "max_abs_err": err, "tol": BF16_TOL,
                "status": status}

    def config(self):
        return {"workload": "ladder_gqa32x8_d128_bf16_chunk512_prompts1041-3788_x2",
                "prompts": [r["n"] for r in self.runs], "last_widths": [r["widths"][-1] for r in self.runs],
                "padded_rows_per_step": self.padded_rows, "l2": L2_NOTE, "cuda_graph": True}


class MixedSchedule:
    """The token-budget workload over a paged cache: 64 running decodes with
    contexts U{512..8192} and 4 waiting prompts of 20000 tokens, 16-token pages
    (seeded page permutation), GQA 32/8 x 128 bf16.  One step of this workload
    is the whole schedule cp_schedule gives for `budget` (10 mixed steps at
    8192, 41 at 2048), each one cp_mixed_step call; ``decode_only`` is instead
    the 64 decode rows alone, one call.  ``overlap``: each step is one
    cp_mixed_step_overlap call instead (split-KV kernels on a side stream
    beside the tensor-core kernel)."""

    HQ, HKV, D = 32, 8, 128

    def __init__(self, dev, budget=8192, decode_only=False, overlap=False):
        import torch
        import chunked_prefill_causal_cp_gb300 as cp
        import synth_inputs as SI

        self.cp, self.torch, self.dev = cp, torch, dev
        self.budget, self.decode_only, self.overlap = budget, decode_only, overlap
        self.handles = (torch.cuda.Stream(dev), torch.cuda.Event(), torch.cuda.Event()) if overlap else None
        mb = SI.mixed_batch()
        if not decode_only:
            # every sequence that decodes gains one position per step: give each one pages for that
            n_steps = 1 + max(e[0] for e in cp.cp_schedule(budget, len(mb.decode_ctx), mb.prompt_lens))
            if n_steps > 64:
                mb = SI.mixed_batch(decode_tail=n_steps)
        self.mb = mb
        bf = torch.bfloat16
        self.desc = cp.layer_desc(bf, 0, self.HQ, self.HKV, self.D, cp.CP_CACHE_PAGED, page_size=mb.page_size,
                                  num_pages=mb.num_pages, max_blocks=mb.max_blocks)
        g = torch.Generator(device=dev).manual_seed(mb.seed)
        self.kp = torch.randn(mb.num_pages, self.HKV, mb.page_size, self.D, generator=g, device=dev).to(bf)
        self.vp = torch.randn(mb.num_pages, self.HKV, mb.page_size, self.D, generator=g, device=dev).to(bf)
        nd = len(mb.decode_ctx)
        pos = [c - 1 for c in mb.decode_ctx] + [0] * len(mb.prompt_lens)
        if decode_only:
            plan = [[(s, -1, 1) for s in range(nd)]]
        else:
            steps = {}
            for st, seq, start, r in cp.cp_schedule(budget, nd, mb.prompt_lens):
                steps.setdefault(st, []).append((seq, start, r))
            plan = [steps[i] for i in sorted(steps)]
        self.steps = []
        row_seq, row_pos = [], []
        off = 0
        kv_row = self.HKV * self.D * 2
        self.flops, self.decode_bytes, self.decode_rows, self.prefill_rows = 0, 0, 0, 0
        for entries in plan:
            seqs = [e[0] for e in entries]
            rows = [e[2] for e in entries]
            past = [pos[s] for s in seqs]
            T = sum(rows)
            st = dict(seqs=seqs, rows=rows, past=past, off=off, T=T, S=len(seqs),
                      max_ctx=max(p + r for p, r in zip(past, rows)))
            cu = [0]
            for r in rows:
                cu.append(cu[-1] + r)
            st["cu"] = torch.tensor(cu, dtype=torch.int32, device=dev)
            st["past0"] = torch.tensor(past, dtype=torch.int32, device=dev)
            st["past_dev"] = st["past0"].clone()
            st["bt"] = mb.block_table[seqs].contiguous().to(dev)
            st["flops"] = sum(4 * self.D * self.HQ * visible_pairs(p, r) for p, r in zip(past, rows))
            st["bytes"] = sum((p + 1) * kv_row * 2 + self.HQ * self.D * 2 * 2 + kv_row * 2
                              for p, r in zip(past, rows) if r == 1)
            self.flops += st["flops"]
            self.decode_bytes += st["bytes"]
            self.decode_rows += sum(1 for r in rows if r == 1)
            self.prefill_rows += sum(r for r in rows if r > 1)
            for s, p, r in zip(seqs, past, rows):
                row_seq += [s] * r
                row_pos += list(range(p, p + r))
                pos[s] = p + r
            off += T
            self.steps.append(st)
        self.R = off
        self.row_seq = torch.tensor(row_seq, dtype=torch.long)
        self.row_pos = torch.tensor(row_pos, dtype=torch.long)
        self.q = torch.randn(self.R, self.HQ, self.D, generator=g, device=dev).to(bf)
        self.kn = torch.randn(self.R, self.HKV, self.D, generator=g, device=dev).to(bf)
        self.vn = torch.randn(self.R, self.HKV, self.D, generator=g, device=dev).to(bf)
        self.out = torch.zeros(self.R, self.HQ, self.D, dtype=bf, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        ws = max(cp.cp_workspace_size(self.desc, st["T"], st["max_ctx"], st["S"]) for st in self.steps)
        self.ws = torch.zeros(max(ws, 16), dtype=torch.uint8, device=dev)
        # launches per cp_mixed_step: append, decode split + combine (when decode rows), tensor-core
        # prefill (when chunks), commit
        self.launches = sum(2 + 2 * any(r == 1 for r in st["rows"]) + any(r > 1 for r in st["rows"])
                            for st in self.steps)
        self.tokens = self.R

    def step(self):
        cp = self.cp
        for st in self.steps:
            st["past_dev"].copy_(st["past0"])
        for st in self.steps:
            sl = slice(st["off"], st["off"] + st["T"])
            if self.overlap:
                cp.cp_mixed_step_overlap(self.desc, self.q[sl], self.kn[sl], self.vn[sl], self.kp, self.vp,
                                         st["bt"], st["cu"], st["past_dev"], st["S"], st["T"], st["max_ctx"],
                                         self.out[sl], self.ws, *self.handles, dev_status=self.status)
            else:
                cp.cp_mixed_step(self.desc, self.q[sl], self.kn[sl], self.vn[sl], self.kp, self.vp, st["bt"],
                                 st["cu"], st["past_dev"], st["S"], st["T"], st["max_ctx"], self.out[sl], self.ws,
                                 dev_status=self.status)

    def self_check(self, n_sample=24, seed=17):
        """Every row's K/V lands in its page slot bit for bit (page =
        block_table[seq][pos / 16], offset pos mod 16); past lengths advance by
        the rows; sampled decode and prefill rows agree with ref_rows over the
        sequence's positions [0, pos] gathered from the pools."""
        torch = self.torch
        torch.cuda.synchronize()
        P = self.mb.page_size
        table = self.mb.block_table.to(self.dev).long()
        seq = self.row_seq.to(self.dev)
        pos = self.row_pos.to(self.dev)
        page = table[seq, pos // P]
        slot = pos % P
        kv_ok = bits_equal(self.kp[page, :, slot], self.kn) and bits_equal(self.vp[page, :, slot], self.vn)
        past_ok = all(st["past_dev"].tolist() == [p + r for p, r in zip(st["past"], st["rows"])]
                      for st in self.steps)
        g = torch.Generator().manual_seed(seed)
        picks = {0, self.R - 1}
        while len(picks) < n_sample:
            picks.add(int(torch.randint(0, self.R, (1,), generator=g)))
        err = 0.0
        for i in sorted(picks):
            s, p = int(self.row_seq[i]), int(self.row_pos[i])
            a = torch.arange(p + 1, device=self.dev)
            pg = table[s, a // P]
            keys = self.kp[pg, :, a % P]
            vals = self.vp[pg, :, a % P]
            ref = ref_rows(self.q[i], keys, vals, self.D ** -0.5)
            err = max(err, float((self.out[i].float() - ref).abs().max()))
        status = int(self.status.item())
        ok = kv_ok and past_ok and status == 0 and err < BF16_TOL
        return {"ok": ok, "pages_bit_exact": kv_ok, "past_len_ok": past_ok, "rows_checked": len(picks),
                "max_abs_err": err, "tol": BF16_TOL, "status": status}

    def config(self):
        name = "decode64" if self.decode_only else f"mixed_budget{self.budget}" + ("_overlap" if self.overlap else "")
        return {"workload": f"paged_{name}_gqa32x8_d128_bf16_page16",
                "schedule_steps": len(self.steps), "rows_per_schedule": self.R,
                "decode_rows": self.decode_rows, "prefill_rows": self.prefill_rows,
                "decode_ctx_mean": sum(self.mb.decode_ctx) / len(self.mb.decode_ctx),
                "prompts": self.mb.prompt_lens, "page_size": self.mb.page_size, "l2": L2_NOTE,
                "cuda_graph": True}


class ShortChunks:
    """Short chunks at long cached lengths over a contiguous cache.

    ``verify``: 64 sequences, each with 4000 cached positions, take a 4-row
    chunk (a speculative-verify step: k = 4 draft tokens checked in one pass;
    the glossary's related techniques), one cp_prefill_chunk call.
    ``varlen``: one cp_prefill_varlen call over 8 sequences with ragged rows
    and different cached lengths (a step filled with chunks of several
    prompts): rows [2048, 1024, 512, 512, 256, 128, 64, 1] at lengths
    [0, 1024, 3000, 512, 6000, 7000, 100, 4095].  GQA 32/8 x 128 bf16, cache
    capacity 8192, N(0,1) history drawn on the device.
    ``deep``: one 8128-row chunk of one sequence at 8128 cached positions (the
    size of a budget-8192 step's prompt chunk), one cp_prefill_chunk call (one
    launch): the kernel's steady state, with its per-launch fixed cost spread
    over a long key walk."""

    HQ, HKV, D = 32, 8, 128

    def __init__(self, dev, mode, overlap=False):
        import torch
        import chunked_prefill_causal_cp_gb300 as cp

        self.cp, self.torch, self.dev, self.mode = cp, torch, dev, mode
        # varlen: the one-row sequence's split-KV kernels on a side stream (cp_prefill_varlen_overlap)
        self.overlap = overlap and mode == "varlen"
        if self.overlap:
            self.side = torch.cuda.Stream(dev)
            self.fork, self.join = torch.cuda.Event(), torch.cuda.Event()
        bf = torch.bfloat16
        if mode == "verify":
            self.B, self.k, self.cap = 64, 4, 4096 + 8
            self.pasts = [4000] * self.B
            self.rows = [self.k] * self.B
        elif mode == "deep":
            self.B, self.cap = 1, 16384
            self.pasts, self.rows = [8128], [8128]
        else:
            self.cap = 8192
            self.rows = [2048, 1024, 512, 512, 256, 128, 64, 1]
            self.pasts = [0, 1024, 3000, 512, 6000, 7000, 100, 4095]
            self.B = len(self.rows)
        g = torch.Generator(device=dev).manual_seed(9)
        self.kc = torch.randn(self.B, self.HKV, self.cap, self.D, generator=g, device=dev).to(bf)
        self.vc = torch.randn(self.B, self.HKV, self.cap, self.D, generator=g, device=dev).to(bf)
        self.T = sum(self.rows)
        self.q = torch.randn(self.T, self.HQ, self.D, generator=g, device=dev).to(bf)
        self.kn = torch.randn(self.T, self.HKV, self.D, generator=g, device=dev).to(bf)
        self.vn = torch.randn(self.T, self.HKV, self.D, generator=g, device=dev).to(bf)
        self.out = torch.zeros(self.T, self.HQ, self.D, dtype=bf, device=dev)
        self.desc = cp.layer_desc(bf, self.B, self.HQ, self.HKV, self.D, cp.CP_CACHE_CONTIG, capacity=self.cap)
        self.past0 = torch.tensor(self.pasts, dtype=torch.int32, device=dev)
        self.lens = self.past0.clone()
        cu = [0]
        for r in self.rows:
            cu.append(cu[-1] + r)
        self.cu_host = cu
        self.cu = torch.tensor(cu, dtype=torch.int32, device=dev)
        self.max_ctx = max(p + r for p, r in zip(self.pasts, self.rows))
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.ws = torch.zeros(max(16, cp.cp_workspace_size(self.desc, self.T, self.max_ctx, self.B)),
                              dtype=torch.uint8, device=dev)
        kv_row = self.HKV * self.D * 2
        self.flops = sum(4 * self.D * self.HQ * visible_pairs(p, r) for p, r in zip(self.pasts, self.rows))
        # algorithmic bytes: cached K/V read once per (sequence, KV head), the new rows' q, k, v and out
        self.bytes = sum(p * kv_row * 2 for p in self.pasts) + self.T * (2 * self.HQ * self.D * 2 + 2 * kv_row)
        self.tokens = self.T
        # verify: append, split-KV kernel (which also advances the lengths), combine; varlen: append,
        # split-KV kernel, combine, tensor-core kernel, commit; deep: one tensor-core launch (append and
        # length advance fused in)
        self.launches = {"verify": 3, "varlen": 5, "deep": 1}[mode]

    def step(self):
        cp = self.cp
        self.lens.copy_(self.past0)
        if self.mode in ("verify", "deep"):
            B, k = self.B, self.rows[0]
            cp.cp_prefill_chunk(self.desc, self.q.view(B, k, self.HQ, self.D), self.kn.view(B, k, self.HKV, self.D),
                                self.vn.view(B, k, self.HKV, self.D), self.kc, self.vc, self.lens, k, k,
                                max(self.pasts), self.out.view(B, k, self.HQ, self.D), self.ws,
                                dev_status=self.status)
        elif self.overlap:
            cp.cp_prefill_varlen_overlap(self.desc, self.q, self.kn, self.vn, self.kc, self.vc, self.cu, self.lens,
                                         self.B, self.T, self.max_ctx, self.out, self.ws, self.side, self.fork,
                                         self.join, dev_status=self.status)
        else:
            cp.cp_prefill_varlen(self.desc, self.q, self.kn, self.vn, self.kc, self.vc, self.cu, self.lens, self.B,
                                 self.T, self.max_ctx, self.out, self.ws, dev_status=self.status)

    def self_check(self, n_sample=24, seed=19):
        """The new rows sit in their slots bit for bit, each length advanced by its
        rows, sampled rows agree with ref_rows over the sequence's slots [0, pos]."""
        torch = self.torch
        torch.cuda.synchronize()
        slots_ok = True
        for s, (p, r) in enumerate(zip(self.pasts, self.rows)):
            t = self.cu_host[s]
            slots_ok = slots_ok and bits_equal(self.kc[s, :, p:p + r].transpose(0, 1), self.kn[t:t + r]) \
                and bits_equal(self.vc[s, :, p:p + r].transpose(0, 1), self.vn[t:t + r])
        lens_ok = self.lens.tolist() == [p + r for p, r in zip(self.pasts, self.rows)]
        g = torch.Generator().manual_seed(seed)
        picks = {0, self.T - 1}
        while len(picks) < n_sample:
            picks.add(int(torch.randint(0, self.T, (1,), generator=g)))
        err = 0.0
        for i in sorted(picks):
            s = max(j for j in range(self.B) if self.cu_host[j] <= i)
            pos = self.pasts[s] + (i - self.cu_host[s])
            ref = ref_rows(self.q[i], self.kc[s, :, :pos + 1].transpose(0, 1), self.vc[s, :, :pos + 1].transpose(0, 1),
                           self.D ** -0.5)
            err = max(err, float((self.out[i].float() - ref).abs().max()))
        status = int(self.status.item())
        ok = slots_ok and lens_ok and status == 0 and err < BF16_TOL
        return {"ok": ok, "slots_bit_exact": slots_ok, "lengths_ok": lens_ok, "rows_checked": len(picks),
                "max_abs_err": err, "tol": BF16_TOL, "status": status}

    def config(self):
        if self.mode == "verify":
            return {"workload": "verify_k4_x64_past4000_gqa32x8_d128_bf16", "sequences": self.B, "k": self.k,
                    "past": self.pasts[0], "l2": L2_NOTE, "cuda_graph": True}
        if self.mode == "deep":
            return {"workload": "deep_chunk_rows8128_past8128_gqa32x8_d128_bf16", "rows": self.rows[0],
                    "past": self.pasts[0], "capacity": self.cap, "l2": L2_NOTE, "cuda_graph": True}
        name = "varlen8_overlap_gqa32x8_d128_bf16_cap8192" if self.overlap else "varlen8_gqa32x8_d128_bf16_cap8192"
        return {"workload": name, "rows": self.rows, "pasts": self.pasts, "l2": L2_NOTE, "cuda_graph": True}


class AppendRows:
    """The KV append alone ([Wiki] 一.1: chunk k writes its own slots): 64
    sequences each append a 512-row chunk after 4000 cached positions, GQA 8
    KV heads x 128 bf16, one cp_kv_append call.  ``contig``: a contiguous cache
    of capacity 4608; ``paged``: 16-token pages from a seeded permutation of
    the pool.  Algorithmic bytes: the rows' K and V read once and written once
    (268 MB per call)."""

    HKV, D, B, R, PAST = 8, 128, 64, 512, 4000

    def __init__(self, dev, mode):
        import torch
        import chunked_prefill_causal_cp_gb300 as cp

        self.cp, self.torch, self.dev, self.mode = cp, torch, dev, mode
        bf = torch.bfloat16
        B, R, H, D = self.B, self.R, self.HKV, self.D
        g = torch.Generator(device=dev).manual_seed(13)
        self.kn = torch.randn(B, R, H, D, generator=g, device=dev).to(bf)
        self.vn = torch.randn(B, R, H, D, generator=g, device=dev).to(bf)
        self.lens = torch.full((B,), self.PAST, dtype=torch.int32, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        n = self.PAST + R
        if mode == "contig":
            self.cap = 4608
            self.desc = cp.layer_desc(bf, B, 4 * H, H, D, cp.CP_CACHE_CONTIG, capacity=self.cap)
            self.kc = torch.full((B, H, self.cap, D), -7.0, dtype=bf, device=dev)
            self.vc = torch.full_like(self.kc, -7.0)
            self.table = None
        else:
            self.page = 16
            nb = -(-n // self.page)
            perm = torch.randperm(B * nb, generator=torch.Generator().manual_seed(14))
            self.table = perm.view(B, nb).to(torch.int32).to(dev)
            self.desc = cp.layer_desc(bf, B, 4 * H, H, D, cp.CP_CACHE_PAGED, page_size=self.page,
                                      num_pages=B * nb, max_blocks=nb)
            self.kc = torch.full((B * nb, H, self.page, D), -7.0, dtype=bf, device=dev)
            self.vc = torch.full_like(self.kc, -7.0)
        self.bytes = 2 * 2 * B * R * H * D * 2
        self.tokens = B * R
        self.flops = 0
        self.launches = 1

    def step(self):
        self.cp.cp_kv_append(self.desc, self.kn, self.vn, self.R, self.kc, self.vc, self.lens, self.PAST,
                             block_table=self.table, dev_status=self.status)

    def _slots(self, cache):
        """[B, R, H, D] view of the slots of positions [PAST, PAST + R)."""
        torch = self.torch
        pos = torch.arange(self.PAST, self.PAST + self.R, device=self.dev)
        if self.mode == "contig":
            return cache[:, :, self.PAST:self.PAST + self.R].transpose(1, 2)
        pages = self.table[:, pos // self.page].long()  # [B, R]
        return cache[pages, :, (pos % self.page).expand(self.B, -1)]

    def self_check(self):
        """Every appended row sits in its slot bit for bit; every other slot still
        holds the fill value; the lengths are not modified."""
        torch = self.torch
        torch.cuda.synchronize()
        rows_ok = bits_equal(self._slots(self.kc), self.kn) and bits_equal(self._slots(self.vc), self.vn)
        written = self.B * self.R * self.HKV * self.D
        rest_ok = all(int((c == -7.0).sum()) == c.numel() - written for c in (self.kc, self.vc))
        lens_ok = bool((self.lens == self.PAST).all())
        status = int(self.status.item())
        ok = rows_ok and rest_ok and lens_ok and status == 0
        return {"ok": ok, "rows_bit_exact": rows_ok, "other_slots_untouched": rest_ok, "lengths_untouched": lens_ok,
                "status": status}

    def config(self):
        c = {"workload": f"append_{self.mode}_x64_r512_past4000_kv8_d128_bf16", "sequences": self.B, "rows": self.R,
             "past": self.PAST, "bytes_per_call": self.bytes, "l2": L2_NOTE, "cuda_graph": True}
        if self.mode == "contig":
            c["capacity"] = self.cap
        else:
            c["page_size"] = self.page
        return c


# --------------------------------------------------------------------------- measurement

def measure(wl, graph, flush, reps, warmup, torch, check_kw=None):
    """Warm-up replays, the workload's own check (a failure ends the run), then
    `reps` timed replays with L2 flushed between.  Returns (mean ms, check)."""
    for _ in range(max(warmup, 3)):
        graph.replay()
    torch.cuda.synchronize()
    check = require(wl.self_check(**(check_kw or {})), type(wl).__name__)
    times = time_steps(graph.replay, flush, reps, torch)
    return sum(times) / len(times), check


def other_configs(dev, flush, pk, reps, warmup):
    """One measurement of each other workload, each checked before it is timed."""
    import torch
    tc, hbm = float(pk["bf16_tflops"]), float(pk["hbm_gbs"])
    res = {}

    wl = ChunkLoop(dev, "fp32")
    ms, chk = measure(wl, capture(wl.step, dev), flush, reps, warmup, torch)
    alu = fp32_alu_peak_tflops(dev)
    res["fp32_example"] = {**wl.config(), "tokens_per_s": wl.tokens / (ms / 1e3), "ms_per_step": ms,
                           "tflops": wl.flops / (ms / 1e3) / 1e12, "alu_peak_tflops": alu,
                           "alu_frac_whole_step": wl.flops / (ms / 1e3) / 1e12 / alu, "dtype": "f32", "check": chk,
                           "gpu_launches_per_step": wl.launches}
    del wl

    unp = LadderRuns(dev, pad=False)
    g_unp = capture(unp.step, dev)
    g_unp.replay()
    wl = LadderRuns(dev, pad=True)
    ms, chk = measure(wl, capture(wl.step, dev), flush, reps, warmup, torch, {"unpadded": unp})
    res["padding_ladder"] = {**wl.config(), "tokens_per_s": wl.tokens / (ms / 1e3), "ms_per_step": ms,
                             "tflops_real_rows": wl.flops / (ms / 1e3) / 1e12,
                             "tensor_frac_whole_step": wl.flops / (ms / 1e3) / 1e12 / tc, "dtype": "bf16",
                             "check": chk, "gpu_launches_per_step": wl.launches}
    del wl, unp, g_unp

    wl = ChunkLoop(dev, "rolling")
    ms, chk = measure(wl, capture(wl.step, dev), flush, reps, warmup, torch)
    res["rolling"] = {**wl.config(), "tokens_per_s": wl.tokens / (ms / 1e3), "ms_per_step": ms,
                      "tflops": wl.flops / (ms / 1e3) / 1e12,
                      "tensor_frac_whole_step": wl.flops / (ms / 1e3) / 1e12 / tc, "dtype": "f16",
                      "check": chk, "gpu_launches_per_step": wl.launches}
    del wl

    wl = MixedSchedule(dev, decode_only=True)
    ms, chk = measure(wl, capture(wl.step, dev), flush, reps, warmup, torch)
    gbs = wl.decode_bytes / (ms / 1e3) / 1e9
    res["decode"] = {**wl.config(), "rows_per_s": wl.tokens / (ms / 1e3), "ms_per_step": ms,
                     "decode_bytes_per_step": wl.decode_bytes, "gbs_whole_step": gbs, "hbm_frac_whole_step": gbs / hbm,
                     "hbm_frac_nominal": gbs / HBM_NOMINAL_GBS,
                     "traffic": kernel_traffic("decode_split_paged.json"),
                     "scope": ("K/V, q and out bytes of the 64 decode rows over the whole cp_mixed_step call "
                               "(append, split-KV kernel, combine, commit): a lower bound on the kernel's rate"),
                     "dtype": "bf16", "check": chk, "gpu_launches_per_step": wl.launches}
    del wl

    for mode in ("verify", "varlen", "varlen_overlap", "deep"):
        wl = ShortChunks(dev, mode.replace("_overlap", ""), overlap=mode.endswith("_overlap"))
        ms, chk = measure(wl, capture(wl.step, dev), flush, reps, warmup, torch)
        gbs = wl.bytes / (ms / 1e3) / 1e9
        tf = wl.flops / (ms / 1e3) / 1e12
        res[mode] = {**wl.config(), "rows_per_s": wl.tokens / (ms / 1e3), "ms_per_step": ms, "tflops": tf,
                     "tensor_frac": tf / tc, "gbs_algorithmic": gbs, "hbm_frac": gbs / hbm,
                     "hbm_frac_nominal": gbs / HBM_NOMINAL_GBS,
                     "roofline_time_us": max(wl.flops / (tc * 1e12), wl.bytes / (hbm * 1e9)) * 1e6,
                     "dtype": "bf16", "check": chk, "gpu_launches_per_step": wl.launches}
        if mode == "deep":
            res[mode]["tensor_frac_sustained"] = tf / float(pk.get("bf16_tflops_sustained", tc))
        del wl

    for mode in ("contig", "paged"):
        wl = AppendRows(dev, mode)
        ms, chk = measure(wl, capture(wl.step, dev), flush, reps, warmup, torch)
        gbs = wl.bytes / (ms / 1e3) / 1e9
        res[f"append_{mode}"] = {**wl.config(), "rows_per_s": wl.tokens / (ms / 1e3), "ms_per_step": ms,
                                 "gbs_algorithmic": gbs, "hbm_frac": gbs / hbm,
                                 "hbm_frac_nominal": gbs / HBM_NOMINAL_GBS,
                                 "traffic": kernel_traffic(f"kv_append_{mode}.json"), "dtype": "bf16", "check": chk,
                                 "gpu_launches_per_step": wl.launches}
        del wl

    for budget, overlap in ((8192, False), (8192, True), (2048, False), (2048, True)):
        wl = MixedSchedule(dev, budget=budget, overlap=overlap)
        ms, chk = measure(wl, capture(wl.step, dev), flush, max(3, reps // 4), warmup, torch)
        t_star, t_serial = mixed_rooflines(wl.steps, tc, hbm)
        res[f"mixed_budget{budget}" + ("_overlap" if overlap else "")] = {
            **wl.config(), "rows_per_s": wl.tokens / (ms / 1e3), "ms_per_schedule": ms,
            "flops_per_schedule": wl.flops, "decode_bytes_per_schedule": wl.decode_bytes,
            "roofline_time_ms": t_star, "roofline_frac": t_star / ms,
            "roofline_serial_time_ms": t_serial, "roofline_serial_frac": t_serial / ms, "dtype": "bf16",
            "check": chk, "gpu_launches_per_step": wl.launches}
        del wl
    torch.cuda.synchronize()
    return res


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
    if args.sweep:
        return run_sweep(args, dev, pk)
    if args.workload != "gqa_prefill":
        return run_single(args, rank, world, dev, pk, pk_src)

    wl = GqaPrefill(dev, pad=not args.no_pad, N=args.prompt, W=args.chunk)
    wl.capture()
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    for _ in range(max(args.warmup, 3)):
        wl.graph.replay()
    torch.cuda.synchronize()
    check = require(wl.self_check(), "gqa_prefill")

    bus = None
    try:
        bus = torch.cuda.get_device_properties(dev).pci_bus_id
    except AttributeError:
        pass
    clocks = ClockSampler(bus)
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    # the clock record starts under the same load: replays of the step for about half a second
    t_end = time.perf_counter() + 0.5
    while time.perf_counter() < t_end:
        for _ in range(50):
            flush.zero_()
            wl.graph.replay()
        torch.cuda.synchronize()
    times = time_steps(wl.graph.replay, flush, args.steps, torch)
    clk = clocks.stop()
    torch.cuda.synchronize()
    barrier(world)
    total_ms, value = job_throughput(sum(times), wl.tokens, args.steps, world)
    ms_per_step = total_ms / args.steps
    if int(wl.status.item()) != 0:
        raise CheckFailed(f"device status {int(wl.status.item())} after the timed steps")

    # ---- in-situ time of the attention launches: prefix graphs of the same launch chain
    wl.capture_prefixes()
    reps = max(20, min(args.steps, 200))
    n = len(wl.sizes)
    acc = [0.0] * (n + 1)
    for _ in range(reps):
        for k in range(n + 1):
            t = time_steps(wl.prefix_graphs[k].replay, flush, 1, torch)[0]
            acc[k] += t / reps
    attn_ms = acc[n] - acc[0]
    per_chunk_us = [round((acc[k + 1] - acc[k]) * 1e3, 2) for k in range(n)]
    attn_tflops = wl.flops / (attn_ms / 1e3) / 1e12
    peak = float(pk["bf16_tflops"])
    traffic = kernel_traffic("attn_tc_gqa_prefill.json")

    # ---- end to end: host buffers in, result out, through the captured public calls
    wl.pin()
    e2e_steps = max(20, min(args.steps // 10, 300))
    wl.capture_e2e()
    for _ in range(3):
        wl.e2e_graph.replay()
    torch.cuda.synchronize()
    e2e_times = time_steps(wl.e2e_graph.replay, flush, e2e_steps, torch)
    _, e2e_value = job_throughput(sum(e2e_times), wl.tokens, e2e_steps, world)
    e2e_ok = bits_equal(wl.ho, wl.out[:wl.N].cpu())
    if int(wl.status.item()) != 0 or not e2e_ok:
        raise CheckFailed("end-to-end graph: device status set or host output differs from the device rows")

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) q/k/v)",
        "config": wl.config(),
        "effective_tflops": wl.flops * args.steps * world / (total_ms / 1e3) / 1e12,
        "flops_per_step": wl.flops,
        "check": check,
        "roofline": {"bound": "tensor", "achieved": attn_tflops, "peak": peak, "unit": "TFLOP/s",
                     "frac": attn_tflops / peak, "traffic": traffic, "kernel": "attn_tc_kernel",
                     "peak_source": f"{pk_src} bf16_tflops (burst)",
                     "frac_of_sustained": attn_tflops / float(pk.get("bf16_tflops_sustained", peak)),
                     "attention_ms_per_step": attn_ms, "launches_per_step": n,
                     "per_chunk_us": per_chunk_us,
                     "per_chunk_tflops": [round(f / (t / 1e6) / 1e12, 1) if t > 0 else None
                                          for f, t in zip(wl.flops_chunk, per_chunk_us)],
                     "kernel_timing": ("in situ: CUDA events around graphs of the first k chunk calls of the "
                                       "step (k = 0..n, the same launch chain without the pad launch), L2 "
                                       f"flushed before each, mean of {reps}; attention = T(n) - T(0), "
                                       "chunk k = T(k+1) - T(k)"),
                     "traffic_note": "mean DRAM bytes per launch over the step's chunk launches (ncu)"},
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": wl.h2d,
                "d2h_bytes_per_step": wl.d2h,
                "path": ("one captured graph per step of the public calls with its host traffic: each chunk's "
                         "q/k/v rows staged back to back in pinned host memory and copied host -> device in one "
                         "copy, all queued in chunk order on a copy stream; each chunk's call waits for its own "
                         "rows; its output rows go device -> pinned host on a second copy stream once it is done")},
        "gpu_launches": wl.launches * args.steps,
        "clocks": clk,
    }
    if rank == 0 and world == 1 and not args.no_extras:
        line["configs"] = other_configs(dev, flush, pk, max(10, min(args.steps, 50)), args.warmup)
    if rank == 0 and world == 1 and not args.skip_cpu:
        v_cpu, sample, _, diff, heads, threads = wl.cpu_sample(args.cpu_seconds)
        if not diff < BF16_TOL:
            raise CheckFailed(f"GPU output differs from the oracle by {diff} on the sampled heads")
        v1, t1 = oracle_single_thread_fp32()
        line["cpu_baseline"] = {"value": v_cpu, "unit": "tokens/s", "cores": threads,
                                "kind": "oracle (C++ fp64, std::thread)", "sample": sample,
                                "parity": {"max_abs_err_vs_gpu": diff, "tol": BF16_TOL, "query_heads": heads,
                                           "rows": wl.N},
                                "single_thread_fp32_example": {"tokens_per_s": v1, "seconds": t1, "cores": 1,
                                                               "workload": "fp32_mha8_d64_prompt1000_chunk256"},
                                "configs": oracle_config_samples()}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_sweep(args, dev, pk):
    """Sweeps of the chunk width W of the GQA prompt and of the token budget of
    the mixed schedule, one line each (each checked first)."""
    import torch
    tc, hbm = float(pk["bf16_tflops"]), float(pk["hbm_gbs"])
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    reps = max(5, min(args.steps, 50))
    for W in (128, 256, 512, 1024, 2048, 4096):
        wl = GqaPrefill(dev, N=args.prompt, W=W)
        ms, chk = measure(wl, wl.capture(), flush, reps, args.warmup, torch)
        print(json.dumps({"sweep": "chunk", "W": W, "prompt": wl.N, "chunks": len(wl.sizes),
                          "query_widths": sorted(set(wl.widths)),
                          "padded_rows": sum(w - r for r, w in zip(wl.sizes, wl.widths)),
                          "tokens_per_s": wl.tokens / (ms / 1e3), "ms_per_step": ms,
                          "tflops": wl.flops / (ms / 1e3) / 1e12, "check_ok": chk["ok"],
                          "max_abs_err": chk["max_abs_err"]}), flush=True)
        del wl
    for budget in (512, 1024, 2048, 4096, 8192, 16384):
        wl = MixedSchedule(dev, budget=budget)
        ms, chk = measure(wl, capture(wl.step, dev), flush, max(3, reps // 5), args.warmup, torch)
        t_star, t_serial = mixed_rooflines(wl.steps, tc, hbm)
        print(json.dumps({"sweep": "budget", "budget": budget, "schedule_steps": len(wl.steps),
                          "rows_per_schedule": wl.R, "rows_per_s": wl.tokens / (ms / 1e3), "ms_per_schedule": ms,
                          "roofline_time_ms": t_star, "roofline_frac": t_star / ms,
                          "roofline_serial_time_ms": t_serial, "roofline_serial_frac": t_serial / ms,
                          "check_ok": chk["ok"], "max_abs_err": chk["max_abs_err"]}), flush=True)
        del wl
        torch.cuda.empty_cache()


def run_single(args, rank, world, dev, pk, pk_src):
    """One line for one of the other workloads."""
    import torch
    tc, hbm = float(pk["bf16_tflops"]), float(pk["hbm_gbs"])
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    kw = None
    if args.workload in ("fp32", "rolling"):
        wl = ChunkLoop(dev, args.workload)
    elif args.workload in ("verify", "varlen", "deep"):
        wl = ShortChunks(dev, args.workload, overlap=args.overlap)
    elif args.workload in ("append", "append_paged"):
        wl = AppendRows(dev, "paged" if args.workload == "append_paged" else "contig")
    elif args.workload == "ladder":
        unp = LadderRuns(dev, pad=False)
        capture(unp.step, dev).replay()
        kw = {"unpadded": unp}
        wl = LadderRuns(dev, pad=not args.no_pad)
    else:
        wl = MixedSchedule(dev, budget=args.budget, decode_only=args.workload == "decode", overlap=args.overlap)
    g = capture(wl.step, dev)
    for _ in range(max(args.warmup, 3)):
        g.replay()
    torch.cuda.synchronize()
    check = require(wl.self_check(**(kw or {})), args.workload)
    clocks = ClockSampler()
    clocks.start()
    times = time_steps(g.replay, flush, args.steps, torch)
    clk = clocks.stop()
    total_ms = max_over_ranks(sum(times), world)
    ms = total_ms / args.steps
    if int(wl.status.item()) != 0:
        raise CheckFailed(f"device status {int(wl.status.item())} after the timed steps")
    units = wl.tokens
    line = {"metric": f"{args.workload} tokens/s", "value": world * units * args.steps / (total_ms / 1e3),
            "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "data": "synthetic",
            "config": wl.config(), "flops_per_step": wl.flops, "tflops_whole_step": wl.flops / (ms / 1e3) / 1e12,
            "check": check, "gpu_launches": wl.launches * args.steps, "clocks": clk, "peaks": pk_src}
    if args.workload == "fp32":
        line["dtype"] = "f32"
        alu = fp32_alu_peak_tflops(dev)
        line["roofline"] = {"bound": "alu", "achieved": wl.flops / (ms / 1e3) / 1e12, "peak": alu, "unit": "TFLOP/s",
                            "frac": wl.flops / (ms / 1e3) / 1e12 / alu, "kernel": "attn_f32_kernel",
                            "peak_source": "SMs x 128 FP32 FMA lanes x 2 x 2070 MHz",
                            "scope": "algorithmic FLOPs over the whole step (append, attention and commit launches)"}
    else:
        line["dtype"] = "f16" if args.workload == "rolling" else "bf16"
        line["tensor_frac_whole_step"] = wl.flops / (ms / 1e3) / 1e12 / tc
    if args.workload == "decode":
        gbs = wl.decode_bytes / (ms / 1e3) / 1e9
        line["roofline"] = {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                            "frac_of_nominal": gbs / HBM_NOMINAL_GBS,
                            "traffic": kernel_traffic("decode_split_paged.json"), "kernel": "decode_split_kernel",
                            "scope": "decode rows' bytes over the whole call: a lower bound on the kernel's rate"}
    if args.workload == "mixed":
        t_star, t_serial = mixed_rooflines(wl.steps, tc, hbm)
        line["roofline_time_ms"] = t_star
        line["roofline_frac"] = t_star / ms
        line["roofline_serial_time_ms"] = t_serial
        line["roofline_serial_frac"] = t_serial / ms
    if args.workload == "ladder":
        line["padded_rows_per_step"] = wl.padded_rows
    if args.workload in ("verify", "varlen", "deep"):
        gbs = wl.bytes / (ms / 1e3) / 1e9
        line["roofline"] = {"bound": "hbm" if args.workload == "verify" else "tensor",
                            "achieved": gbs if args.workload == "verify" else wl.flops / (ms / 1e3) / 1e12,
                            "peak": hbm if args.workload == "verify" else tc,
                            "unit": "GB/s" if args.workload == "verify" else "TFLOP/s",
                            "scope": "algorithmic bytes or FLOPs over the whole call"}
        line["roofline"]["frac"] = line["roofline"]["achieved"] / line["roofline"]["peak"]
        if args.workload == "verify":
            line["roofline"]["frac_of_nominal"] = gbs / HBM_NOMINAL_GBS
    if args.workload in ("append", "append_paged"):
        gbs = wl.bytes / (ms / 1e3) / 1e9
        line["roofline"] = {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                            "frac_of_nominal": gbs / HBM_NOMINAL_GBS,
                            "traffic": kernel_traffic(f"kv_append_{wl.mode}.json"), "kernel": "kv_append_kernel",
                            "scope": "the rows' K/V read and written once, over the call (one launch)"}
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_reference(args):
    """The C++ CPU oracle as the reference arm (rank 0 only): each step is one
    KV-head group of the default workload (its 4 query heads over the whole
    4000-token prompt in chunks of 512), threaded over every host core;
    tokens/s is scaled to all 8 groups."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from oracle import cpp as oracle
    import synth_inputs as SI
    N, W, HQ, HKV = 4000, 512, GqaPrefill.HQ, GqaPrefill.HKV
    oracle.build()
    oracle.set_threads(0)
    q, k, v = SI.gqa_prompt(N, seed=1)
    qn, kn, vn = (t.double().numpy() for t in (q, k, v))
    G = HQ // HKV
    sizes = oracle.chunk_plan(N, W)

    def one_group(g):
        oracle.chunked_prefill(qn[:, g * G:(g + 1) * G], kn[:, g:g + 1], vn[:, g:g + 1], W)

    for i in range(args.warmup):
        one_group(i % HKV)
    times = []
    t_budget = 150.0
    t_start = time.perf_counter()
    for i in range(args.steps):
        t0 = time.perf_counter()
        one_group(i % HKV)
        times.append(time.perf_counter() - t0)
        if time.perf_counter() - t_start > t_budget:
            break
    per_group = sum(times) / len(times)
    value = N / (per_group * HKV)
    sample = (f"each step: C++ oracle chunked_prefill of the 4000-token prompt (chunks {sizes}) for one KV-head "
              f"group ({G} of {HQ} query heads); tokens/s scaled to all {HKV} groups; "
              f"{len(times)} of {args.steps} requested steps timed within a {t_budget:.0f} s budget")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": len(times), "steps_requested": args.steps, "warmup": args.warmup,
            "ms_per_step": per_group * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic (seeded N(0,1) q/k/v)",
            "config": {"workload": "gqa32x8_d128_bf16_prompt4000_chunk512_cap8192", "prompt_tokens": 4000,
                       "chunk": 512, "kv_capacity": 8192, "heads_q": 32, "heads_kv": 8, "head_dim": 128},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle.threads(),
                             "kind": "oracle (C++ fp64, std::thread)", "sample": sample},
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
