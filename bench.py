"""Benchmark of the multi-head attention forward pass on GB300.

One step = the whole sublayer (Q/K/V projections + head split, fused attention
+ concat, output projection) over one batch of the long-sequence causal
self-attention workload: B=4, L=8192, d_model=1024, h=16, d_k=64, causal mask,
bf16 storage, fp32 accumulation, synthetic N(0,1) inputs and Xavier-uniform
weights (seeded), inputs resident in HBM. The L2 cache (129 MB) is flushed
before every timed step by writing a 256 MB buffer outside the timed events.

Prints ONE JSON line (rank 0). ``value`` is algorithmic TFLOP/s (4 projection
GEMMs + 4*d_k flops per allowed query/key pair per head) of the whole job.
``--impl reference`` times the fp64 CPU oracle on a bounded causal-prefix
sample of the same workload instead.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MHA fwd TFLOP/s (bf16) and % of GB300 dense-BF16 peak; tokens/s"
WORKLOAD = "long"
DESCRIPTION = {
    "enc": "encoder self-attention B32 L128 d_model512 h8 d_k64, key padding U{64..128}",
    "dec": "decoder masked self-attention B32 L256 d_model512 h8 d_k64, causal AND key padding U{128..256}",
    "xattn": "encoder-decoder attention B16 Lq256 Lk320 d_model1024 h16 d_k64, memory as key/value, padding U{160..320}",
    "long": "long-sequence causal self-attention B4 L8192 d_model1024 h16 d_k64",
    "long_d128": "long-sequence causal self-attention B4 L8192 d_model1024 h8 d_k128",
    "tiny": "tiny fp32 self-attention B2 L10 d_model512 h8 d_k64, key padding valid lens [10, 7]",
}
KERNEL_SOURCES = {"qkv_projection_gemm": "gemm_tc2.cu", "attention_core": "attn_tc.cu",
                  "output_projection_gemm": "gemm_tc2.cu"}


def kernel_source(kernel: str, workload: str = WORKLOAD) -> str:
    """Source file of the kernel that runs `kernel` on `workload` (head width 128 has its own attention)."""
    if kernel == "attention_core" and workload == "long_d128":
        return "attn_tc_d128.cu"
    return KERNEL_SOURCES[kernel]


def source_digest(kernel: str, workload: str = WORKLOAD) -> str:
    import hashlib
    csrc = os.path.join(ROOT, "transformer_head_scaled_fwd_gb300", "csrc")
    h = hashlib.sha1()
    for f in (kernel_source(kernel, workload), "ptx.cuh", "mha_internal.h", "tmem_ldst.inc"):
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def committed_traffic(kernel: str, workload: str):
    """DRAM bytes per launch (ncu dram__bytes_read.sum + dram__bytes_write.sum) recorded in a
    profiles/*.md summary for this kernel and workload, if the kernel source is unchanged since."""
    import glob
    import re
    pat = re.compile(r"<!-- bench-traffic kernel=(\S+) workload=(\S+) source_sha1=(\S+) bytes_per_launch=(\d+) -->")
    for f in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        for m in pat.finditer(open(f).read()):
            if m.group(1) == kernel and m.group(2) == workload and m.group(3) == source_digest(kernel, workload):
                return int(m.group(4))
    return None


PEAKS_FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(PEAKS_FALLBACK), "fallback"


def algorithmic_flops(B, Lq, Lk, d, h, causal, valid_lens=None):
    """4 projection GEMMs (2*M*N*K each) + 4*d_k flops per allowed (query, key) pair per head."""
    dk = d // h
    proj = 2.0 * d * d * (2 * B * Lq + 2 * B * Lk)
    pairs = 0
    for b in range(B):
        vl = Lk if valid_lens is None else max(0, min(int(valid_lens[b]), Lk))
        if causal:
            # key j allowed iff j <= i and j < vl; with vl == 0 every key carries weight
            if vl == 0:
                pairs += Lq * Lk
            else:
                i = np.arange(Lq)
                pairs += int(np.minimum(i + 1, vl).sum())
        else:
            pairs += Lq * (vl if vl > 0 else Lk)
    attn = 4.0 * dk * pairs * h
    return proj, attn


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms while the timed regions run."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(self.gpu)], stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.file is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.file.flush()
        rows = []
        with open(self.file.name) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.file.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        smax = [v for v in (num(r[2]) for r in rows) if v is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in rows for k in range(4) if r[5 + k].lower() == "active"})
        power = [v for v in (num(r[3]) for r in rows) if v is not None]
        # "under load": samples drawing at least half the peak power seen (and 150 W), i.e. taken
        # while kernels ran rather than between the timed loops
        p_max = max(power) if power else None
        cut = max(150.0, 0.5 * p_max) if p_max else None
        loaded = [r for r in rows if cut is not None and num(r[3]) is not None and num(r[3]) >= cut]
        sm_loaded = [v for v in (num(r[1]) for r in loaded) if v is not None]
        sm_all = [v for v in (num(r[1]) for r in rows) if v is not None]
        sm = sm_loaded or sm_all
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows), "samples_under_load": len(sm_loaded),
                "sm_mhz_min_under_load": min(sm_loaded) if sm_loaded else None,
                "power_w_max": p_max}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def rank_inputs(wl, rank: int):
    """Weak scaling: every rank processes a full per-GPU batch of the workload, drawn
    with its own seed (independent sequences, no data-path exchange between ranks)."""
    from transformer_head_scaled_fwd_gb300 import workloads as W
    return W.make_inputs(wl, seed_offset=rank)


def job_times(local_total_ms: float, local_e2e_ms: float, world: int, device=None):
    """Whole-job timing: the slowest rank's totals (max over ranks)."""
    if world == 1:
        return local_total_ms, local_e2e_ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([local_total_ms, local_e2e_ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t[0].item()), float(t[1].item())


def job_throughput(world: int, flops_per_rank: float, ms_per_step: float) -> float:
    """TFLOP/s of the whole job: units all ranks processed / the max-over-ranks time."""
    return world * flops_per_rank / (ms_per_step * 1e-3) / 1e12


def oracle_sample(workload: str, prefix: int):
    """A bounded, complete sub-problem of ``workload`` for the fp64 oracle.

    Long sequences: one sequence's causal prefix of ``prefix`` tokens (rows
    0..P-1 of a causal output depend only on tokens 0..P-1). Short ones: the
    whole batch of the workload with its masks (a second or two of fp64
    work). Returns (run, flops, tokens, description)."""
    import oracle
    from transformer_head_scaled_fwd_gb300 import workloads as W
    oracle.build()
    wl = W.WORKLOADS[workload]
    if wl.Lq > prefix:
        assert wl.causal and wl.self_attn
        inp = W.make_inputs(wl, B=1)
        x = np.ascontiguousarray(inp.query[:, :prefix])
        q = k = v = x
        Bs, Lq, Lk = 1, prefix, prefix
        vl = None
        desc = f"1 sequence, causal prefix of {prefix} tokens"
    else:
        inp = W.make_inputs(wl)
        q = np.ascontiguousarray(inp.query)
        k = q if inp.key is inp.query else np.ascontiguousarray(inp.key)
        v = k
        Bs, Lq, Lk = q.shape[0], q.shape[1], k.shape[1]
        vl = None if inp.valid_lens is None else np.ascontiguousarray(inp.valid_lens)
        desc = f"the whole workload ({Bs} sequences, L_q {Lq}, L_k {Lk}) with its masks"
    w = inp.weights
    proj, attn = algorithmic_flops(Bs, Lq, Lk, wl.d_model, wl.h, wl.causal, vl)

    def run():
        oracle.mha_forward(q, k, v, w["w_q"], w["b_q"], w["w_k"], w["b_k"], w["w_v"], w["b_v"], w["w_o"],
                           w["b_o"], wl.h, causal=wl.causal, valid_lens=vl)

    desc += f" (d_model {wl.d_model}, h {wl.h}), fp64 C oracle, OpenMP"
    return run, proj + attn, Bs * Lq, desc


def run_reference(args):
    """The fp64 oracle on the host cores, on a bounded sample of the workload."""
    world, rank, _ = dist_setup()
    if rank != 0:
        return
    import oracle
    run, flops, tokens, sample = oracle_sample(args.workload, args.ref_prefix)
    times = []
    for s in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        run()
        dt = time.perf_counter() - t0
        if s >= args.warmup:
            times.append(dt)
    mean = sum(times) / len(times)
    value = flops / mean / 1e12
    cores = oracle.num_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": DESCRIPTION[args.workload] + " (oracle sample)", "sample": sample},
        "tokens_per_s": tokens / mean,
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def cpu_baseline(workload: str, prefix: int):
    import oracle
    run, flops, _, sample = oracle_sample(workload, prefix)
    runs, t0 = 0, time.perf_counter()
    while True:   # about 10 s of CPU work: repeat the sample
        run()
        runs += 1
        dt = time.perf_counter() - t0
        if dt >= 10.0 or runs >= 30:
            break
    return {"value": runs * flops / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(),
            "kind": "oracle", "seconds": dt, "sample": f"{runs} runs of {sample}"}


def host_pipeline_launches(B: int, L_q: int, L_k: int, d_model: int, q_distinct: bool, kv_distinct: bool) -> int:
    """Library kernels one bf16 mha_forward_host call launches: 3 per chunk of sequences
    (up to 4 chunks when the host input is at least 32 MiB, else up to 2), plus one more
    projection at each end when query, key and value are one host buffer (the first chunk's
    Q/K/V projection and the last chunk's output projection each run in 2 row windows; one
    chunk holds both ends when B = 1)."""
    in_bytes = 2 * B * d_model * (L_q + (L_k if q_distinct else 0) + (L_k if kv_distinct else 0))
    n = 3 * min(B, 4 if in_bytes >= 32 << 20 else 2)
    if not q_distinct and not kv_distinct and L_q == L_k and L_q >= 256:
        n += 2
    return n


class WorkloadRun:
    """One workload on the current GPU, inputs resident in HBM: the whole sublayer through the
    public entry point mha_forward (one call per step), and the three stage entry points timed
    one by one with CUDA events between them (the per-kernel breakdown and the attention core)."""

    def __init__(self, name, rank=0, device=0):
        import torch
        from transformer_head_scaled_fwd_gb300 import binding
        from transformer_head_scaled_fwd_gb300 import workloads as W
        self.torch, self.binding = torch, binding
        self.name = name
        self.wl = wl = W.WORKLOADS[name]
        self.inp = inp = rank_inputs(wl, rank)
        self.tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
        self.dt = binding.MHA_BF16 if wl.dtype == "bf16" else binding.MHA_F32
        dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(f"cuda:{device}").to(self.tdt)
        self.q = dev(inp.query)
        self.k = self.q if inp.key is inp.query else dev(inp.key)
        self.v = self.k if inp.value is inp.key else dev(inp.value)
        self.Wt = {n: dev(a) for n, a in inp.weights.items()}
        self.B, self.Lq, self.d = inp.query.shape
        self.Lk = inp.key.shape[1]
        self.h = wl.h
        vl = None if inp.valid_lens is None else torch.from_numpy(inp.valid_lens).cuda()
        self.vl = vl
        self.mask = binding.make_mask(wl.causal, vl, None)
        self.ws = torch.empty(binding.workspace_size(self.dt, self.B, self.Lq, self.Lk, self.d, self.h),
                              dtype=torch.uint8, device="cuda")
        self.out = torch.empty(self.B, self.Lq, self.d, dtype=self.tdt, device="cuda")
        self.proj, self.attn = algorithmic_flops(self.B, self.Lq, self.Lk, self.d, self.h, wl.causal,
                                                 inp.valid_lens)
        self.flops = self.proj + self.attn
        # launches of one mha_forward: the Q/K/V projection, the attention, the output projection
        # (bf16 and fp32 alike)
        self.launches_per_step = 3
        # attention-core algorithmic bytes: Q, K, V read once, ctx written
        es = 2 if wl.dtype == "bf16" else 4
        self.core_bytes = es * (self.B * self.Lq * self.d + 2 * self.B * self.Lk * self.d + self.B * self.Lq * self.d)

    def forward(self, stream):
        W = self.Wt
        self.binding.mha_forward(self.q, self.k, self.v, W["w_q"], W["b_q"], W["w_k"], W["b_k"], W["w_v"],
                                 W["b_v"], W["w_o"], W["b_o"], self.h, out=self.out, workspace=self.ws,
                                 mask=self.mask, stream=stream)

    def stages(self, stream, marks):
        W, b = self.Wt, self.binding
        b.mha_qkv_projection(self.q, self.k, self.v, W["w_q"], W["b_q"], W["w_k"], W["b_k"], W["w_v"], W["b_v"],
                             self.h, workspace=self.ws, stream=stream)
        marks[1].record(stream)
        b.mha_attention_core(self.dt, self.B, self.Lq, self.Lk, self.d, self.h, workspace=self.ws,
                             mask=self.mask, stream=stream)
        marks[2].record(stream)
        b.mha_output_projection(W["w_o"], W["b_o"], self.B, self.Lq, self.Lk, self.h, out=self.out,
                                workspace=self.ws, stream=stream)

    def time_steps(self, steps, warmup, flush, stream):
        """Mean and median ms of `steps` mha_forward calls (L2 flushed before each, outside the events)."""
        torch = self.torch
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps + warmup)]
        for s in range(warmup + steps):
            flush.zero_()
            ev[s][0].record(stream)
            self.forward(stream)
            ev[s][1].record(stream)
        torch.cuda.synchronize()
        ms = [a.elapsed_time(b) for a, b in ev[warmup:]]
        return ms

    def time_stages(self, steps, warmup, flush, stream):
        """Per-stage ms from the three stage entry points with events between them."""
        torch = self.torch
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps + warmup)]
        for s in range(warmup + steps):
            flush.zero_()
            evs[s][0].record(stream)
            self.stages(stream, evs[s])
            evs[s][3].record(stream)
        torch.cuda.synchronize()
        t = evs[warmup:]
        return ([e[0].elapsed_time(e[1]) for e in t], [e[1].elapsed_time(e[2]) for e in t],
                [e[2].elapsed_time(e[3]) for e in t])

    def core_record(self, att_ms, peaks):
        m = statistics.mean(att_ms)
        return {"ms": m, "median_ms": statistics.median(att_ms), "tflops": self.attn / (m * 1e-3) / 1e12,
                "algorithmic_bytes": self.core_bytes, "gbs": self.core_bytes / (m * 1e-3) / 1e9,
                "hbm_frac": self.core_bytes / (m * 1e-3) / 1e9 / float(peaks["hbm_gbs"]),
                "bf16_frac": self.attn / (m * 1e-3) / 1e12 / float(peaks["bf16_tflops"])}


def per_workload_records(names, peaks, flush, stream, steps=50, warmup=5):
    """Short records of the other workloads (one GPU, rank 0): step time through mha_forward,
    TFLOP/s, and the attention core's time, GB/s and fractions of the measured peaks."""
    out, launches = {}, 0
    for name in names:
        r = WorkloadRun(name)
        ms = r.time_steps(steps, warmup, flush, stream)
        q_ms, a_ms, o_ms = r.time_stages(steps, warmup, flush, stream)
        # mha_forward calls and stage triples, warm-up included (the fp32 stages also launch 4 kernels)
        launches += 2 * r.launches_per_step * (steps + warmup)
        mean = statistics.mean(ms)
        core = r.core_record(a_ms, peaks)
        bound = "tensor" if name.startswith("long") else ("latency" if r.wl.dtype == "f32" else "hbm")
        frac = core["bf16_frac"] if bound == "tensor" else (core["hbm_frac"] if bound == "hbm" else None)
        out[name] = {"workload": DESCRIPTION[name], "dtype": r.wl.dtype, "steps": steps,
                     "ms_per_step": mean, "median_ms_per_step": statistics.median(ms),
                     "tflops": r.flops / (mean * 1e-3) / 1e12, "tokens_per_s": r.B * r.Lq / (mean * 1e-3),
                     "stage_ms": {"qkv_projection_gemm": round(statistics.mean(q_ms), 5),
                                  "attention_core": round(statistics.mean(a_ms), 5),
                                  "output_projection_gemm": round(statistics.mean(o_ms), 5)},
                     "attention_core": {**core, "bound": bound, "frac": frac}}
        del r
    return out, launches


def run_gpu(args):
    import torch
    import torch.distributed as dist

    from transformer_head_scaled_fwd_gb300 import binding
    from transformer_head_scaled_fwd_gb300 import build as B

    world, rank, local = dist_setup()
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    B.build()
    binding.load()
    peaks, peak_src = load_peaks()

    # CPU baseline first (rank 0, N=1 only), before any GPU work is timed.
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args.workload, args.ref_prefix)

    # weak scaling: every rank runs the full per-GPU batch with its own seed
    r = WorkloadRun(args.workload, rank, local)
    wl, inp = r.wl, r.inp
    dt = r.tdt
    Bn, Lq, Lk, d, h = r.B, r.Lq, r.Lk, r.d, r.h
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    proj, attn, flops = r.proj, r.attn, r.flops
    K, Wm = args.steps, args.warmup
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K + Wm)]

    # ---- end to end through the host-buffer entry point (pinned host in/out)
    hq = torch.from_numpy(np.ascontiguousarray(inp.query)).to(dt).pin_memory()
    hk = hq if inp.key is inp.query else torch.from_numpy(inp.key).to(dt).pin_memory()
    hv = hk if inp.value is inp.key else torch.from_numpy(inp.value).to(dt).pin_memory()
    hout = torch.empty(Bn, Lq, d, dtype=dt).pin_memory()
    staging = torch.empty(binding.host_staging_size(binding.MHA_BF16, Bn, Lq, Lk, d, hv is not hk, hk is not hq),
                          dtype=torch.uint8, device="cuda")
    h2d = hq.numel() * 2 + (hk.numel() * 2 if hk is not hq else 0) + (hv.numel() * 2 if hv is not hk else 0)
    d2h = hout.numel() * 2
    e2e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(Wm + K)]
    Wt, mask, ws = r.Wt, r.mask, r.ws

    def e2e_step(s):
        flush.zero_()
        e2e_ev[s][0].record(stream)
        binding.mha_forward_host(hq, hk, hv, Wt["w_q"], Wt["b_q"], Wt["w_k"], Wt["b_k"], Wt["w_v"], Wt["b_v"],
                                 Wt["w_o"], Wt["b_o"], h, h_out=hout, staging=staging, workspace=ws, mask=mask,
                                 stream=stream)
        e2e_ev[s][1].record(stream)

    def dev_step(s):
        flush.zero_()                      # evict L2 between steps (outside the events)
        evs[s][0].record(stream)
        r.forward(stream)
        evs[s][1].record(stream)

    # warm-up (untimed): device steps and host-buffer steps
    for s in range(Wm):
        dev_step(s)
        e2e_step(s)
    torch.cuda.synchronize()

    # ---- the same call captured once in a CUDA graph (replayed below)
    graph = None
    if not args.no_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            r.forward(torch.cuda.current_stream())
        for s in range(Wm):
            flush.zero_()
            graph.replay()
        torch.cuda.synchronize()
    g_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]

    launches = 0
    stage_steps = min(K, 100)
    with ClockSampler(local) as clk:
        time.sleep(0.3)                        # let the sampler start
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        for s in range(Wm, Wm + K):
            dev_step(s)
            launches += r.launches_per_step
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        # the per-kernel breakdown: the three stage entry points with events between them
        q_ms, att_ms, out_ms = r.time_stages(stage_steps, 2, flush, stream)
        launches += r.launches_per_step * (stage_steps + 2)
        per_e2e = host_pipeline_launches(Bn, Lq, Lk, d, inp.key is not inp.query, inp.value is not inp.key)
        for s in range(Wm, Wm + K):
            e2e_step(s)
            launches += per_e2e
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        if graph is not None:
            for s in range(K):
                flush.zero_()
                g_ev[s][0].record(stream)
                graph.replay()
                g_ev[s][1].record(stream)
                launches += r.launches_per_step
            torch.cuda.synchronize()
            if world > 1:
                dist.barrier()
        per_wl = None
        if rank == 0 and world == 1 and not args.no_per_workload:
            names = [n for n in ("enc", "dec", "xattn", "tiny", "long_d128", "long") if n != args.workload]
            per_wl, n_l = per_workload_records(names, peaks, flush, stream)
            launches += n_l
    status = binding.mha_check_device_status(reset=True)
    if status != 0:
        raise RuntimeError(f"a pipeline wait gave up inside a kernel (status 0x{status:x})")
    step_ms = [a.elapsed_time(b) for a, b in evs[Wm:]]
    total_ms, e2e_total = job_times(sum(step_ms), sum(a.elapsed_time(b) for a, b in e2e_ev[Wm:]), world,
                                    device="cuda")
    ms_per_step = total_ms / K
    value = job_throughput(world, flops, ms_per_step)
    e2e_ms = e2e_total / K
    e2e_value = job_throughput(world, flops, e2e_ms)

    graph_line = None
    if graph is not None:
        g_ms = [a.elapsed_time(b) for a, b in g_ev]
        g_total, _ = job_times(sum(g_ms), 0.0, world, device="cuda")
        graph_line = {"ms_per_step": g_total / K, "median_ms_per_step": statistics.median(g_ms),
                      "value": job_throughput(world, flops, g_total / K), "unit": "TFLOP/s",
                      "note": "the mha_forward call captured once in a CUDA graph, replayed; L2 flushed between replays"}
    core = r.core_record(att_ms, peaks)

    # ---- roofline of the dominant kernel (largest share of the step)
    shares = {"qkv_projection_gemm": statistics.mean(q_ms), "attention_core": statistics.mean(att_ms),
              "output_projection_gemm": statistics.mean(out_ms)}
    dom = max(shares, key=shares.get)
    dom_flops = {"qkv_projection_gemm": 0.75 * proj, "attention_core": attn, "output_projection_gemm": 0.25 * proj}
    achieved = dom_flops[dom] / (shares[dom] * 1e-3) / 1e12
    peak = float(peaks["bf16_tflops"])
    clocks = clk.summary()
    traffic = committed_traffic(dom, args.workload)
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": K, "warmup": Wm,
        "ms_per_step": ms_per_step, "median_ms_per_step": statistics.median(step_ms),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded N(0,1) activations, Xavier-uniform weights)",
        "config": {"workload": DESCRIPTION[args.workload],
                   "B_per_gpu": Bn, "global_batch": Bn * world, "seq_len": Lq, "d_model": d, "h": h,
                   "mask": ("causal" if wl.causal else "") + (" key padding" if r.vl is not None else ""),
                   "parallelism": f"dp{world} (batch sharded, no collective)",
                   "step": "one mha_forward call (the three kernels back to back)",
                   "l2": "flushed before every step (256 MB write outside the timed events)"},
        "tokens_per_s": world * Bn * Lq / (ms_per_step * 1e-3),
        "pct_of_bf16_peak": 100.0 * value / peak,
        "stage_ms": {k2: round(v2, 4) for k2, v2 in shares.items()},
        "stage_note": f"{stage_steps} steps of the three stage entry points with CUDA events between them",
        "attention_core": core,
        "graph": graph_line,
        "roofline": {"kernel": dom, "source_sha1": source_digest(dom, args.workload), "bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "peak_source": f"{peak_src} bf16_tflops (burst); sustained {peaks.get('bf16_tflops_sustained')}"},
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "api": "mha_forward_host (pinned host query in, out back)"},
        "per_workload": per_wl,
        "gpu_launches": launches,
        "clocks": clocks,
        "cpu_baseline": cpu,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_gpu_pattn(args):
    """The optional attention weights (p_attn, fp32 [B, h, L_q, L_k]): the attention stage timed
    with and without them on the same workload. The difference is the p_attn pass (the scores
    recomputed from Qh, Kh and the row statistics, normalised and written); HBM-write bound, so
    it is reported as GB/s of the fp32 weights written against the measured copy bandwidth."""
    import torch

    from transformer_head_scaled_fwd_gb300 import binding
    from transformer_head_scaled_fwd_gb300 import build as B

    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    B.build()
    binding.load()
    peaks, peak_src = load_peaks()
    r = WorkloadRun(args.workload, rank, local)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    p_attn = torch.empty(r.B, r.h, r.Lq, r.Lk, dtype=torch.float32, device="cuda")
    K, Wm = args.steps, args.warmup
    binding.mha_qkv_projection(r.q, r.k, r.v, r.Wt["w_q"], r.Wt["b_q"], r.Wt["w_k"], r.Wt["b_k"], r.Wt["w_v"],
                               r.Wt["b_v"], r.h, workspace=r.ws, stream=stream)

    def attn_ms(with_p):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K + Wm)]
        for s_ in range(Wm + K):
            flush.zero_()
            ev[s_][0].record(stream)
            binding.mha_attention_core(r.dt, r.B, r.Lq, r.Lk, r.d, r.h, workspace=r.ws, mask=r.mask,
                                       p_attn=p_attn if with_p else None, stream=stream)
            ev[s_][1].record(stream)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in ev[Wm:]]

    with ClockSampler(local) as clk:
        torch.cuda.synchronize()
        without = attn_ms(False)
        with_p = attn_ms(True)
    if binding.mha_check_device_status(reset=True) != 0:
        raise RuntimeError("a pipeline wait gave up inside a kernel")
    rows = p_attn.sum(-1)
    rowsum_err = float((rows - 1.0).abs().max().item())
    ms = statistics.mean(with_p) - statistics.mean(without)
    nbytes = p_attn.numel() * 4
    gbs = nbytes / (ms * 1e-3) / 1e9
    peak = float(peaks["hbm_gbs"])
    line = {
        "metric": "MHA p_attn pass GB/s (fp32 weights written)", "value": gbs, "unit": "GB/s", "n_gpus": 1,
        "steps": K, "warmup": Wm, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded)",
        "config": {"workload": DESCRIPTION[args.workload] + ", with p_attn", "l2": "flushed before every step"},
        "attention_ms": {"without_p_attn": statistics.mean(without), "with_p_attn": statistics.mean(with_p)},
        "p_attn_bytes": nbytes, "p_attn_row_sum_max_err": rowsum_err,
        "roofline": {"kernel": "pattn_bf16_kernel", "bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s",
                     "frac": gbs / peak, "traffic": None, "peak_source": f"{peak_src} hbm_gbs"},
        "gpu_launches": 3 * (K + Wm) + 2, "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)


def run_gpu_ffn(args):
    """Position-wise FFN (max(0, x W_1 + b_1) W_2 + b_2) on one GPU: TFLOP/s of the two GEMMs."""
    import torch

    from transformer_head_scaled_fwd_gb300 import binding
    from transformer_head_scaled_fwd_gb300 import build as B
    from transformer_head_scaled_fwd_gb300 import workloads as W

    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    B.build()
    binding.load()
    peaks, peak_src = load_peaks()
    cfg = W.FFN_WORKLOADS[args.ffn_workload]
    inp = W.make_ffn_inputs(cfg["B"], cfg["L"], cfg["d_model"], cfg["d_ff"], seed=rank)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda().to(torch.bfloat16)
    x, w1, b1, w2, b2 = dev(inp.x), dev(inp.w_1), dev(inp.b_1), dev(inp.w_2), dev(inp.b_2)
    Bn, L, d = x.shape
    d_ff = w1.shape[0]
    ws = torch.empty(binding.ffn_workspace_size(binding.MHA_BF16, Bn, L, d, d_ff), dtype=torch.uint8,
                     device="cuda")
    out = torch.empty_like(x)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    flops = 4.0 * Bn * L * d * d_ff
    K, Wm = args.steps, args.warmup
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K + Wm)]
    with ClockSampler(local) as clk:
        torch.cuda.synchronize()
        for s_ in range(Wm + K):
            flush.zero_()
            evs[s_][0].record(stream)
            binding.mha_ffn_forward(x, w1, b1, w2, b2, out=out, workspace=ws, stream=stream)
            evs[s_][1].record(stream)
        torch.cuda.synchronize()
    if binding.mha_check_device_status(reset=True) != 0:
        raise RuntimeError("a pipeline wait gave up inside a kernel")
    ms = sum(a.elapsed_time(b) for a, b in evs[Wm:]) / K
    value = flops / (ms * 1e-3) / 1e12
    peak = float(peaks["bf16_tflops"])
    line = {
        "metric": "FFN fwd TFLOP/s (bf16)", "value": value, "unit": "TFLOP/s", "n_gpus": 1, "steps": K,
        "warmup": Wm, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded N(0,1) activations, Xavier-uniform weights)",
        "config": {"workload": f"position-wise FFN B{Bn} L{L} d_model{d} d_ff{d_ff}", "tokens": Bn * L,
                   "l2": "flushed before every step"},
        "tokens_per_s": Bn * L / (ms * 1e-3),
        "roofline": {"kernel": "gemm_bf16_tc (2 launches)", "bound": "tensor", "achieved": value, "peak": peak,
                     "unit": "TFLOP/s", "frac": value / peak, "traffic": None,
                     "peak_source": f"{peak_src} bf16_tflops (burst)"},
        "gpu_launches": 2 * K, "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)


def run_gpu_sublayer(args):
    """Pre-norm residual sublayer x + MHA(LayerNorm(x)) on the long workload: TFLOP/s counts the
    attention sublayer's algorithmic flops (LayerNorm and the residual add are HBM-bound extras)."""
    import torch

    from transformer_head_scaled_fwd_gb300 import binding
    from transformer_head_scaled_fwd_gb300 import build as B
    from transformer_head_scaled_fwd_gb300 import workloads as W

    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    B.build()
    binding.load()
    peaks, peak_src = load_peaks()
    wl = W.WORKLOADS[args.workload]
    inp = rank_inputs(wl, rank)
    ln = W.make_ln_params(wl.d_model, seed=rank)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda().to(torch.bfloat16)
    x = dev(inp.query)
    Wt = [dev(inp.weights[n]) for n in ("w_q", "b_q", "w_k", "b_k", "w_v", "b_v", "w_o", "b_o")]
    g, bb = dev(ln[0]), dev(ln[1])
    Bn, L, d = x.shape
    vl = None if inp.valid_lens is None else torch.from_numpy(inp.valid_lens).cuda()
    mask = binding.make_mask(wl.causal, vl, None)
    ws = torch.empty(binding.sublayer_workspace_size(binding.MHA_BF16, Bn, L, 0, d, wl.h), dtype=torch.uint8,
                     device="cuda")
    out = torch.empty_like(x)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    proj, attn = algorithmic_flops(Bn, L, L, d, wl.h, wl.causal, inp.valid_lens)
    K, Wm = args.steps, args.warmup
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K + Wm)]
    with ClockSampler(local) as clk:
        torch.cuda.synchronize()
        for s_ in range(Wm + K):
            flush.zero_()
            evs[s_][0].record(stream)
            binding.mha_sublayer_forward(x, g, bb, 1e-6, 0, *Wt, wl.h, out=out, workspace=ws, mask=mask,
                                         stream=stream)
            evs[s_][1].record(stream)
        torch.cuda.synchronize()
    if binding.mha_check_device_status(reset=True) != 0:
        raise RuntimeError("a pipeline wait gave up inside a kernel")
    ms = sum(a.elapsed_time(b) for a, b in evs[Wm:]) / K
    value = (proj + attn) / (ms * 1e-3) / 1e12
    peak = float(peaks["bf16_tflops"])
    line = {
        "metric": "pre-norm residual MHA sublayer fwd TFLOP/s (bf16)", "value": value, "unit": "TFLOP/s",
        "n_gpus": 1, "steps": K, "warmup": Wm, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded)",
        "config": {"workload": "x + MHA(LayerNorm(x)): " + DESCRIPTION[args.workload],
                   "layernorm": "unbiased std + eps 1e-6", "l2": "flushed before every step"},
        "tokens_per_s": Bn * L / (ms * 1e-3), "pct_of_bf16_peak": 100 * value / peak,
        "gpu_launches": 4 * K, "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)


def run_gpu_decode(args):
    """Incremental decoding: one new token per sequence against an 8192-token key/value cache.
    HBM-bound: reports decoded tokens/s and the achieved GB/s of algorithmic bytes (cache read once,
    weights read once, new k/v written) against the measured copy bandwidth."""
    import torch

    from transformer_head_scaled_fwd_gb300 import binding
    from transformer_head_scaled_fwd_gb300 import build as B
    from transformer_head_scaled_fwd_gb300 import workloads as W

    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    B.build()
    binding.load()
    peaks, peak_src = load_peaks()
    Bn, d, h, P = args.decode_batch, 1024, args.decode_heads, args.decode_context
    dk = d // h
    K, Wm = args.steps, args.warmup
    L_max = P + 2 * (K + Wm) + 8   # room for the direct loop and the graph replays
    inp = W.random_case(500 + rank, Bn, P + 1, P + 1, d, h, self_attn=True, bias_scale=0.0)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda().to(torch.bfloat16)
    w = [dev(inp.weights[n]) for n in ("w_q", "b_q", "w_k", "b_k", "w_v", "b_v", "w_o", "b_o")]
    kc = torch.zeros(Bn, h, L_max, dk, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    binding.mha_kv_cache_prefill(dev(inp.query[:, :P]), w[2], w[3], w[4], w[5], h, k_cache=kc, v_cache=vc)
    clen = torch.full((Bn,), P, dtype=torch.int32, device="cuda")
    ws = torch.empty(binding.decode_workspace_size(Bn, d, h, L_max), dtype=torch.uint8, device="cuda")
    x_new = dev(inp.query[:, P])
    out = torch.empty(Bn, d, dtype=torch.bfloat16, device="cuda")
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K + Wm)]
    with ClockSampler(local) as clk:
        torch.cuda.synchronize()
        for s_ in range(Wm + K):
            flush.zero_()
            evs[s_][0].record(stream)
            binding.mha_decode_step(x_new, *w, h, k_cache=kc, v_cache=vc, cache_len=clen, out=out, workspace=ws,
                                    stream=stream)
            evs[s_][1].record(stream)
        torch.cuda.synchronize()
        # the same step captured once in a CUDA graph and replayed (cache_len lives on the
        # device, so every replay appends the next token); L2 flushed between replays
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            binding.mha_decode_step(x_new, *w, h, k_cache=kc, v_cache=vc, cache_len=clen, out=out, workspace=ws,
                                    stream=torch.cuda.current_stream())
        g_evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K + Wm)]
        for s_ in range(Wm + K):
            flush.zero_()
            g_evs[s_][0].record(stream)
            graph.replay()
            g_evs[s_][1].record(stream)
        torch.cuda.synchronize()
    if binding.mha_check_device_status(reset=True) != 0:
        raise RuntimeError("a kernel reported an error")
    ms = sum(a.elapsed_time(b) for a, b in evs[Wm:]) / K
    g_ms = sum(a.elapsed_time(b) for a, b in g_evs[Wm:]) / K
    mean_ctx = P + Wm + (K + 1) / 2.0          # cached tokens attended per step, on average
    cache_bytes = Bn * h * mean_ctx * dk * 2 * 2
    bytes_step = cache_bytes + 4 * d * d * 2 + 4 * Bn * d * 2 + Bn * h * dk * 2 * 2
    gbs = bytes_step / (ms * 1e-3) / 1e9
    peak = float(peaks["hbm_gbs"])
    line = {
        "metric": "MHA incremental decode tokens/s (bf16, KV cache)", "value": Bn / (ms * 1e-3),
        "unit": "tokens/s", "n_gpus": 1, "steps": K, "warmup": Wm, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded)",
        "config": {"workload": f"decode step B{Bn} d_model{d} h{h} d_k{dk}, cache ~{P} tokens",
                   "l2": "flushed before every step"},
        "roofline": {"kernel": "decode step (projection GEMMs + split-K cache attention)", "bound": "hbm",
                     "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak, "traffic": None,
                     "algorithmic_bytes_per_step": bytes_step, "peak_source": f"{peak_src} hbm_gbs"},
        "graph": {"ms_per_step": g_ms, "value": Bn / (g_ms * 1e-3), "unit": "tokens/s",
                  "note": "the step captured once in a CUDA graph, replayed; L2 flushed between replays"},
        "gpu_launches": 8 * K, "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--workload", default=WORKLOAD, choices=["enc", "dec", "xattn", "long", "long_d128"])
    ap.add_argument("--ref-prefix", type=int, default=2048, help="causal prefix length of the oracle sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="skip the CUDA graph replay variant")
    ap.add_argument("--no-per-workload", action="store_true",
                    help="skip the short records of the other workloads in the JSON line")
    ap.add_argument("--decode-batch", type=int, default=16)
    ap.add_argument("--decode-context", type=int, default=8192)
    ap.add_argument("--decode-heads", type=int, default=16, help="heads at d_model 1024 (16: d_k 64, 8: d_k 128)")
    ap.add_argument("--path", choices=["mha", "ffn", "sublayer", "decode", "pattn"], default="mha",
                    help="mha: the attention sublayer (default); ffn: the position-wise FFN; "
                         "sublayer: x + MHA(LayerNorm(x)); decode: one token per sequence vs a KV cache; "
                         "pattn: the attention stage with and without the p_attn weights")
    ap.add_argument("--ffn-workload", default="ffn_long", choices=["ffn_base", "ffn_long"])
    args = ap.parse_args()
    if args.warmup < 3 and args.impl != "reference":
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.path == "ffn":
        run_gpu_ffn(args)
    elif args.path == "sublayer":
        run_gpu_sublayer(args)
    elif args.path == "decode":
        run_gpu_decode(args)
    elif args.path == "pattn":
        run_gpu_pattn(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
