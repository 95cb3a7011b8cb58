#!/usr/bin/env python3
"""Benchmark of one block-diffusion denoising round on GB300 (sm_103a), through libbdlm.

Workload (the metric's configuration): batch 128, block length 4, SDAR-4B-shaped attention
(32 query / 8 KV heads, head dim 128, bf16) with prefixes uniform in [512, 4096] in a
shuffled 140 000-page pool of 16-token pages; half of every block masked; threshold 0.75,
T = 1; the selective LM head at the SDAR-4B shape (hidden 2560, W 151936x2560 bf16).

One step = one denoising round of that batch, every step of the hot path on the device:
block attention -> selective LM head on the still-masked rows -> confidence/commit over
those logits -> mask update.  value = block positions (B*L) per second.  The JSON line also
carries config 2 exactly as printed (the commit over the supplied logits, no LM head),
per-kernel times and rooflines, the end-to-end figure through host buffers and the fp64 CPU
oracle timed on the host cores.

    python bench.py [--gpus N --steps K --warmup W] [--impl reference] [--quick]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads as W  # noqa: E402

METRIC = "denoised block-positions/s per round (B=128, SDAR-4B shape); % HBM roofline"
UNIT = "block-positions/s"
WORKLOAD = ("config2: B=128 L=4 Hq=32 Hkv=8 D=128 bf16, prefix U[512,4096], page 16, "
            "shuffled 140000-page pool, mask 1/2 per block, tau=0.75 T=1; LM head H=2560 "
            "V=151936 on the 256 masked rows (hidden N(0,1), W N(0,0.02^2)) fused with the "
            "confidence/commit")
L2_BYTES = 129 * 1024 * 1024


# --------------------------------------------------------------------------- helpers
def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--seed", type=int, default=W.seed_for(2))
    ap.add_argument("--quick", action="store_true",
                    help="skip the end-to-end and CPU-baseline legs (profiling runs)")
    ap.add_argument("--eager", action="store_true",
                    help="time eager launches instead of one CUDA graph per round")
    ap.add_argument("--compact-pool", action="store_true",
                    help="pool of exactly the referenced pages x1.25 (smaller device footprint)")
    ap.add_argument("--attention-shapes", action="store_true",
                    help="time the block attention alone at the config 2-4 shapes and exit")
    ap.add_argument("--shape", choices=["c2", "c3_L16", "c3_L32", "c4"], default=None,
                    help="with --attention-shapes: only this shape")
    return ap.parse_args(argv)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def rank_seed(seed: int, rank: int) -> int:
    """Each rank denoises its own batch: a distinct, reproducible seed per rank."""
    return seed + 7919 * rank


def max_over_ranks(x: float, world: int) -> float:
    """Largest value of `x` over all ranks (the slowest rank sets the job's time)."""
    if world == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    dev = (torch.device("cuda", torch.cuda.current_device())
           if dist.get_backend() == "nccl" else torch.device("cpu"))
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(units_per_rank: int, world: int, ms_max: float) -> float:
    """Whole-job throughput: the units every rank processed over the slowest rank's time."""
    return units_per_rank * world / (ms_max / 1e3)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def source_digest(srcs) -> str:
    """sha256 over the concatenated bytes of a kernel's source files (under csrc/, in order)."""
    h = hashlib.sha256()
    for s in srcs:
        h.update(open(os.path.join(ROOT, "block_diffusion_gb300", "csrc", s), "rb").read())
    return h.hexdigest()


def profile_traffic(name: str, srcs):
    """DRAM bytes per launch from the committed ncu summary of kernel `name`, or None when
    the kernel's sources changed since the capture (the summary records their sha256)."""
    path = os.path.join(ROOT, "profiles", f"{name}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    digest = source_digest(srcs)
    rec = {}
    for line in text.splitlines():
        line = line.strip().lstrip("-* ")
        if ":" in line and line.startswith(("source_sha256", "traffic_bytes_per_launch")):
            k, v = line.split(":", 1)
            v = v.strip()
            rec[k.strip()] = v.split("`")[1] if v.startswith("`") else v
    if rec.get("source_sha256") != digest:
        return None
    try:
        return float(rec["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[4:]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in rows:
            for n, v in zip(names, r[3][1:]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(r[0] for r in rows),
                "sm_max_mhz": max(r[1] for r in rows),
                "power_w_max": max(r[2] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows)}


# --------------------------------------------------------------------------- workload
H_LM = 2560          # SDAR-4B hidden size
REF_SEQS = 16        # sequences per step of the CPU oracle's bounded sample
REF_SEQS_1CORE = 2   # sequences of the one-core oracle sample


def make_workload(seed: int, compact_pool: bool = False):
    """Config-2 attention and commit inputs, plus the LM head's hidden rows and weights
    (SDAR-4B hidden size, W N(0, 0.02^2)) for the rows still masked."""
    c = W.CONFIGS[2]
    rng = np.random.default_rng(seed)
    a = W.make_attention(rng, c["B"], c["L"], c["Hq"], c["Hkv"], c["D"],
                         prefix_range=c["prefix"],
                         pool_pages=None if compact_pool else c["pool_pages"], poison=False)
    ci = W.commit_inputs(2, rng, c["B"], c["L"], c["V"], poison=False)
    act = np.nonzero(ci.mask.reshape(-1))[0].astype(np.int32)
    lm = W.lm_head_inputs(np.random.default_rng(seed + 1), a.B * a.L, H_LM, ci.V, act)
    return c, a, ci, lm


def algorithmic(a, ci, lm):
    """Bytes (and flops) each step must move: every K/V element once per KV head (exact
    token count), Q in and O out; W once, the active hidden rows in and their logits out;
    the masked logits rows once."""
    kv_tokens = int(a.kv_lens.sum())
    n_act = len(lm.active_idx)
    return {
        "attention": (kv_tokens * a.Hkv * a.D * 2 * 2 + a.B * a.L * a.Hq * a.D * 2 * 2,
                      4 * a.L * a.Hq * a.D * kv_tokens),
        "lm_head": (ci.V * lm.H * 2 + n_act * lm.H * 2 + n_act * ci.V * 2,
                    2 * n_act * lm.H * ci.V),
        "commit": (int(ci.mask.sum()) * ci.V * 2, 0),
        # fused LM head + confidence: W once and the scored rows in; the logits never leave
        # the SMs (tok/conf/commit out are a few KB)
        "lm_head_commit": (ci.V * lm.H * 2 + n_act * lm.H * 2, 2 * n_act * lm.H * ci.V),
    }


class Round:
    """Device-resident inputs and the launch sequence of one round.  Modes:
    fused     attention -> LM head fused with confidence/commit -> mask update (the headline);
    unfused   attention -> LM head (logits to HBM) -> confidence/commit -> mask update;
    supplied  attention -> confidence/commit over the supplied logits -> mask update."""

    STAGES = {"fused": ("attention", "lm_head_commit", "mask_update"),
              "unfused": ("attention", "lm_head", "commit", "mask_update"),
              "supplied": ("attention", "commit", "mask_update")}
    # attention + split merge; [scored rows + fused GEMM + finalize | row gather + LM head];
    # commit (one launch); mask update
    LAUNCHES = {"fused": 2 + 3 + 1, "unfused": 2 + 2 + 1 + 1, "supplied": 2 + 1 + 1}

    def __init__(self, lib, a, ci, lm, device, mode="fused"):
        import torch
        self.torch = torch
        self.lib = lib
        self.mode = mode
        self.a, self.ci = a, ci
        self.B, self.L, self.V = a.B, a.L, ci.V
        shape = (a.pool_pages, a.P, a.Hkv, a.D)
        self.kp = torch.zeros(shape, dtype=torch.bfloat16, device=device)
        self.vp = torch.zeros(shape, dtype=torch.bfloat16, device=device)
        ids = torch.from_numpy(a.ref_page_ids.astype(np.int64)).to(device)
        self.kp[ids] = _bf16(a.k_ref, device)
        self.vp[ids] = _bf16(a.v_ref, device)
        self.q = _bf16(a.q, device)
        self.pt = torch.from_numpy(a.page_table).to(device)
        self.pl = torch.from_numpy(a.prefix_lens).to(device)
        self.out = torch.empty((a.B, a.L, a.Hq, a.D), dtype=torch.bfloat16, device=device)
        if mode == "fused":
            self.logits = None
        elif mode == "supplied":
            self.logits = _bf16(ci.logits.reshape(a.B * a.L, ci.V), device)
        else:
            self.logits = torch.empty((a.B * a.L, ci.V), dtype=torch.bfloat16, device=device)
        self.mask0 = torch.from_numpy(ci.mask).to(device)
        self.mask = self.mask0.clone()
        self.tok = torch.empty((a.B, a.L), dtype=torch.int32, device=device)
        self.conf = torch.empty((a.B, a.L), dtype=torch.float32, device=device)
        self.commit = torch.empty((a.B, a.L), dtype=torch.uint8, device=device)
        self.desc = lib.attn_desc(a.B, a.L, a.Hq, a.Hkv, a.D, a.page_table.shape[1],
                                  a.pool_pages)
        self.n_act = 0
        if mode != "supplied":
            self.H = lm.H
            self.hidden = _bf16(lm.hidden, device)
            self.w = _bf16(lm.w, device)
            self.act = torch.from_numpy(lm.active_idx).to(device)
            self.n_act = len(lm.active_idx)

    def stages(self):
        return self.STAGES[self.mode]

    def launches_per_step(self):
        return self.LAUNCHES[self.mode]

    def step(self, stream, events=None):
        """Enqueue one round on `stream`; events (list) get a record before the first stage
        and after each stage."""
        lib, s = self.lib, stream.cuda_stream
        k = 0

        def mark():
            nonlocal k
            if events is not None:
                events[k].record(stream)
            k += 1

        mark()
        lib.bdlm_block_attention(self.desc, self.q, self.kp, self.vp, self.pt, self.pl, self.L,
                                 self.out, s)
        mark()
        if self.mode == "fused":
            lib.bdlm_lm_head_commit(self.hidden, self.w, self.mask, None, self.B, self.L,
                                    self.H, self.V, lib.BDLM_COMMIT_THRESHOLD, 1,
                                    self.ci.threshold, self.ci.temperature, self.tok, self.conf,
                                    self.commit, None, s)
            mark()
        else:
            if self.mode == "unfused":
                lib.bdlm_lm_head(self.hidden, self.w, self.act, self.n_act, self.B * self.L,
                                 self.H, self.V, self.logits, s)
                mark()
            lib.bdlm_confidence_commit(self.logits, self.mask, self.B, self.L, self.V,
                                       self.ci.threshold, self.ci.temperature, self.tok,
                                       self.conf, self.commit, s)
            mark()
        lib.bdlm_apply_commit(self.mask, self.commit, self.B * self.L, s)
        mark()

    def reset_mask(self, stream):
        with self.torch.cuda.stream(stream):
            self.mask.copy_(self.mask0)


def _bf16(bits, device):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16))
    return t.to(device).view(torch.bfloat16)


def time_round(rnd: Round, stream, steps: int, warmup: int, flush, barrier):
    """Per-step CUDA-event times (ms) of the whole round and of each stage; L2 flushed
    before every step, outside the timed events."""
    torch = rnd.torch
    for _ in range(warmup):
        rnd.reset_mask(stream)
        flush(stream)
        rnd.step(stream)
    torch.cuda.synchronize()
    ns = len(rnd.stages())
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(ns + 1)] for _ in range(steps)]
    barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for k in range(steps):
        rnd.reset_mask(stream)
        flush(stream)
        rnd.step(stream, evs[k])
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    barrier()
    stage = np.array([[evs[k][i].elapsed_time(evs[k][i + 1]) for i in range(ns)]
                      for k in range(steps)])
    total = np.array([evs[k][0].elapsed_time(evs[k][ns]) for k in range(steps)])
    return total, stage, wall


def time_round_graph(rnd: Round, stream, steps: int, warmup: int, flush, barrier,
                     sustain_s: float = 0.0, gpu_index: int = 0):
    """Per-step times (ms) of the round replayed as one CUDA graph (captured once, after the
    eager warm-up has sized the library's workspace); L2 flushed before every replay.  With
    sustain_s > 0 the graph is then replayed for about that long under its own clock sampler
    (the `sustained` record: mean per-step time and the clocks seen)."""
    torch = rnd.torch
    for _ in range(warmup):
        rnd.reset_mask(stream)
        flush(stream)
        rnd.step(stream)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        rnd.step(stream)
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for k in range(steps):
            rnd.reset_mask(stream)
            flush(stream)
            evs[k][0].record(stream)
            graph.replay()
            evs[k][1].record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    barrier()
    times = np.array([a.elapsed_time(b) for a, b in evs])
    if sustain_s <= 0:
        return times, wall
    n = max(1, int(sustain_s / (float(times.mean()) * 2e-3)))   # a step + its flush ~ 2 steps
    sampler = ClockSampler(gpu_index)
    sampler.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev_steps = []
    with torch.cuda.stream(stream):
        e0.record(stream)
        for k in range(n):
            rnd.reset_mask(stream)
            flush(stream)
            a_ev, b_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a_ev.record(stream)
            graph.replay()
            b_ev.record(stream)
            ev_steps.append((a_ev, b_ev))
        e1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    sus = {"steps": n, "ms_per_step": float(np.mean([a.elapsed_time(b) for a, b in ev_steps])),
           "region_s": e0.elapsed_time(e1) / 1e3, "clocks": clocks,
           "note": "the same graph replayed back to back (L2 flushed before each replay) for "
                   "about a second and a half, so that the clock record has samples under load"}
    return times, wall, sus


def e2e_round(lib, a, ci, lm, device, steps, warmup, seed):
    """The round through the C-ABI from pinned host buffers.  The paged K/V cache and W are
    resident device state (the cache holds every sequence's prefix); every step copies its own
    inputs host->device (q, the block's new K/V, the hidden rows, the mask), runs the attention
    with the block's K/V-cache write fused in, the LM head fused with confidence/commit and the
    mask update, and copies tok/conf/commit back.  As in a serving loop, the inputs are
    double-buffered on the device and step k+1's host->device copies run on a copy stream while
    step k computes (events order each buffer's copy after the step that last read it)."""
    import torch
    stream = torch.cuda.Stream(device=device)
    copy_stream = torch.cuda.Stream(device=device)
    rng = np.random.default_rng(seed)
    B, L = a.B, a.L
    k_new = W._normal_bf16(rng, (B, L, a.Hkv, a.D), 0.5)
    v_new = W._normal_bf16(rng, (B, L, a.Hkv, a.D), 0.5)
    h = {
        "q": torch.from_numpy(a.q.view(np.int16)).pin_memory(),
        "kn": torch.from_numpy(k_new.view(np.int16)).pin_memory(),
        "vn": torch.from_numpy(v_new.view(np.int16)).pin_memory(),
        "hid": torch.from_numpy(lm.hidden.view(np.int16)).pin_memory(),
        "mk": torch.from_numpy(ci.mask).pin_memory(),
    }
    dbuf = [{k: torch.empty_like(v, device=device) for k, v in h.items()} for _ in range(2)]
    copied = [torch.cuda.Event(), torch.cuda.Event()]   # buffer i holds its step's inputs
    used = [None, None]                                 # the step that last read buffer i
    kp, vp = _bf16(a.k_ref, device), _bf16(a.v_ref, device)      # resident cache
    pt = torch.from_numpy(a.page_table_ref).to(device)
    pl = torch.from_numpy(a.prefix_lens).to(device)
    w = _bf16(lm.w, device)                                       # resident weights
    outs_h = {"tok": torch.empty((B, L), dtype=torch.int32).pin_memory(),
              "conf": torch.empty((B, L), dtype=torch.float32).pin_memory(),
              "com": torch.empty((B, L), dtype=torch.uint8).pin_memory()}
    outs_d = {k: torch.empty_like(v, device=device) for k, v in outs_h.items()}
    out = torch.empty((B, L, a.Hq, a.D), dtype=torch.bfloat16, device=device)
    desc = lib.attn_desc(B, L, a.Hq, a.Hkv, a.D, a.page_table_ref.shape[1], a.k_ref.shape[0])
    h2d = sum(v.numel() * v.element_size() for v in h.values())
    d2h = sum(v.numel() * v.element_size() for v in outs_h.values())

    def upload(i):
        if used[i] is not None:
            copy_stream.wait_event(used[i])
        with torch.cuda.stream(copy_stream):
            for k in h:
                dbuf[i][k].copy_(h[k], non_blocking=True)
        copied[i].record(copy_stream)

    def compute(i):
        d = dbuf[i]
        s = stream.cuda_stream
        stream.wait_event(copied[i])
        with torch.cuda.stream(stream):
            bf = torch.bfloat16
            lib.bdlm_block_attention_kv(desc, d["q"].view(bf), d["kn"].view(bf), d["vn"].view(bf),
                                        kp, vp, pt, pl, L, out, s)
            lib.bdlm_lm_head_commit(d["hid"].view(bf), w, d["mk"], None, B, L, lm.H, ci.V,
                                    lib.BDLM_COMMIT_THRESHOLD, 1, ci.threshold, ci.temperature,
                                    outs_d["tok"], outs_d["conf"], outs_d["com"], None, s)
            lib.bdlm_apply_commit(d["mk"], outs_d["com"], B * L, s)
            ev = torch.cuda.Event()
            ev.record(stream)
            used[i] = ev
            for k in outs_h:
                outs_h[k].copy_(outs_d[k], non_blocking=True)

    def run(n):
        upload(0)
        for t in range(n):
            if t + 1 < n:
                upload((t + 1) % 2)
            compute(t % 2)

    run(warmup)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    copy_stream.wait_event(e0)   # the first step's copies start inside the timed region
    run(steps)
    e1.record(stream)            # after the last step's compute and its device->host read
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    del w, kp, vp
    return ms, h2d, d2h


# --------------------------------------------------------------------------- CPU oracle
def cpu_oracle_round(a, ci, lm, seqs):
    """The round of the listed sequences by the fp64 oracle: attention, LM head on their
    masked rows (rounded once to bf16), confidence and commit."""
    import oracle
    oracle.block_attention(a.q, a.k_ref, a.v_ref, a.page_table_ref, a.prefix_lens, a.L, a.Hq,
                           a.Hkv, a.D, a.P, seqs=seqs)
    mask = ci.mask[seqs]
    sel = mask.astype(bool)
    rows = (seqs[:, None] * a.L + np.arange(a.L)[None, :])[sel].astype(np.int32)
    local = (np.arange(len(seqs))[:, None] * a.L + np.arange(a.L)[None, :])[sel]
    logits = np.zeros((len(seqs) * a.L, ci.V), dtype=np.uint16)
    logits[local] = oracle.round_logits_to_bf16(oracle.lm_head(lm.hidden, lm.w, rows))
    oracle.confidence_commit(logits, mask, ci.threshold, ci.temperature)


def cpu_baseline(a, ci, lm, min_seconds=10.0):
    """The fp64 oracle as it stands on the host cores, on a bounded sample: the round of
    REF_SEQS sequences, repeated until at least `min_seconds` of work."""
    import oracle
    oracle.build()
    seqs = np.arange(REF_SEQS, dtype=np.int32)
    reps, t0 = 0, time.perf_counter()
    while True:
        cpu_oracle_round(a, ci, lm, seqs)
        reps += 1
        el = time.perf_counter() - t0
        if el >= min_seconds:
            break
    per = el / reps
    cores = oracle.num_threads()
    # the same oracle on one core, over a smaller sample
    one = np.arange(REF_SEQS_1CORE, dtype=np.int32)
    oracle.set_num_threads(1)
    try:
        t1 = time.perf_counter()
        cpu_oracle_round(a, ci, lm, one)
        el1 = time.perf_counter() - t1
    finally:
        oracle.set_num_threads(cores)
    return {"value": len(seqs) * a.L / per, "unit": UNIT, "cores": cores,
            "kind": "oracle",
            "sample": f"{reps} x the round of {REF_SEQS} of the 128 config-2 sequences "
                      f"(attention, LM head on their masked rows, commit), fp64 C++ OpenMP, "
                      f"{per:.2f} s each",
            "value_1core": len(one) * a.L / el1,
            "sample_1core": f"the round of {REF_SEQS_1CORE} sequences on one thread, {el1:.2f} s"}


def line_config(world: int, n_act: int, seed: int) -> dict:
    """The `config` object of the JSON line; the same for both arms."""
    return {"workload": WORKLOAD, "global_batch": 128 * world, "block_len": 4,
            "lm_head_rows": int(n_act), "hidden": H_LM,
            "l2": "flushed before every step (256 MB fill, outside the timed events)",
            "parallelism": f"dp{world} (independent batches, no collective)", "seed": seed}


# --------------------------------------------------------------------------- arms
def run_reference(args, rank, world):
    """The oracle as the reference arm: rank 0 times it on the host cores; others exit."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    c, a, ci, lm = make_workload(args.seed, compact_pool=True)
    seqs = np.arange(REF_SEQS, dtype=np.int32)   # bounded sample per step
    for _ in range(max(0, min(args.warmup, 3))):
        cpu_oracle_round(a, ci, lm, seqs)
    steps = max(1, min(args.steps, 20))
    t0 = time.perf_counter()
    for _ in range(steps):
        cpu_oracle_round(a, ci, lm, seqs)
    el = (time.perf_counter() - t0) / steps
    value = len(seqs) * a.L / el
    sample = (f"the round of {REF_SEQS} of the 128 sequences per step (attention, LM head on "
              f"their masked rows, commit)")
    line = {"metric": METRIC, "value": value, "unit": UNIT, "impl": "reference",
            "n_gpus": args.gpus, "steps": steps, "warmup": args.warmup,
            "ms_per_step": el * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": line_config(world, len(lm.active_idx), args.seed),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.num_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


def chain_config5(bd, device, flush, reps: int, seed: int):
    """Config 5's whole block on the device: the round loop (one CUDA graph with a WHILE node)
    over 4 steps of fresh Q, block K/V and hidden (B=128, L=4, SDAR-8B LM head, W N(0,0.02^2),
    prefixes U[256, 4096], every position masked, threshold 0.75), L2 flushed before each
    launch.  Returns the figures of one block."""
    import torch
    c = W.CONFIGS[5]
    B, L, Hq, Hkv, D, H, V, S = (c["B"], c["L"], c["Hq"], c["Hkv"], c["D"], c["H"], c["V"],
                                 c["steps"])
    rng = np.random.default_rng(seed)
    a = W.make_attention(rng, B, L, Hq, Hkv, D, prefix_range=c["prefix"], poison=False)
    kp, vp = _bf16(a.k_ref, device), _bf16(a.v_ref, device)
    pt = torch.from_numpy(a.page_table_ref).to(device)
    pl = torch.from_numpy(a.prefix_lens).to(device)
    q = _bf16(W._normal_bf16(rng, (S, B, L, Hq, D), 0.5), device)
    kn = _bf16(W._normal_bf16(rng, (S, B, L, Hkv, D), 0.5), device)
    vn = _bf16(W._normal_bf16(rng, (S, B, L, Hkv, D), 0.5), device)
    hid = _bf16(W._normal_bf16(rng, (S, B * L, H), 1.0), device)
    w = _bf16(W._normal_bf16(rng, (V, H), 0.02), device)
    mask0 = torch.ones((B, L), dtype=torch.uint8, device=device)
    mask = mask0.clone()
    tok = torch.empty((S, B, L), dtype=torch.int32, device=device)
    conf = torch.empty((S, B, L), dtype=torch.float32, device=device)
    com = torch.empty((S, B, L), dtype=torch.uint8, device=device)
    done = torch.zeros((1,), dtype=torch.int32, device=device)
    desc = bd.attn_desc(B, L, Hq, Hkv, D, a.page_table_ref.shape[1], a.k_ref.shape[0])
    d = bd.round_loop_desc(desc, S, H, V, bd.BDLM_COMMIT_THRESHOLD, 1, c["threshold"],
                           c["temperature"], q_steps=q, k_new_steps=kn, v_new_steps=vn,
                           hidden_steps=hid, k_pages=kp, v_pages=vp, page_table=pt,
                           prefix_lens=pl, w=w, mask=mask, denoising=None, tok_steps=tok,
                           conf_steps=conf, commit_steps=com, steps_done=done)
    loop = bd.bdlm_round_loop_create(d)
    stream = torch.cuda.Stream(device=device)
    try:
        evs = []
        with torch.cuda.stream(stream):
            for i in range(3 + reps):
                mask.copy_(mask0)
                flush(stream)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                bd.bdlm_round_loop_launch(loop, stream.cuda_stream)
                e1.record(stream)
                if i >= 3:
                    evs.append((e0, e1))
        torch.cuda.synchronize()
    finally:
        bd.bdlm_round_loop_destroy(loop)
    assert bd.bdlm_device_error() == 0
    ms = float(np.mean([x.elapsed_time(y) for x, y in evs]))
    rounds = int(done.item())
    kv_bytes = int((a.prefix_lens.astype(np.int64) + L).sum()) * Hkv * D * 2 * 2
    return {"workload": "config 5: B=128 L=4 Hq=32 Hkv=8 D=128, prefix U[256,4096], LM head "
                        "H=4096 V=151936 on the still-masked rows, threshold 0.75, 4 steps of "
                        "fresh Q / block K/V / hidden; one graph launch per block (WHILE node)",
            "ms_per_block": ms, "rounds": rounds, "ms_per_round": ms / max(rounds, 1),
            "value": B * L / (ms / 1e3), "unit": UNIT,
            "rounds_per_s": rounds / (ms / 1e3),
            "hbm_bytes_per_block": kv_bytes * rounds + V * H * 2 * rounds,
            "gpu_launches_per_block": 1}


def prefill_bench(bd, device, flush, reps: int, seed: int, B=128, n=512, L=4):
    """Block prefill of fresh prompts (B=128 prompts of 512 tokens, SDAR-4B attention shape,
    block length 4): the prompt's K/V written into a shuffled page pool and block-causal
    attention over the prompt.  L2 flushed before each call."""
    import torch
    rng = np.random.default_rng(seed)
    Hq, Hkv, D = 32, 8, 128
    a = W.make_attention(rng, B, n, Hq, Hkv, D, prefix_lens=np.zeros(B, np.int64), poison=False)
    kp = torch.zeros((a.k_ref.shape[0], 16, Hkv, D), dtype=torch.bfloat16, device=device)
    vp = torch.zeros_like(kp)
    pt = torch.from_numpy(a.page_table_ref).to(device)
    pl = torch.zeros((B,), dtype=torch.int32, device=device)
    q = _bf16(W._normal_bf16(rng, (B, n, Hq, D), 0.5), device)
    kn = _bf16(W._normal_bf16(rng, (B, n, Hkv, D), 0.5), device)
    vn = _bf16(W._normal_bf16(rng, (B, n, Hkv, D), 0.5), device)
    out = torch.empty((B, n, Hq, D), dtype=torch.bfloat16, device=device)
    desc = bd.attn_desc(B, L, Hq, Hkv, D, a.page_table_ref.shape[1], a.k_ref.shape[0])
    stream = torch.cuda.Stream(device=device)
    evs = []
    with torch.cuda.stream(stream):
        for i in range(3 + reps):
            flush(stream)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            bd.bdlm_prefill_attention(desc, n, q, kn, vn, kp, vp, pt, pl, out, stream.cuda_stream)
            e1.record(stream)
            if i >= 3:
                evs.append((e0, e1))
    torch.cuda.synchronize()
    assert bd.bdlm_device_error() == 0
    ms = float(np.mean([x.elapsed_time(y) for x, y in evs]))
    # the library cuts the prompt into chunks of Lq queries (the largest multiple of L dividing n
    # with Lq * G <= 256 rows), block-causal inside a chunk; chunk c reads the K/V of the
    # (c + 1) * Lq tokens up to its end once per KV head
    G = Hq // Hkv
    Lq = max([c for c in range(L, n + 1, L) if n % c == 0 and c * G <= 256] or [L])
    if Lq * G <= 32:
        Lq = L
    nq = n // Lq
    kv_read = B * Hkv * D * 2 * 2 * Lq * nq * (nq + 1) // 2
    qo = B * n * Hq * D * 2 * 2
    written = B * n * Hkv * D * 2 * 2
    return {"workload": f"prefill: {B} fresh prompts of {n} tokens, block length {L}, "
                        "Hq=32 Hkv=8 D=128, shuffled pages",
            "ms": ms, "tokens_per_s": B * n / (ms / 1e3),
            "bytes": kv_read + qo + written,
            "achieved_gbs": (kv_read + qo + written) / (ms / 1e3) / 1e9,
            "note": f"the prompt's K/V written into the cache, then block-causal attention over "
                    f"chunks of {Lq} queries (query rows on the UMMA M side), each chunk reading "
                    f"the K/V before its end once"}


# --------------------------------------------------------------------------- other configs
def time_call(fn, stream, flush, reps: int, warmup: int = 3) -> float:
    """Mean CUDA-event time (ms) of fn(stream handle) on `stream`, L2 flushed before each
    call outside the events."""
    import torch
    evs = []
    with torch.cuda.stream(stream):
        for i in range(warmup + reps):
            flush(stream)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn(stream.cuda_stream)
            e1.record(stream)
            if i >= warmup:
                evs.append((e0, e1))
    torch.cuda.synchronize()
    return float(np.mean([x.elapsed_time(y) for x, y in evs]))


def attention_bytes_flops(a, L):
    kv_tok = int((a.prefix_lens.astype(np.int64) + L).sum())
    return (kv_tok * a.Hkv * a.D * 2 * 2 + a.B * L * a.Hq * a.D * 2 * 2,
            4 * L * a.Hq * a.D * kv_tok)


def roofline_entry(ms, nbytes, flops, peaks, bound=None):
    """Achieved rates of one call against the measured peaks.  `bound` names the roofline the
    call is held to; by default the larger of its HBM and bf16 tensor times."""
    t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9)
    t_tc = flops / (peaks["bf16_tflops"] * 1e12)
    if bound is None:
        bound = "tensor" if t_tc > t_hbm else "hbm"
    r = {"us": ms * 1e3, "algorithmic_bytes": int(nbytes), "flops": int(flops),
         "achieved_gbs": nbytes / (ms / 1e3) / 1e9,
         "frac_hbm": nbytes / (ms / 1e3) / 1e9 / peaks["hbm_gbs"],
         "tflops": flops / (ms / 1e3) / 1e12, "bound": bound}
    r["frac_tensor_burst"] = r["tflops"] / peaks["bf16_tflops"]
    r["frac_tensor_sustained"] = r["tflops"] / peaks["bf16_tflops_sustained"]
    r["roofline_us"] = max(t_hbm, t_tc) * 1e6
    r["frac"] = r["frac_tensor_burst"] if bound == "tensor" else r["frac_hbm"]
    return r


def attn_parity(out, a, L, seqs):
    """Attention output of the listed sequences against the fp64 oracle."""
    import oracle
    got = out.float().cpu().numpy().astype(np.float64)
    ref = oracle.block_attention(a.q, a.k_ref, a.v_ref, a.page_table_ref, a.prefix_lens, L,
                                 a.Hq, a.Hkv, a.D, a.P, seqs=np.asarray(seqs, np.int32))
    d = np.abs(got[seqs] - ref[seqs])
    tol = 1e-2 + 1e-2 * np.abs(ref[seqs])
    return {"sequences": [int(x) for x in seqs], "max_abs_err": float(d.max()),
            "max_err_minus_tol": float((d - tol).max()), "ok": bool((d <= tol).all())}


def logits_parity(logits_d, hidden, w, rows):
    """Stored bf16 logits of the listed rows against the fp64 oracle's LM head."""
    import oracle
    rows = np.asarray(rows, np.int32)
    ref = oracle.lm_head(hidden, w, rows)
    got = logits_d[rows.tolist()].float().cpu().numpy().astype(np.float64)
    d = np.abs(got - ref)
    tol = 1e-2 + 1e-2 * np.abs(ref)
    return {"rows": len(rows), "max_abs_err": float(d.max()),
            "max_err_minus_tol": float((d - tol).max()), "ok": bool((d <= tol).all())}


def commit_parity(ref, tok, conf, com, mask):
    """GPU tokens, confidences and commits against the oracle's: token mismatches (exact),
    the largest relative confidence error (tolerance 1e-5), blocks whose commit differs
    outside a flagged near-threshold / near-tie decision, and the near-threshold count."""
    m = mask.astype(bool)
    tok_mis = int((tok[m] != ref.tok[m]).sum()) + int((tok[~m] != -1).sum())
    rel = np.abs(conf[m].astype(np.float64) - ref.conf[m]) / np.abs(ref.conf[m])
    differ = np.any(com != ref.commit, axis=1)
    near = np.any(ref.near != 0, axis=1)
    bad = int((differ & ~near).sum())
    conf_err = float(rel.max(initial=0.0))
    return {"rows": int(m.sum()), "token_mismatches": tok_mis, "conf_max_rel_err": conf_err,
            "commit_mismatch_blocks": bad, "near_threshold_positions": int(ref.near.sum()),
            "near_blocks_differing": int((differ & near).sum()),
            "ok": tok_mis == 0 and conf_err <= 1e-5 and bad == 0}


def _dev_attention(bd, a, L, device):
    import torch
    kp, vp = _bf16(a.k_ref, device), _bf16(a.v_ref, device)
    q = _bf16(a.q, device)
    pt = torch.from_numpy(a.page_table_ref).to(device)
    pl = torch.from_numpy(a.prefix_lens).to(device)
    out = torch.empty((a.B, L, a.Hq, a.D), dtype=torch.bfloat16, device=device)
    desc = bd.attn_desc(a.B, L, a.Hq, a.Hkv, a.D, a.page_table_ref.shape[1], a.k_ref.shape[0])

    def call(s):
        bd.bdlm_block_attention(desc, q, kp, vp, pt, pl, L, out, s)
    return call, out


def _dev_commit(bd, logits_d, mask, L, V, tau, T, device):
    import torch
    B = mask.shape[0]
    mk = torch.from_numpy(np.ascontiguousarray(mask)).to(device)
    tok = torch.empty((B, L), dtype=torch.int32, device=device)
    conf = torch.empty((B, L), dtype=torch.float32, device=device)
    com = torch.empty((B, L), dtype=torch.uint8, device=device)

    def call(s):
        bd.bdlm_confidence_commit(logits_d, mk, B, L, V, tau, T, tok, conf, com, s)

    def result():
        return tok.cpu().numpy(), conf.cpu().numpy(), com.cpu().numpy()
    return call, result


def bench_config1(bd, device, flush, peaks, reps):
    """Config 1: one sequence, L=4, prefix 60 in 4 identity pages, 16 q / 8 KV heads;
    logits 4 x 151936 with +8 peaks in rows 0-2, positions 1 and 3 masked, tau 0.9."""
    import oracle
    import torch
    c = W.CONFIGS[1]
    rng = np.random.default_rng(W.seed_for(1))
    a = W.make_attention(rng, 1, 4, 16, 8, 128, prefix_range=(60, 60), identity_pages=True,
                         poison=False)
    ci = W.commit_inputs(1, rng, 1, 4, c["V"], poison=False)
    attn, out = _dev_attention(bd, a, 4, device)
    lg = _bf16(ci.logits, device)
    commit, result = _dev_commit(bd, lg, ci.mask, 4, c["V"], ci.threshold, ci.temperature, device)

    def round_(s):
        attn(s)
        commit(s)
    t_attn = time_call(attn, torch.cuda.Stream(device=device), flush, reps)
    s1 = torch.cuda.Stream(device=device)
    t_commit = time_call(commit, s1, flush, reps)
    t_round = time_call(round_, s1, flush, reps)
    ab, af = attention_bytes_flops(a, 4)
    cb = int(ci.mask.sum()) * c["V"] * 2
    tok, conf, com = result()
    ref = oracle.confidence_commit(ci.logits, ci.mask, ci.threshold, ci.temperature)
    return {"workload": "config 1: B=1 L=4 prefix 60 (4 identity pages) Hq=16 Hkv=8 D=128; "
                        "logits 4x151936 N(0,2^2) +8 peaks in rows 0-2, positions 1, 3 masked, "
                        "tau 0.9, T 1",
            "attention": roofline_entry(t_attn, ab, af, peaks),
            "commit": roofline_entry(t_commit, cb, 0, peaks, "hbm"),
            "round_us": t_round * 1e3,
            "note": "a single sequence: launch-latency bound, far from any roofline",
            "parity": {"attention": attn_parity(out, a, 4, [0]),
                       "commit": commit_parity(ref, tok, conf, com, ci.mask)}}


def bench_config3(bd, device, flush, peaks, reps):
    """Config 3: B=64, L=16 and L=32, prefixes U[1024, 8192]; the LM head (H=2560, W
    N(0,0.02^2)) on every row of the DENOISING sequences (75%), logits stored, then the commit
    over the masked rows (half of each DENOISING block; SAVING blocks have none), tau 0.9."""
    import oracle
    import torch
    c = W.CONFIGS[3]
    H, V = c["H"], c["V"]
    w = None
    res = {}
    stream = torch.cuda.Stream(device=device)
    for L in (16, 32):
        rng = np.random.default_rng(W.seed_for(3, L))
        a = W.make_attention(rng, c["B"], L, c["Hq"], c["Hkv"], c["D"], prefix_range=c["prefix"],
                             poison=False)
        den = W.denoising_sequences(rng, c["B"])
        act = W.rows_of_sequences(den, L)
        lm = W.lm_head_inputs(rng, c["B"] * L, H, V, act, w=w)
        w = lm.w
        mask = W.make_mask_fixed_fraction(rng, c["B"], L, np.where(den != 0, 0.5, 0.0))
        attn, out = _dev_attention(bd, a, L, device)
        t_attn = time_call(attn, stream, flush, reps)
        ap = attn_parity(out, a, L, [int(np.argmin(a.prefix_lens)), int(np.argmax(a.prefix_lens))])
        del attn, out
        hid = _bf16(lm.hidden, device)
        if L == 16:
            w_d = _bf16(w, device)
        act_d = torch.from_numpy(act).to(device)
        logits = torch.empty((c["B"] * L, V), dtype=torch.bfloat16, device=device)

        def lmh(s):
            bd.bdlm_lm_head(hid, w_d, act_d, len(act), c["B"] * L, H, V, logits, s)
        t_lm = time_call(lmh, stream, flush, reps)
        commit, result = _dev_commit(bd, logits, mask, L, V, c["threshold"], c["temperature"],
                                     device)
        t_commit = time_call(commit, stream, flush, reps)
        ab, af = attention_bytes_flops(a, L)
        n = len(act)
        lb, lf = V * H * 2 + n * H * 2 + n * V * 2, 2 * n * H * V
        cb = int(mask.sum()) * V * 2
        tok, conf, com = result()
        lg_bits = logits.view(torch.int16).cpu().numpy().view(np.uint16)
        ref = oracle.confidence_commit(lg_bits, mask, c["threshold"], c["temperature"])
        pick = [int(act[0]), int(act[len(act) // 2]), int(act[-1])]
        res[f"L{L}"] = {
            "attention": roofline_entry(t_attn, ab, af, peaks),
            "lm_head": dict(roofline_entry(t_lm, lb, lf, peaks), rows=n),
            "commit": dict(roofline_entry(t_commit, cb, 0, peaks, "hbm"), rows=int(mask.sum())),
            "round_us": (t_attn + t_lm + t_commit) * 1e3,
            "parity": {"attention": ap, "logits": logits_parity(logits, lm.hidden, w, pick),
                       "commit": commit_parity(ref, tok, conf, com, mask)}}
        del hid, act_d, logits, commit, lmh
        torch.cuda.empty_cache()
    del w_d
    return dict(res, workload="config 3: B=64, L=16 and 32, Hq=32 Hkv=8 D=128, prefix "
                              "U[1024,8192], shuffled pages; LM head H=2560 V=151936 on every "
                              "row of the DENOISING sequences (75%), logits stored; commit over "
                              "the masked rows (half of each DENOISING block), tau 0.9",
                note="stages timed one by one (CUDA events, L2 flushed before each); round_us "
                     "is their sum")


def bench_config4(bd, device, flush, peaks, reps):
    """Config 4: B=16, L=64, prefixes U[8192, 16384]; logits 16 x 64 x 151936 with Zipf(1.1)
    peaks, masked fraction U[0.1, 0.9] per block, tau 0.75."""
    import oracle
    import torch
    c = W.CONFIGS[4]
    rng = np.random.default_rng(W.seed_for(4))
    a = W.make_attention(rng, c["B"], c["L"], c["Hq"], c["Hkv"], c["D"], prefix_range=c["prefix"],
                         poison=False)
    ci = W.commit_inputs(4, rng, c["B"], c["L"], c["V"], poison=False)
    stream = torch.cuda.Stream(device=device)
    attn, out = _dev_attention(bd, a, c["L"], device)
    t_attn = time_call(attn, stream, flush, reps)
    ap = attn_parity(out, a, c["L"], [int(np.argmax(a.prefix_lens))])
    del attn, out
    lg = _bf16(ci.logits, device)
    commit, result = _dev_commit(bd, lg, ci.mask, c["L"], c["V"], ci.threshold, ci.temperature,
                                 device)
    t_commit = time_call(commit, stream, flush, reps)
    tok, conf, com = result()
    ref = oracle.confidence_commit(ci.logits, ci.mask, ci.threshold, ci.temperature)
    ab, af = attention_bytes_flops(a, c["L"])
    cb = int(ci.mask.sum()) * c["V"] * 2
    del lg
    torch.cuda.empty_cache()
    return {"workload": "config 4: B=16 L=64 Hq=32 Hkv=8 D=128, prefix U[8192,16384], shuffled "
                        "pages; logits 16x64x151936 N(0,2^2) with Zipf(1.1) peaks, masked "
                        "fraction U[0.1,0.9] per block, tau 0.75",
            "attention": roofline_entry(t_attn, ab, af, peaks),
            "commit": dict(roofline_entry(t_commit, cb, 0, peaks, "hbm"), rows=int(ci.mask.sum())),
            "round_us": (t_attn + t_commit) * 1e3,
            "parity": {"attention": ap, "commit": commit_parity(ref, tok, conf, com, ci.mask)}}


def bench_fused_kv(bd, device, flush, peaks, reps, seed):
    """Config 2's attention with the block's K/V-cache write: the separate write kernel followed
    by the attention, against the attention that writes the block's K/V itself (CUDA events,
    L2 flushed before each call); and the attention alone, with the block already in the
    cache."""
    import torch
    c = W.CONFIGS[2]
    rng = np.random.default_rng(seed)
    a = W.make_attention(rng, c["B"], c["L"], c["Hq"], c["Hkv"], c["D"], prefix_range=c["prefix"],
                         poison=False)
    kn = _bf16(W._normal_bf16(rng, (a.B, a.L, a.Hkv, a.D), 0.5), device)
    vn = _bf16(W._normal_bf16(rng, (a.B, a.L, a.Hkv, a.D), 0.5), device)
    kp, vp = _bf16(a.k_ref, device), _bf16(a.v_ref, device)
    q = _bf16(a.q, device)
    pt = torch.from_numpy(a.page_table_ref).to(device)
    pl = torch.from_numpy(a.prefix_lens).to(device)
    out = torch.empty((a.B, a.L, a.Hq, a.D), dtype=torch.bfloat16, device=device)
    desc = bd.attn_desc(a.B, a.L, a.Hq, a.Hkv, a.D, a.page_table_ref.shape[1], a.k_ref.shape[0])
    stream = torch.cuda.Stream(device=device)

    def attn(s):
        bd.bdlm_block_attention(desc, q, kp, vp, pt, pl, a.L, out, s)

    def unfused(s):
        bd.bdlm_write_block_kv(desc, kn, vn, kp, vp, pt, pl, s)
        bd.bdlm_block_attention(desc, q, kp, vp, pt, pl, a.L, out, s)

    def fused(s):
        bd.bdlm_block_attention_kv(desc, q, kn, vn, kp, vp, pt, pl, a.L, out, s)
    t_a = time_call(attn, stream, flush, reps)
    t_u = time_call(unfused, stream, flush, reps)
    t_f = time_call(fused, stream, flush, reps)
    assert bd.bdlm_device_error() == 0
    nbytes, flops = attention_bytes_flops(a, a.L)
    nbytes += 2 * a.B * a.L * a.Hkv * a.D * 2 * 2   # the block's K/V read in and written out
    return {"workload": "config 2 attention with the block's new K/V written into the cache",
            "attention_us": t_a * 1e3, "write_then_attention_us": t_u * 1e3,
            "fused_us": t_f * 1e3, "fused": roofline_entry(t_f, nbytes, flops, peaks, "hbm"),
            "gpu_launches": {"write_then_attention": 3, "fused": 2}}


def headline_parity(bd, a, ci, lm, device):
    """Parity of the headline round on the timed inputs: one fused round (attention, LM head +
    confidence/commit, the scored rows' bf16 logits stored), attention of sampled sequences
    and logits of sampled rows against the oracle, every position's token, confidence and
    commit against the oracle over the GPU's stored logits; and config 2 as printed (the
    commit over the supplied logits) against the oracle over the same logits."""
    import oracle
    import torch
    rnd = Round(bd, a, ci, lm, device, mode="fused")
    stream = torch.cuda.Stream(device=device)
    rnd.step(stream)
    torch.cuda.synchronize()
    tok0, conf0, com0 = rnd.tok.cpu().numpy(), rnd.conf.cpu().numpy(), rnd.commit.cpu().numpy()
    logits = torch.full((a.B * a.L, ci.V), float("nan"), dtype=torch.bfloat16, device=device)
    mask0 = torch.from_numpy(ci.mask).to(device)
    bd.bdlm_lm_head_commit(rnd.hidden, rnd.w, mask0, None, a.B, a.L, lm.H, ci.V,
                           bd.BDLM_COMMIT_THRESHOLD, 1, ci.threshold, ci.temperature, rnd.tok,
                           rnd.conf, rnd.commit, logits, stream.cuda_stream)
    torch.cuda.synchronize()
    same = (np.array_equal(tok0, rnd.tok.cpu().numpy()) and
            np.array_equal(conf0, rnd.conf.cpu().numpy()) and
            np.array_equal(com0, rnd.commit.cpu().numpy()))
    lg_bits = logits.view(torch.int16).cpu().numpy().view(np.uint16)
    ref = oracle.confidence_commit(lg_bits, ci.mask, ci.threshold, ci.temperature)
    seqs = sorted({int(np.argmin(a.prefix_lens)), int(np.argmax(a.prefix_lens)), 1, 64})
    act = lm.active_idx
    out = {"attention": attn_parity(rnd.out, a, a.L, seqs),
           "logits": logits_parity(logits, lm.hidden, lm.w, [int(act[0]), int(act[-1])]),
           "commit": commit_parity(ref, tok0, conf0, com0, ci.mask),
           "stored_logits_path_identical": bool(same)}
    del rnd, logits
    sup = Round(bd, a, ci, lm, device, mode="supplied")
    sup.step(stream)
    torch.cuda.synchronize()
    ref_s = oracle.confidence_commit(ci.logits, ci.mask, ci.threshold, ci.temperature)
    out["commit_supplied_logits"] = commit_parity(ref_s, sup.tok.cpu().numpy(),
                                                  sup.conf.cpu().numpy(),
                                                  sup.commit.cpu().numpy(), ci.mask)
    del sup
    torch.cuda.empty_cache()
    out["ok"] = all(v["ok"] for k, v in out.items() if isinstance(v, dict)) and bool(same)
    out["note"] = ("tolerances: attention and logits |err| <= 1e-2 + 1e-2 |ref|; tokens exact; "
                   "confidence 1e-5 relative; commits exact outside flagged near-threshold blocks")
    return out


# kernel -> (ncu summary under profiles/, the source files its device code is compiled from)
KERNEL_SOURCES = {
    "attention": ("attention_config2",
                  ("attention.cu", "attention_common.cuh", "kernels.h", "ptx.cuh")),
    "lm_head_commit": ("lm_conf_config2_256rows",
                       ("lm_conf.cu", "lm_common.cuh", "confidence.cuh", "kernels.h", "ptx.cuh")),
    "lm_head": ("lm_head_config2_256rows", ("lm_head.cu", "lm_common.cuh", "kernels.h", "ptx.cuh")),
    "commit": ("commit_config2", ("commit.cu", "confidence.cuh", "kernels.h", "ptx.cuh"))}


def kernel_roofline(name, alg, ms, peaks):
    """HBM roofline of one call: algorithmic bytes over its CUDA-event time."""
    nbytes, flops = alg[name]
    prof, src = KERNEL_SOURCES[name]
    achieved = nbytes / (ms / 1e3) / 1e9
    r = {"kernel": name, "bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
         "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
         "traffic": profile_traffic(prof, src),
         "algorithmic_bytes": nbytes, "ms": ms,
         "peak_source": f"{peaks['source']} (copy bandwidth)"}
    if flops:
        r["tflops"] = flops / (ms / 1e3) / 1e12
    if name in ("lm_head", "lm_head_commit"):
        r["frac_tensor"] = r["tflops"] / peaks["bf16_tflops"]
    return r


def run_ours(args, rank, world, local):
    import torch
    import block_diffusion_gb300 as bd
    from block_diffusion_gb300 import build as bbuild

    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if not os.path.exists(bbuild.OUT):
        bbuild.build()
    bd.load_library()
    peaks = load_peaks()

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    flush_buf = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=device)

    def flush(stream):
        with torch.cuda.stream(stream):
            flush_buf.fill_(rank & 0xFF)

    # each rank denoises its own batch of 128 sequences (data parallel, no collective)
    c, a, ci, lm = make_workload(rank_seed(args.seed, rank), compact_pool=args.compact_pool)
    rnd = Round(bd, a, ci, lm, device, mode="fused")
    stream = torch.cuda.Stream(device=device)
    sampler = ClockSampler(local)
    sampler.start()
    if args.eager:
        total, stage, wall = time_round(rnd, stream, args.steps, max(3, args.warmup), flush,
                                        barrier)
        sustained = None
    else:
        total, wall = time_round_graph(rnd, stream, args.steps, max(3, args.warmup), flush,
                                       barrier)
    clocks = sampler.stop()
    if not args.eager:
        sustained = time_round_graph(rnd, stream, 3, 3, flush, lambda: None,
                                     sustain_s=0.0 if args.quick else 1.5, gpu_index=local)
        sustained = sustained[2] if len(sustained) == 3 else None
    assert bd.bdlm_device_error() == 0, "device error during the timed round"
    eager_n = max(20, min(args.steps, 200))
    eager_total, stage, _ = time_round(rnd, stream, eager_n, 3, flush, barrier)
    n_act = rnd.n_act
    del rnd
    torch.cuda.empty_cache()

    ms = float(total.mean())
    ms_max = max_over_ranks(ms, world)
    value = job_value(a.B * a.L, world, ms_max)

    alg = algorithmic(a, ci, lm)
    stage_ms = {k: float(stage[:, i].mean()) for i, k in enumerate(Round.STAGES["fused"])}
    kernels = {k: kernel_roofline(k, alg, stage_ms[k], peaks)
               for k in ("attention", "lm_head_commit")}
    dominant = max(("attention", "lm_head_commit"), key=lambda k: stage_ms[k])
    roofline = dict(kernels[dominant])
    step_bytes = alg["attention"][0] + alg["lm_head_commit"][0]
    roofline["round_frac"] = step_bytes / (ms / 1e3) / 1e9 / peaks["hbm_gbs"]

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": ms_max,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": line_config(world, n_act, args.seed),
            "clocks": clocks,
            "gpu_launches": Round.LAUNCHES["fused"] * args.steps,
            "launch": "eager" if args.eager else "cuda_graph",
            "eager_ms_per_step": float(eager_total.mean()),
            "stages_ms": dict(stage_ms, note="eager launches; each stage includes its launch "
                                             "gap; attention includes the split merge; "
                                             "lm_head_commit includes the scored-row list, "
                                             "the row gather and the per-block finalize"),
            "roofline": roofline,
            "kernels": kernels,
            "wall_s": wall}
    if sustained is not None:
        sustained["value"] = job_value(a.B * a.L, 1, sustained["ms_per_step"])
        line["sustained"] = sustained

    if rank == 0:
        # the same round with the logits written to HBM and read back by the commit kernel
        unf = Round(bd, a, ci, lm, device, mode="unfused")
        u_steps = max(20, min(args.steps, 500))
        if args.eager:
            utotal, _, _ = time_round(unf, stream, u_steps, 3, flush, lambda: None)
        else:
            utotal, _ = time_round_graph(unf, stream, u_steps, 3, flush, lambda: None)
        _, ustage, _ = time_round(unf, stream, eager_n, 3, flush, lambda: None)
        ustage_ms = {k: float(ustage[:, i].mean()) for i, k in enumerate(Round.STAGES["unfused"])}
        for k in ("lm_head", "commit"):
            kernels[k] = kernel_roofline(k, alg, ustage_ms[k], peaks)
        line["round_unfused"] = {
            "value": a.B * a.L / (float(utotal.mean()) / 1e3), "unit": UNIT,
            "ms_per_step": float(utotal.mean()),
            "workload": "the same round with the LM head's logits stored to HBM and read back "
                        "by the streaming confidence/commit kernel",
            "stages_ms": ustage_ms,
            "gpu_launches": Round.LAUNCHES["unfused"] * u_steps}
        del unf
        torch.cuda.empty_cache()
        # config 2 as printed: the commit reads the supplied logits, no LM head
        sup = Round(bd, a, ci, lm, device, mode="supplied")
        s_steps = max(20, min(args.steps, 500))
        if args.eager:
            stotal, _, _ = time_round(sup, stream, s_steps, 3, flush, lambda: None)
        else:
            stotal, _ = time_round_graph(sup, stream, s_steps, 3, flush, lambda: None)
        line["round_supplied_logits"] = {
            "value": a.B * a.L / (float(stotal.mean()) / 1e3), "unit": UNIT,
            "ms_per_step": float(stotal.mean()),
            "workload": "config 2 as printed: attention -> commit over the supplied logits -> "
                        "mask update (no LM head)",
            "hbm_frac": (alg["attention"][0] + alg["commit"][0]) / (float(stotal.mean()) / 1e3)
                        / 1e9 / peaks["hbm_gbs"],
            "gpu_launches": Round.LAUNCHES["supplied"] * s_steps}
        del sup
        torch.cuda.empty_cache()
    if not args.quick and rank == 0:
        torch.cuda.empty_cache()
        line["parity"] = headline_parity(bd, a, ci, lm, device)
        torch.cuda.empty_cache()
        line["fused_kv_write"] = bench_fused_kv(bd, device, flush, peaks, 20, W.seed_for(2, 5))
        torch.cuda.empty_cache()
        line["configs"] = {"1": bench_config1(bd, device, flush, peaks, 20),
                           "3": bench_config3(bd, device, flush, peaks, 10),
                           "4": bench_config4(bd, device, flush, peaks, 10)}
        torch.cuda.empty_cache()
        line["chain"] = chain_config5(bd, device, flush, 20, W.seed_for(5))
        torch.cuda.empty_cache()
        line["prefill"] = prefill_bench(bd, device, flush, 10, W.seed_for(2, 9))
        torch.cuda.empty_cache()
    if not args.quick:
        barrier()
        e2e_ms, h2d, d2h = e2e_round(bd, a, ci, lm, device, max(20, args.steps // 20), 3,
                                     rank_seed(args.seed, rank) + 2)
        e2e_max = max_over_ranks(e2e_ms, world)
        line["e2e"] = {"value": job_value(a.B * a.L, world, e2e_max), "unit": UNIT,
                       "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                       "ms_per_step": e2e_max,
                       "note": "per rank and step: q, the block's new K/V, hidden rows and "
                               "mask copied in from pinned host memory (double-buffered on a "
                               "copy stream, overlapping the previous step's compute), "
                               "attention with the block K/V written into the resident cache "
                               "in the same kernel, fused LM head + commit, "
                               "mask update, tok/conf/commit copied back; the paged cache "
                               "(every prefix) and W are resident"}
        if rank == 0:
            line["cpu_baseline"] = cpu_baseline(a, ci, lm)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


ATTN_SHAPES = {"c2": (2, 4), "c3_L16": (3, 16), "c3_L32": (3, 32), "c4": (4, 64)}


def attention_shapes(args):
    """The block attention alone at the config 2-4 shapes (B, L and prefix range of each
    config, 32 q / 8 KV heads, D = 128, pools of the referenced pages x1.25): CUDA events
    around each call, L2 flushed before it; one JSON line."""
    import torch
    import block_diffusion_gb300 as bd
    from block_diffusion_gb300 import build as bbuild
    device = torch.device("cuda", 0)
    torch.cuda.set_device(device)
    if not os.path.exists(bbuild.OUT):
        bbuild.build()
    bd.load_library()
    peaks = load_peaks()
    flush_buf = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=device)
    stream = torch.cuda.Stream(device=device)
    out_rows = []
    for name, (cfg, L) in ATTN_SHAPES.items():
        if args.shape is not None and name != args.shape:
            continue
        c = W.CONFIGS[cfg]
        rng = np.random.default_rng(W.seed_for(cfg))
        a = W.make_attention(rng, c["B"], L, c["Hq"], c["Hkv"], c["D"], prefix_range=c["prefix"],
                             poison=False)
        kp, vp = _bf16(a.k_ref, device), _bf16(a.v_ref, device)
        q = _bf16(a.q, device)
        pt = torch.from_numpy(a.page_table_ref).to(device)
        pl = torch.from_numpy(a.prefix_lens).to(device)
        out = torch.empty((a.B, L, a.Hq, a.D), dtype=torch.bfloat16, device=device)
        desc = bd.attn_desc(a.B, L, a.Hq, a.Hkv, a.D, a.page_table_ref.shape[1], a.k_ref.shape[0])
        evs = []
        with torch.cuda.stream(stream):
            for i in range(max(3, args.warmup) + args.steps):
                flush_buf.fill_(i & 0xFF)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                bd.bdlm_block_attention(desc, q, kp, vp, pt, pl, L, out, stream.cuda_stream)
                e1.record(stream)
                if i >= max(3, args.warmup):
                    evs.append((e0, e1))
        torch.cuda.synchronize()
        assert bd.bdlm_device_error() == 0
        us = float(np.mean([x.elapsed_time(y) for x, y in evs])) * 1e3
        kv_tok = int((a.prefix_lens.astype(np.int64) + L).sum())
        nbytes = kv_tok * a.Hkv * a.D * 2 * 2 + a.B * L * a.Hq * a.D * 2 * 2
        flops = 4 * L * a.Hq * a.D * kv_tok
        out_rows.append({"shape": name, "B": a.B, "L": L, "us": us, "algorithmic_bytes": nbytes,
                         "achieved_gbs": nbytes / us / 1e3,
                         "frac_hbm": nbytes / us / 1e3 / peaks["hbm_gbs"],
                         "tflops": flops / us / 1e6})
        del kp, vp, q, out, a
        torch.cuda.empty_cache()
    print(json.dumps({"attention_shapes": out_rows, "steps": args.steps,
                      "peak_hbm_gbs": peaks["hbm_gbs"], "l2": "flushed before every call"}),
          flush=True)


def main(argv=None):
    args = parse_args(argv)
    rank, world, local = dist_env()
    if args.attention_shapes:
        attention_shapes(args)
        return
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local)


if __name__ == "__main__":
    main()
